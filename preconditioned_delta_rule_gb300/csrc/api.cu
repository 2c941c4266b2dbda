// api.cu -- the extern "C" entry points declared in include/osdn.h: argument validation on the
// host (no launch on any error), dispatch to the kernels, status reporting.
#include <math.h>
#include <stdint.h>

#include "common.cuh"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool dtype_ok(int dt) { return dt == OSDN_F32 || dt == OSDN_BF16 || dt == OSDN_F16; }
bool head_dim_ok(int x) { return x == 64 || x == 128; }

// Pointer check: required pointers must be non-null; every non-null pointer 16-byte aligned.
osdn_status ptr(const void* p, bool required) {
    if (!p) return required ? OSDN_ERR_ARG : OSDN_OK;
    return aligned16(p) ? OSDN_OK : OSDN_ERR_ALIGN;
}

#define OSDN_TRY(expr)                       \
    do {                                     \
        osdn_status _st = (expr);            \
        if (_st != OSDN_OK) return _st;      \
    } while (0)

osdn_status phase1_scalars(float eta, float d_min, float d_max, float eps) {
    if (!(eta >= 0.f) || !isfinite(eta)) return OSDN_ERR_ARG;
    if (!(eps > 0.f) || !isfinite(eps)) return OSDN_ERR_ARG;
    if (isnan(d_min) || isnan(d_max) || d_min > d_max) return OSDN_ERR_ARG;
    return OSDN_OK;
}

// The CUDA error behind this thread's last OSDN_ERR_CUDA (reported by osdn_last_cuda_error).
thread_local cudaError_t t_last_cuda_error = cudaSuccess;
osdn_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return OSDN_OK;
    t_last_cuda_error = e;
    return OSDN_ERR_CUDA;
}

// phase 2 on the tensor cores where they apply, else the fp32 CUDA-core kernel
cudaError_t chunk_dispatch(const OsdnChunkArgs& a, void* ws, size_t ws_bytes, cudaStream_t s) {
    if (a.T > 0 && a.dtype != OSDN_F32 && a.K == 128 && a.V == 128) {
        cudaError_t e = osdn_launch_chunk_tc(a, ws, ws_bytes, s);
        if (e != cudaErrorNotSupported) return e;
    }
    return osdn_launch_chunk_simt(a, s);
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// phase 1 then phase 2: the fused layer path when it applies, else the two calls, each with its
// part of the workspace when it fits
cudaError_t layer_dispatch(const OsdnScanArgs& sa, const OsdnChunkArgs& ca, void* workspace, size_t workspace_bytes,
                           cudaStream_t s) {
    if (sa.T > 0) {
        cudaError_t e = osdn_launch_layer(sa, ca, workspace, workspace_bytes, s);
        if (e != cudaErrorNotSupported) return e;
    }
    const size_t need_s = osdn_scan_block_workspace_bytes(sa);
    const size_t need_c = osdn_chunk_tc_workspace_bytes(ca);
    unsigned char* w = static_cast<unsigned char*>(workspace);
    void* ws_s = nullptr;
    void* ws_c = nullptr;
    if (w && workspace_bytes >= align256(need_s) + need_c) {
        ws_s = need_s ? w : nullptr;
        ws_c = need_c ? w + align256(need_s) : nullptr;
    } else if (w && need_c && workspace_bytes >= need_c) {
        ws_c = w;
    } else if (w && need_s && workspace_bytes >= need_s) {
        ws_s = w;
    }
    cudaError_t e = osdn_launch_scan(sa, ws_s, ws_s ? need_s : 0, s);
    if (e != cudaSuccess) return e;
    return chunk_dispatch(ca, ws_c, ws_c ? need_c : 0, s);
}


}  // namespace

// Argument checks of osdn_chunk_fwd (everything but the workspace), shared with the entry
// points that call it; `empty` is set when there is nothing to compute (B or H zero).
osdn_status osdn_chunk_validate(const void* q, const void* k, const void* k_tilde, const void* v, osdn_dtype dtype,
                                const float* beta, const float* alpha, int alpha_per_key, const float* S0, void* o,
                                float* S_out, int B, int T, int H, int K, int V, int chunk, float scale,
                                OsdnChunkArgs* out, bool* empty) {
    *empty = false;
    if (B < 0 || T < 0 || H < 0 || chunk <= 0) return OSDN_ERR_SHAPE;
    if (!head_dim_ok(K) || !head_dim_ok(V)) return (K > 0 && V > 0) ? OSDN_ERR_UNSUPPORTED : OSDN_ERR_SHAPE;
    if (chunk != 64) return OSDN_ERR_UNSUPPORTED;
    if (T % chunk != 0) return OSDN_ERR_SHAPE;
    if (!dtype_ok(dtype)) return OSDN_ERR_DTYPE;
    if (!isfinite(scale)) return OSDN_ERR_ARG;
    if (alpha_per_key != 0 && alpha_per_key != 1) return OSDN_ERR_ARG;
    if ((long long)B * H > 0x7fffffffLL) return OSDN_ERR_SHAPE;
    if (B == 0 || H == 0) {
        *empty = true;
        return OSDN_OK;
    }
    const bool seq = T > 0;
    OSDN_TRY(ptr(q, seq));
    OSDN_TRY(ptr(k, seq));
    OSDN_TRY(ptr(k_tilde, seq));
    OSDN_TRY(ptr(v, seq));
    OSDN_TRY(ptr(beta, seq));
    OSDN_TRY(ptr(alpha, false));
    OSDN_TRY(ptr(o, seq));
    OSDN_TRY(ptr(S0, false));
    OSDN_TRY(ptr(S_out, true));
    *out = OsdnChunkArgs{q, k, k_tilde, v, dtype, beta, S0, o, S_out, B, T, H, K, V, chunk, scale, alpha,
                         alpha ? alpha_per_key : 0};
    return OSDN_OK;
}

// Scratch of the two-kernel tensor-core path for these (validated) arguments, without the
// segment split of the state pass (which needs more): 0 where that path does not apply.
size_t osdn_chunk_scratch_bytes(const OsdnChunkArgs& a) {
    if (a.T > 0 && a.dtype != OSDN_F32 && a.K == 128 && a.V == 128) return osdn_chunk_tc_plain_workspace_bytes(a);
    return 0;
}

extern "C" {

osdn_status osdn_precond_scan(const void* k, osdn_dtype k_dtype, const float* beta,
                              const float* r, int r_per_key, const float* d0, void* k_tilde,
                              osdn_dtype kt_dtype, float* d_out, int B, int T, int H, int K,
                              float eta, float d_min, float d_max, float eps, int beta_aware,
                              void* workspace, size_t workspace_bytes, void* stream) {
    if (B < 0 || T < 0 || H < 0) return OSDN_ERR_SHAPE;
    if (!head_dim_ok(K)) return K > 0 ? OSDN_ERR_UNSUPPORTED : OSDN_ERR_SHAPE;
    if (!dtype_ok(k_dtype) || !dtype_ok(kt_dtype)) return OSDN_ERR_DTYPE;
    OSDN_TRY(phase1_scalars(eta, d_min, d_max, eps));
    if (r_per_key != 0 && r_per_key != 1) return OSDN_ERR_ARG;
    if ((long long)B * H > 0x7fffffffLL) return OSDN_ERR_SHAPE;
    if (B == 0 || H == 0) return OSDN_OK;
    const bool seq = T > 0;
    OSDN_TRY(ptr(k, seq));
    OSDN_TRY(ptr(beta, seq));
    OSDN_TRY(ptr(k_tilde, seq));
    OSDN_TRY(ptr(r, false));
    OSDN_TRY(ptr(d0, false));
    OSDN_TRY(ptr(d_out, true));
    OSDN_TRY(ptr(workspace, false));
    OsdnScanArgs a{k, k_dtype, beta, r, d0, k_tilde, kt_dtype, d_out, B, T, H, K,
                   eta, d_min, d_max, eps, beta_aware ? 1 : 0, r != nullptr ? r_per_key : 0};
    return from_cuda(osdn_launch_scan(a, workspace, workspace_bytes, static_cast<cudaStream_t>(stream)));
}

size_t osdn_precond_scan_workspace_bytes(int B, int T, int H, int K, osdn_dtype k_dtype) {
    if (B <= 0 || T <= 0 || H <= 0) return 0;
    OsdnScanArgs a{};
    a.B = B; a.T = T; a.H = H; a.K = K; a.k_dtype = k_dtype;
    return osdn_scan_block_workspace_bytes(a);
}

osdn_status osdn_chunk_fwd(const void* q, const void* k, const void* k_tilde, const void* v,
                           osdn_dtype dtype, const float* beta, const float* alpha, int alpha_per_key,
                           const float* S0, void* o,
                           float* S_out, int B, int T, int H, int K, int V, int chunk,
                           float scale, void* workspace, size_t workspace_bytes, void* stream) {
    OsdnChunkArgs a{};
    bool empty = false;
    OSDN_TRY(osdn_chunk_validate(q, k, k_tilde, v, dtype, beta, alpha, alpha_per_key, S0, o, S_out, B, T, H, K, V,
                                 chunk, scale, &a, &empty));
    if (empty) return OSDN_OK;
    OSDN_TRY(ptr(workspace, false));
    return from_cuda(chunk_dispatch(a, workspace, workspace_bytes, static_cast<cudaStream_t>(stream)));
}

// A stand-in gate pointer for the size queries (never dereferenced): the workspace only depends
// on whether a gate is given and on its layout.
static const float* gate_tag(int gated) {
    static const float tag = 1.f;
    return gated ? &tag : nullptr;
}

size_t osdn_chunk_fwd_gated_workspace_bytes(int B, int T, int H, int K, int V, int chunk, osdn_dtype dtype,
                                            int gated) {
    if (B <= 0 || T <= 0 || H <= 0 || chunk <= 0 || T % chunk != 0) return 0;
    if (K != 128 || V != 128 || gated < 0 || gated > 2) return 0;
    OsdnChunkArgs a{};
    a.B = B; a.T = T; a.H = H; a.K = K; a.V = V; a.chunk = chunk; a.dtype = dtype;
    a.alpha = gate_tag(gated);
    a.alpha_per_key = gated == 2 ? 1 : 0;
    return osdn_chunk_tc_workspace_bytes(a);
}

size_t osdn_chunk_fwd_workspace_bytes(int B, int T, int H, int K, int V, int chunk,
                                      osdn_dtype dtype) {
    return osdn_chunk_fwd_gated_workspace_bytes(B, T, H, K, V, chunk, dtype, 0);
}

osdn_status osdn_layer_fwd(const void* q, const void* k, const void* v, osdn_dtype dtype, const float* beta,
                           const float* r, int r_per_key, const float* alpha, int alpha_per_key, const float* d0,
                           const float* S0, void* k_tilde, void* o,
                           float* S_out, float* d_out, int B, int T, int H, int K, int V, int chunk,
                           float eta, float d_min, float d_max, float eps, float scale, int beta_aware,
                           void* workspace, size_t workspace_bytes, void* stream) {
    if (B < 0 || T < 0 || H < 0 || chunk <= 0) return OSDN_ERR_SHAPE;
    if (!head_dim_ok(K) || !head_dim_ok(V)) return (K > 0 && V > 0) ? OSDN_ERR_UNSUPPORTED : OSDN_ERR_SHAPE;
    if (chunk != 64) return OSDN_ERR_UNSUPPORTED;
    if (T % chunk != 0) return OSDN_ERR_SHAPE;
    if (!dtype_ok(dtype)) return OSDN_ERR_DTYPE;
    OSDN_TRY(phase1_scalars(eta, d_min, d_max, eps));
    if (!isfinite(scale)) return OSDN_ERR_ARG;
    if (r_per_key != 0 && r_per_key != 1) return OSDN_ERR_ARG;
    if (alpha_per_key != 0 && alpha_per_key != 1) return OSDN_ERR_ARG;
    if ((long long)B * H > 0x7fffffffLL) return OSDN_ERR_SHAPE;
    if (B == 0 || H == 0) return OSDN_OK;
    const bool seq = T > 0;
    OSDN_TRY(ptr(q, seq));
    OSDN_TRY(ptr(k, seq));
    OSDN_TRY(ptr(v, seq));
    OSDN_TRY(ptr(beta, seq));
    OSDN_TRY(ptr(k_tilde, seq));
    OSDN_TRY(ptr(o, seq));
    OSDN_TRY(ptr(r, false));
    OSDN_TRY(ptr(alpha, false));
    OSDN_TRY(ptr(d0, false));
    OSDN_TRY(ptr(S0, false));
    OSDN_TRY(ptr(S_out, true));
    OSDN_TRY(ptr(d_out, true));
    OSDN_TRY(ptr(workspace, false));
    OsdnScanArgs sa{k, dtype, beta, r, d0, k_tilde, dtype, d_out, B, T, H, K, eta, d_min, d_max, eps, beta_aware ? 1 : 0,
                    r != nullptr ? r_per_key : 0};
    OsdnChunkArgs ca{q, k, k_tilde, v, dtype, beta, S0, o, S_out, B, T, H, K, V, chunk, scale, alpha,
                     alpha ? alpha_per_key : 0};
    return from_cuda(layer_dispatch(sa, ca, workspace, workspace_bytes, static_cast<cudaStream_t>(stream)));
}

size_t osdn_layer_fwd_gated_workspace_bytes(int B, int T, int H, int K, int V, int chunk, osdn_dtype dtype,
                                            int gated) {
    if (B <= 0 || T <= 0 || H <= 0 || chunk <= 0 || T % chunk != 0 || gated < 0 || gated > 2) return 0;
    OsdnScanArgs sa{};
    sa.B = B; sa.T = T; sa.H = H; sa.K = K; sa.k_dtype = dtype; sa.kt_dtype = dtype;
    OsdnChunkArgs ca{};
    ca.B = B; ca.T = T; ca.H = H; ca.K = K; ca.V = V; ca.chunk = chunk; ca.dtype = dtype;
    ca.alpha = gate_tag(gated);
    ca.alpha_per_key = gated == 2 ? 1 : 0;
    const size_t fused = osdn_layer_workspace_bytes(sa, ca);
    if (fused) return fused;
    const size_t need_s = osdn_scan_block_workspace_bytes(sa), need_c = osdn_chunk_tc_workspace_bytes(ca);
    return need_c ? align256(need_s) + need_c : need_s;
}

size_t osdn_layer_fwd_workspace_bytes(int B, int T, int H, int K, int V, int chunk, osdn_dtype dtype) {
    return osdn_layer_fwd_gated_workspace_bytes(B, T, H, K, V, chunk, dtype, 0);
}

static OsdnVarlenShape varlen_shape(int N, int max_len, int H, int K, int V, int chunk, osdn_dtype dtype,
                                    int r_mode, int gated, long long total) {
    OsdnVarlenShape v{};
    v.N = N;
    v.Tp = max_len <= chunk ? chunk : ((max_len + chunk - 1) / chunk) * chunk;
    v.H = H;
    v.K = K;
    v.V = V;
    v.total = total;
    v.elt = dtype == OSDN_F32 ? 4 : 2;
    v.r_mode = r_mode;
    v.gated = gated;
    return v;
}

size_t osdn_layer_fwd_varlen_workspace_bytes(int N, int max_len, int H, int K, int V, int chunk, osdn_dtype dtype,
                                             int r_mode, int gated) {
    if (N <= 0 || max_len < 0 || H <= 0 || chunk <= 0 || !head_dim_ok(K) || !head_dim_ok(V) || !dtype_ok(dtype))
        return 0;
    if (r_mode < 0 || r_mode > 2 || gated < 0 || gated > 2) return 0;
    const OsdnVarlenShape v = varlen_shape(N, max_len, H, K, V, chunk, dtype, r_mode, gated, 0);
    return align256(osdn_varlen_pad_bytes(v)) + osdn_layer_fwd_gated_workspace_bytes(N, v.Tp, H, K, V, chunk, dtype, gated);
}

osdn_status osdn_layer_fwd_varlen(const void* q, const void* k, const void* v, osdn_dtype dtype, const float* beta,
                                  const float* r, int r_per_key, const float* alpha, int alpha_per_key,
                                  const int* cu_seqlens, int N,
                                  long long total, int max_len, const float* d0, const float* S0, void* k_tilde,
                                  void* o, float* S_out, float* d_out, int H, int K, int V, int chunk, float eta,
                                  float d_min, float d_max, float eps, float scale, int beta_aware, void* workspace,
                                  size_t workspace_bytes, void* stream) {
    if (N < 0 || total < 0 || max_len < 0 || H < 0 || chunk <= 0) return OSDN_ERR_SHAPE;
    if (!head_dim_ok(K) || !head_dim_ok(V)) return (K > 0 && V > 0) ? OSDN_ERR_UNSUPPORTED : OSDN_ERR_SHAPE;
    if (chunk != 64) return OSDN_ERR_UNSUPPORTED;
    if (!dtype_ok(dtype)) return OSDN_ERR_DTYPE;
    OSDN_TRY(phase1_scalars(eta, d_min, d_max, eps));
    if (!isfinite(scale)) return OSDN_ERR_ARG;
    if (r_per_key != 0 && r_per_key != 1) return OSDN_ERR_ARG;
    if ((long long)N * H > 0x7fffffffLL || total > 0x7fffffffLL) return OSDN_ERR_SHAPE;
    if (N == 0 || H == 0) return OSDN_OK;
    const bool seq = total > 0;
    OSDN_TRY(ptr(cu_seqlens, true));
    OSDN_TRY(ptr(q, seq));
    OSDN_TRY(ptr(k, seq));
    OSDN_TRY(ptr(v, seq));
    OSDN_TRY(ptr(beta, seq));
    OSDN_TRY(ptr(k_tilde, seq));
    OSDN_TRY(ptr(o, seq));
    OSDN_TRY(ptr(r, false));
    OSDN_TRY(ptr(alpha, false));
    OSDN_TRY(ptr(d0, false));
    OSDN_TRY(ptr(S0, false));
    OSDN_TRY(ptr(S_out, true));
    OSDN_TRY(ptr(d_out, true));
    OSDN_TRY(ptr(workspace, true));
    const int r_mode = r ? (r_per_key ? 2 : 1) : 0;
    if (alpha_per_key != 0 && alpha_per_key != 1) return OSDN_ERR_ARG;
    const int g_mode = alpha ? (alpha_per_key ? 2 : 1) : 0;
    const OsdnVarlenShape vs = varlen_shape(N, max_len, H, K, V, chunk, dtype, r_mode, g_mode, total);
    const size_t pad = align256(osdn_varlen_pad_bytes(vs));
    const size_t need_layer = osdn_layer_fwd_gated_workspace_bytes(N, vs.Tp, H, K, V, chunk, dtype, g_mode);
    if (workspace_bytes < pad + need_layer) return OSDN_ERR_ARG;
    // the padded batch, each part 256-byte aligned, then the batched layer's own workspace
    unsigned char* w = static_cast<unsigned char*>(workspace);
    const size_t rows = static_cast<size_t>(N) * vs.Tp;
    auto take = [&](size_t bytes) {
        unsigned char* p = w;
        w += align256(bytes);
        return p;
    };
    OsdnVarlenIo io{};
    io.cu = cu_seqlens;
    io.q = q; io.k = k; io.v = v; io.beta = beta; io.r = r; io.alpha = alpha;
    io.k_tilde = k_tilde; io.o = o; io.d0 = d0; io.d_out = d_out;
    io.pq = take(rows * H * K * vs.elt);
    io.pk = take(rows * H * K * vs.elt);
    io.pkt = take(rows * H * K * vs.elt);
    io.pv = take(rows * H * V * vs.elt);
    io.po = take(rows * H * V * vs.elt);
    io.pbeta = reinterpret_cast<float*>(take(rows * H * 4));
    if (r_mode) io.pr = reinterpret_cast<float*>(take(rows * H * (r_mode == 2 ? K : 1) * 4));
    if (alpha) io.palpha = reinterpret_cast<float*>(take(rows * H * (g_mode == 2 ? K : 1) * 4));
    unsigned char* wl = static_cast<unsigned char*>(workspace) + pad;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = osdn_launch_varlen_pack(io, vs, s);
    if (e != cudaSuccess) return from_cuda(e);
    OsdnScanArgs sa{io.pk, dtype, io.pbeta, io.pr, d0, io.pkt, dtype, d_out, N, vs.Tp, H, K, eta, d_min, d_max, eps,
                    beta_aware ? 1 : 0, r_mode == 2 ? 1 : 0};
    OsdnChunkArgs ca{io.pq, io.pk, io.pkt, io.pv, dtype, io.pbeta, S0, io.po, S_out, N, vs.Tp, H, K, V, chunk, scale,
                     io.palpha, g_mode == 2 ? 1 : 0};
    e = layer_dispatch(sa, ca, wl, need_layer, s);
    if (e != cudaSuccess) return from_cuda(e);
    return from_cuda(osdn_launch_varlen_unpack(io, vs, s));
}

size_t osdn_layer_bwd_workspace_bytes(int B, int T, int H, int K, int V) {
    if (!head_dim_ok(K) || !head_dim_ok(V)) return 0;
    return osdn_bwd_workspace_bytes(B, T, H, K, V);
}

osdn_status osdn_layer_bwd(const void* q, const void* k, const void* v, osdn_dtype dtype, const float* beta,
                           const float* r, int r_per_key, const float* alpha, const float* d0, const float* S0,
                           const float* dout, const float* dS, const float* dd, float* dq, float* dk, float* dv,
                           float* dbeta, float* dr, float* dd0, float* dS0, int B, int T, int H, int K, int V,
                           float eta, float d_min, float d_max, float eps, float scale, int beta_aware,
                           void* workspace, size_t workspace_bytes, void* stream) {
    if (B < 0 || T < 0 || H < 0) return OSDN_ERR_SHAPE;
    if (!head_dim_ok(K) || !head_dim_ok(V)) return (K > 0 && V > 0) ? OSDN_ERR_UNSUPPORTED : OSDN_ERR_SHAPE;
    if (!dtype_ok(dtype)) return OSDN_ERR_DTYPE;
    OSDN_TRY(phase1_scalars(eta, d_min, d_max, eps));
    if (!isfinite(scale)) return OSDN_ERR_ARG;
    if (r_per_key != 0 && r_per_key != 1) return OSDN_ERR_ARG;
    if (alpha) return OSDN_ERR_UNSUPPORTED;  // the gated variant's backward is not built
    if ((long long)B * H > 0x7fffffffLL) return OSDN_ERR_SHAPE;
    if (B == 0 || H == 0 || T == 0) {
        // nothing flows through the tokens: the initial states' gradients are the final ones'
        const size_t ns = static_cast<size_t>(B) * H * V * K, nd = static_cast<size_t>(B) * H * K;
        cudaStream_t s = static_cast<cudaStream_t>(stream);
        if (B == 0 || H == 0) return OSDN_OK;
        if (dS0 && (dS ? cudaMemcpyAsync(dS0, dS, ns * 4, cudaMemcpyDeviceToDevice, s)
                       : cudaMemsetAsync(dS0, 0, ns * 4, s)) != cudaSuccess) return OSDN_ERR_CUDA;
        if (dd0 && (dd ? cudaMemcpyAsync(dd0, dd, nd * 4, cudaMemcpyDeviceToDevice, s)
                       : cudaMemsetAsync(dd0, 0, nd * 4, s)) != cudaSuccess) return OSDN_ERR_CUDA;
        return OSDN_OK;
    }
    OSDN_TRY(ptr(q, true));
    OSDN_TRY(ptr(k, true));
    OSDN_TRY(ptr(v, true));
    OSDN_TRY(ptr(beta, true));
    OSDN_TRY(ptr(dout, true));
    OSDN_TRY(ptr(dq, true));
    OSDN_TRY(ptr(dk, true));
    OSDN_TRY(ptr(dv, true));
    OSDN_TRY(ptr(dbeta, true));
    OSDN_TRY(ptr(r, false));
    OSDN_TRY(ptr(dr, r != nullptr));
    OSDN_TRY(ptr(d0, false));
    OSDN_TRY(ptr(S0, false));
    OSDN_TRY(ptr(dS, false));
    OSDN_TRY(ptr(dd, false));
    OSDN_TRY(ptr(dd0, false));
    OSDN_TRY(ptr(dS0, false));
    OSDN_TRY(ptr(workspace, true));
    if (workspace_bytes < osdn_bwd_workspace_bytes(B, T, H, K, V)) return OSDN_ERR_ARG;
    OsdnBwdArgs a{q, k, v, dtype, beta, r, r ? r_per_key : 0, d0, S0, dout, dS, dd, dq, dk, dv, dbeta, dr, dd0, dS0,
                  B, T, H, K, V, eta, d_min, d_max, eps, scale, beta_aware ? 1 : 0};
    return from_cuda(osdn_launch_bwd(a, workspace, static_cast<cudaStream_t>(stream)));
}

osdn_status osdn_decode_step(const void* q, const void* k, const void* v, osdn_dtype dtype,
                             const float* beta, const float* r, int r_per_key, const float* alpha,
                             int alpha_per_key, float* S, float* d, void* o,
                             int B, int H, int K, int V, float eta, float d_min, float d_max,
                             float eps, float scale, int beta_aware, void* stream) {
    if (B < 0 || H < 0) return OSDN_ERR_SHAPE;
    if (!head_dim_ok(K) || !head_dim_ok(V)) return (K > 0 && V > 0) ? OSDN_ERR_UNSUPPORTED : OSDN_ERR_SHAPE;
    if (!dtype_ok(dtype)) return OSDN_ERR_DTYPE;
    OSDN_TRY(phase1_scalars(eta, d_min, d_max, eps));
    if (!isfinite(scale)) return OSDN_ERR_ARG;
    if (r_per_key != 0 && r_per_key != 1) return OSDN_ERR_ARG;
    if (alpha_per_key != 0 && alpha_per_key != 1) return OSDN_ERR_ARG;
    if ((long long)B * H > 0x7fffffffLL) return OSDN_ERR_SHAPE;
    if (B == 0 || H == 0) return OSDN_OK;
    OSDN_TRY(ptr(q, true));
    OSDN_TRY(ptr(k, true));
    OSDN_TRY(ptr(v, true));
    OSDN_TRY(ptr(beta, true));
    OSDN_TRY(ptr(r, false));
    OSDN_TRY(ptr(alpha, false));
    OSDN_TRY(ptr(S, true));
    OSDN_TRY(ptr(d, true));
    OSDN_TRY(ptr(o, true));
    OsdnDecodeArgs a{q, k, v, dtype, beta, r, S, d, o, B, H, K, V,
                     eta, d_min, d_max, eps, scale, beta_aware ? 1 : 0, r != nullptr ? r_per_key : 0, alpha,
                     alpha ? alpha_per_key : 0};
    return from_cuda(osdn_launch_decode(a, static_cast<cudaStream_t>(stream)));
}

osdn_status osdn_check(void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int flag = 0, bad = 0;
    cudaError_t e = osdn_read_and_clear_timeout(&flag, s);
    if (e != cudaSuccess) return from_cuda(e);
    e = osdn_varlen_read_and_clear_flag(&bad);
    if (e != cudaSuccess) return from_cuda(e);
    unsigned int range = 0;
    e = osdn_read_and_clear_range(&range);
    if (e != cudaSuccess) return from_cuda(e);
    if (flag) return OSDN_ERR_TIMEOUT;
    if (bad) return OSDN_ERR_SHAPE;
    if (range) return OSDN_ERR_RANGE;
    return OSDN_OK;
}

const char* osdn_status_string(int status) {
    switch (status) {
        case OSDN_OK: return "OSDN_OK";
        case OSDN_ERR_ARG: return "OSDN_ERR_ARG: invalid argument (null pointer or bad scalar)";
        case OSDN_ERR_SHAPE: return "OSDN_ERR_SHAPE: invalid sizes (negative, or T not a multiple of the chunk)";
        case OSDN_ERR_DTYPE: return "OSDN_ERR_DTYPE: unknown dtype";
        case OSDN_ERR_ALIGN: return "OSDN_ERR_ALIGN: a pointer is not 16-byte aligned";
        case OSDN_ERR_UNSUPPORTED: return "OSDN_ERR_UNSUPPORTED: valid arguments not covered by a built kernel";
        case OSDN_ERR_CUDA: return "OSDN_ERR_CUDA: a CUDA call or launch failed";
        case OSDN_ERR_TIMEOUT: return "OSDN_ERR_TIMEOUT: a device-side bounded wait gave up";
        case OSDN_ERR_CAPACITY: return "OSDN_ERR_CAPACITY: the request needs more scratch than the fixed no-allocation array holds";
        case OSDN_ERR_RANGE: return "OSDN_ERR_RANGE: a 16-bit tensor-core call produced a non-finite output (a value left fp16's range)";
    }
    return "OSDN: unknown status";
}

int osdn_version(void) { return 200; }

const char* osdn_last_cuda_error(void) {
    return t_last_cuda_error == cudaSuccess ? "cudaSuccess" : cudaGetErrorName(t_last_cuda_error);
}

}  // extern "C"
