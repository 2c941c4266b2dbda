// host_pipeline.cu -- the layer forward on HOST buffers, with the host<->device copies overlapped
// with the compute.
//
// "OSDN: Improving Delta Rule with Provable Online Preconditioning in Linear Attention",
// Algorithm 1 and Eqs. (2), (4), (7): both phases are recurrences over the token axis whose whole
// carried state is (d, S).  So the sequence splits into `segments` consecutive pieces of T / segments
// tokens, and piece i is the layer call started from piece i-1's final (d, S): the same recurrence,
// the same 64-token blocks and chunks (every piece is a whole number of chunks), the carried d
// rounded to fp32 once per piece boundary instead of being kept as an fp32 (hi, lo) pair.
//
// Three streams: `h2d` copies piece i's inputs into one of two device staging slots while
// `stream` runs the layer on piece i-1 from the other slot, and `d2h` copies piece i-1's outputs
// back.  The (d, S) state stays on the device, in two buffers used alternately.  Events order the
// reuse of a slot: piece i+2's inputs go into slot i % 2 only after piece i's outputs have left it.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "common.cuh"

namespace {

size_t up256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct HostLayout {  // byte offsets of the parts of the device workspace
    size_t d[2], S[2];
    size_t slot[2];
    size_t q, k, v, beta, r, alpha, kt, o;  // offsets inside a slot
    size_t slot_bytes, layer, total;
};

HostLayout host_layout(int B, int T, int H, int K, int V, int chunk, osdn_dtype dtype, int r_mode, int g_mode,
                       int segments) {
    HostLayout L{};
    const size_t e = dtype == OSDN_F32 ? 4 : 2;
    const size_t Ts = static_cast<size_t>(T / segments);
    const size_t rows = static_cast<size_t>(B) * Ts * H;
    size_t o = 0;
    for (int i = 0; i < 2; ++i) {
        L.d[i] = o;
        o += up256(static_cast<size_t>(B) * H * K * 4);
        L.S[i] = o;
        o += up256(static_cast<size_t>(B) * H * V * K * 4);
    }
    size_t s = 0;
    L.q = s; s += up256(rows * K * e);
    L.k = s; s += up256(rows * K * e);
    L.v = s; s += up256(rows * V * e);
    L.beta = s; s += up256(rows * 4);
    L.r = s; s += r_mode ? up256(rows * (r_mode == 2 ? K : 1) * 4) : 0;
    L.alpha = s; s += g_mode ? up256(rows * (g_mode == 2 ? K : 1) * 4) : 0;
    L.kt = s; s += up256(rows * K * e);
    L.o = s; s += up256(rows * V * e);
    L.slot_bytes = s;
    L.slot[0] = o;
    L.slot[1] = o + s;
    o += 2 * s;
    L.layer = o;
    o += osdn_layer_fwd_gated_workspace_bytes(B, static_cast<int>(Ts), H, K, V, chunk, dtype, g_mode);
    L.total = o;
    return L;
}

// rows [t0, t0 + Ts) of every batch entry of a host [B, T, row] tensor <-> a device [B, Ts, row] one
cudaError_t copy_piece(void* dst, const void* src, size_t row_bytes, int B, int T, int Ts, int t0, bool to_device,
                       cudaStream_t s) {
    const size_t width = row_bytes * Ts, full = row_bytes * T;
    if (to_device) {
        const unsigned char* h = static_cast<const unsigned char*>(src) + row_bytes * t0;
        if (B == 1) return cudaMemcpyAsync(dst, h, width, cudaMemcpyHostToDevice, s);
        return cudaMemcpy2DAsync(dst, width, h, full, width, B, cudaMemcpyHostToDevice, s);
    }
    unsigned char* h = static_cast<unsigned char*>(dst) + row_bytes * t0;
    if (B == 1) return cudaMemcpyAsync(h, src, width, cudaMemcpyDeviceToHost, s);
    return cudaMemcpy2DAsync(h, full, src, width, width, B, cudaMemcpyDeviceToHost, s);
}

struct Events {
    cudaEvent_t ev[8] = {};
    int n = 0;
    cudaError_t make() {
        for (; n < 8; ++n) {
            cudaError_t e = cudaEventCreateWithFlags(&ev[n], cudaEventDisableTiming);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    ~Events() {  // a pending event's resources are released once it completes
        for (int i = 0; i < n; ++i) cudaEventDestroy(ev[i]);
    }
};

}  // namespace

extern "C" size_t osdn_layer_fwd_host_workspace_bytes(int B, int T, int H, int K, int V, int chunk, osdn_dtype dtype,
                                                      int r_mode, int gated, int segments) {
    if (B <= 0 || T <= 0 || H <= 0 || chunk <= 0 || segments <= 0) return 0;
    if ((K != 64 && K != 128) || (V != 64 && V != 128)) return 0;
    if (dtype != OSDN_F32 && dtype != OSDN_BF16 && dtype != OSDN_F16) return 0;
    if (r_mode < 0 || r_mode > 2 || gated < 0 || gated > 2) return 0;
    if (T % segments != 0 || (T / segments) % chunk != 0) return 0;
    return host_layout(B, T, H, K, V, chunk, dtype, r_mode, gated, segments).total;
}

extern "C" osdn_status osdn_layer_fwd_host(const void* q, const void* k, const void* v, osdn_dtype dtype,
                                           const float* beta, const float* r, int r_per_key, const float* alpha,
                                           int alpha_per_key, const float* d0, const float* S0, void* o,
                                           float* S_out, float* d_out, int B, int T, int H, int K, int V, int chunk,
                                           float eta, float d_min, float d_max, float eps, float scale,
                                           int beta_aware, int segments, void* workspace, size_t workspace_bytes,
                                           void* stream, void* h2d_stream, void* d2h_stream) {
    if (B < 0 || T < 0 || H < 0 || chunk <= 0) return OSDN_ERR_SHAPE;
    if (segments <= 0) return OSDN_ERR_ARG;
    if ((K != 64 && K != 128) || (V != 64 && V != 128)) return (K > 0 && V > 0) ? OSDN_ERR_UNSUPPORTED : OSDN_ERR_SHAPE;
    if (chunk != 64) return OSDN_ERR_UNSUPPORTED;
    if (T % segments != 0 || (T / segments) % chunk != 0) return OSDN_ERR_SHAPE;
    if (dtype != OSDN_F32 && dtype != OSDN_BF16 && dtype != OSDN_F16) return OSDN_ERR_DTYPE;
    if (r_per_key != 0 && r_per_key != 1) return OSDN_ERR_ARG;
    if (alpha_per_key != 0 && alpha_per_key != 1) return OSDN_ERR_ARG;
    // the scalar checks of osdn_layer_fwd, here so that no copy is queued for a call it would reject
    if (!(eta >= 0.f) || !isfinite(eta) || !(eps > 0.f) || !isfinite(eps)) return OSDN_ERR_ARG;
    if (isnan(d_min) || isnan(d_max) || d_min > d_max || !isfinite(scale)) return OSDN_ERR_ARG;
    if ((long long)B * H > 0x7fffffffLL) return OSDN_ERR_SHAPE;
    if (B == 0 || H == 0) return OSDN_OK;
    if (!S_out || !d_out) return OSDN_ERR_ARG;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const size_t n_d = static_cast<size_t>(B) * H * K, n_S = static_cast<size_t>(B) * H * V * K;
    if (T == 0) {  // no tokens: the outputs are the start state, written on the host once `stream` is idle
        if (cudaStreamSynchronize(cs) != cudaSuccess) return OSDN_ERR_CUDA;
        for (size_t i = 0; i < n_d; ++i) d_out[i] = d0 ? d0[i] : 1.f;
        if (S0) memmove(S_out, S0, n_S * 4);
        else memset(S_out, 0, n_S * 4);
        return OSDN_OK;
    }
    if (!q || !k || !v || !beta || !o) return OSDN_ERR_ARG;
    if (!workspace) return OSDN_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return OSDN_ERR_ALIGN;
    const int r_mode = r ? (r_per_key ? 2 : 1) : 0;
    const int g_mode = alpha ? (alpha_per_key ? 2 : 1) : 0;
    const int nseg = segments;
    const int Ts = T / nseg;
    const HostLayout L = host_layout(B, T, H, K, V, chunk, dtype, r_mode, g_mode, nseg);
    if (workspace_bytes < L.total) return OSDN_ERR_ARG;

    cudaStream_t hs = h2d_stream ? static_cast<cudaStream_t>(h2d_stream) : cs;
    cudaStream_t ds = d2h_stream ? static_cast<cudaStream_t>(d2h_stream) : cs;
    unsigned char* w = static_cast<unsigned char*>(workspace);
    const size_t e = dtype == OSDN_F32 ? 4 : 2;
    const size_t d_bytes = n_d * 4, S_bytes = n_S * 4;

    Events E;
    if (E.make() != cudaSuccess) return OSDN_ERR_CUDA;
    cudaEvent_t ev_start = E.ev[0], ev_end = E.ev[1];
    cudaEvent_t* ev_in = E.ev + 2;   // [2] piece's inputs are in slot
    cudaEvent_t* ev_out = E.ev + 4;  // [2] slot's outputs have left it
    cudaEvent_t* ev_done = E.ev + 6; // [2] piece's layer call finished
#define HP_TRY(x)                                  \
    do {                                           \
        if ((x) != cudaSuccess) return OSDN_ERR_CUDA; \
    } while (0)
    // work the caller queued on `stream` earlier (e.g. a previous call on this workspace) first
    HP_TRY(cudaEventRecord(ev_start, cs));
    if (hs != cs) HP_TRY(cudaStreamWaitEvent(hs, ev_start, 0));
    if (ds != cs) HP_TRY(cudaStreamWaitEvent(ds, ev_start, 0));

    float* dbuf[2] = {reinterpret_cast<float*>(w + L.d[0]), reinterpret_cast<float*>(w + L.d[1])};
    float* Sbuf[2] = {reinterpret_cast<float*>(w + L.S[0]), reinterpret_cast<float*>(w + L.S[1])};
    if (d0) HP_TRY(cudaMemcpyAsync(dbuf[0], d0, d_bytes, cudaMemcpyHostToDevice, hs));
    if (S0) HP_TRY(cudaMemcpyAsync(Sbuf[0], S0, S_bytes, cudaMemcpyHostToDevice, hs));

    const size_t rq = static_cast<size_t>(H) * K * e, rv = static_cast<size_t>(H) * V * e;
    const size_t rb = static_cast<size_t>(H) * 4;
    const size_t rr = static_cast<size_t>(H) * (r_mode == 2 ? K : 1) * 4;
    const size_t ra = static_cast<size_t>(H) * (g_mode == 2 ? K : 1) * 4;
    for (int i = 0; i < nseg; ++i) {
        const int sl = i & 1;
        unsigned char* slot = w + L.slot[sl];
        const int t0 = i * Ts;
        if (i >= 2) HP_TRY(cudaStreamWaitEvent(hs, ev_out[sl], 0));
        HP_TRY(copy_piece(slot + L.q, q, rq, B, T, Ts, t0, true, hs));
        HP_TRY(copy_piece(slot + L.k, k, rq, B, T, Ts, t0, true, hs));
        HP_TRY(copy_piece(slot + L.v, v, rv, B, T, Ts, t0, true, hs));
        HP_TRY(copy_piece(slot + L.beta, beta, rb, B, T, Ts, t0, true, hs));
        if (r) HP_TRY(copy_piece(slot + L.r, r, rr, B, T, Ts, t0, true, hs));
        if (alpha) HP_TRY(copy_piece(slot + L.alpha, alpha, ra, B, T, Ts, t0, true, hs));
        HP_TRY(cudaEventRecord(ev_in[sl], hs));
        if (hs != cs) HP_TRY(cudaStreamWaitEvent(cs, ev_in[sl], 0));
        // piece i starts from buffer i % 2 (or the caller's defaults: NULL d0 / S0 mean ones / zeros)
        const bool first = i == 0;
        const float* din = first ? (d0 ? dbuf[0] : nullptr) : dbuf[sl];
        const float* Sin = first ? (S0 ? Sbuf[0] : nullptr) : Sbuf[sl];
        const osdn_status st = osdn_layer_fwd(
            slot + L.q, slot + L.k, slot + L.v, dtype, reinterpret_cast<const float*>(slot + L.beta),
            r ? reinterpret_cast<const float*>(slot + L.r) : nullptr, r_per_key,
            alpha ? reinterpret_cast<const float*>(slot + L.alpha) : nullptr, alpha_per_key, din, Sin,
            slot + L.kt, slot + L.o, Sbuf[sl ^ 1], dbuf[sl ^ 1], B, Ts, H, K, V, chunk, eta, d_min, d_max, eps, scale,
            beta_aware, L.total > L.layer ? w + L.layer : nullptr, L.total - L.layer, cs);
        if (st != OSDN_OK) return st;
        HP_TRY(cudaEventRecord(ev_done[sl], cs));
        if (ds != cs) HP_TRY(cudaStreamWaitEvent(ds, ev_done[sl], 0));
        HP_TRY(copy_piece(o, slot + L.o, rv, B, T, Ts, t0, false, ds));
        HP_TRY(cudaEventRecord(ev_out[sl], ds));
    }
    const int fin = nseg & 1;  // the last piece wrote buffer nseg % 2
    HP_TRY(cudaMemcpyAsync(d_out, dbuf[fin], d_bytes, cudaMemcpyDeviceToHost, ds));
    HP_TRY(cudaMemcpyAsync(S_out, Sbuf[fin], S_bytes, cudaMemcpyDeviceToHost, ds));
    HP_TRY(cudaEventRecord(ev_end, ds));
    if (ds != cs) HP_TRY(cudaStreamWaitEvent(cs, ev_end, 0));
#undef HP_TRY
    return OSDN_OK;
}
