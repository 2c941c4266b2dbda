// common.cuh -- internal helpers shared by the OSDN kernels (not part of the public ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "osdn.h"

namespace osdn {

// ---- element load/store in the three storage dtypes -----------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}
template <> __device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }

// Load N consecutive elements (N * sizeof(T) bytes, naturally aligned) as floats.
template <typename T, int N> struct VecIO;
template <int N> struct VecIO<float, N> {
    static_assert(N == 2 || N == 4, "");
    __device__ __forceinline__ static void load(const float* p, float* out) {
        if constexpr (N == 4) {
            float4 v = *reinterpret_cast<const float4*>(p);
            out[0] = v.x; out[1] = v.y; out[2] = v.z; out[3] = v.w;
        } else {
            float2 v = *reinterpret_cast<const float2*>(p);
            out[0] = v.x; out[1] = v.y;
        }
    }
    __device__ __forceinline__ static void store(float* p, const float* in) {
        if constexpr (N == 4) *reinterpret_cast<float4*>(p) = make_float4(in[0], in[1], in[2], in[3]);
        else *reinterpret_cast<float2*>(p) = make_float2(in[0], in[1]);
    }
};
template <typename H, int N> struct VecIO16 {  // 16-bit types
    static_assert(N == 2 || N == 4, "");
    __device__ __forceinline__ static void load(const H* p, float* out) {
        if constexpr (N == 4) {
            uint2 v = *reinterpret_cast<const uint2*>(p);
            const H* h = reinterpret_cast<const H*>(&v);
#pragma unroll
            for (int i = 0; i < 4; ++i) out[i] = to_f32(h[i]);
        } else {
            uint32_t v = *reinterpret_cast<const uint32_t*>(p);
            const H* h = reinterpret_cast<const H*>(&v);
            out[0] = to_f32(h[0]);
            out[1] = to_f32(h[1]);
        }
    }
    __device__ __forceinline__ static void store(H* p, const float* in) {
        if constexpr (N == 4) {
            uint2 v;
            H* h = reinterpret_cast<H*>(&v);
#pragma unroll
            for (int i = 0; i < 4; ++i) h[i] = from_f32<H>(in[i]);
            *reinterpret_cast<uint2*>(p) = v;
        } else {
            uint32_t v;
            H* h = reinterpret_cast<H*>(&v);
            h[0] = from_f32<H>(in[0]);
            h[1] = from_f32<H>(in[1]);
            *reinterpret_cast<uint32_t*>(p) = v;
        }
    }
};
template <int N> struct VecIO<__nv_bfloat16, N> : VecIO16<__nv_bfloat16, N> {};
template <int N> struct VecIO<__half, N> : VecIO16<__half, N> {};

// One token of the preconditioner replay for one key coordinate ("OSDN: Improving Delta Rule with
// Provable Online Preconditioning in Linear Attention", Algorithm 1, Eq. (4)): with the step size
// g_t fixed by the scan, d <- clip(r_t d + g_t k_t^2, d_min, d_max).  The increment g_t k_t^2 is
// rounded once by itself (k_t^2 is exact for 16-bit keys), so that it is formed ahead of the
// serial dependency on d; every kernel that replays the recurrence uses these two functions, so
// all of them produce the same write keys.
__device__ __forceinline__ float replay_inc(float g, float k) { return g * (k * k); }
__device__ __forceinline__ float replay_step(float d, float r, float inc, float dmin, float dmax) {
    return fminf(fmaxf(fmaf(r, d, inc), dmin), dmax);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

}  // namespace osdn

// ---- host-side launchers, one per kernel family (defined in the .cu files) -------------------
struct OsdnScanArgs {
    const void* k; osdn_dtype k_dtype; const float* beta; const float* r; const float* d0;
    void* k_tilde; osdn_dtype kt_dtype; float* d_out;
    int B, T, H, K; float eta, d_min, d_max, eps; int beta_aware;
    int r_per_key;  // 1: r [B,T,H,K], one retention per key coordinate (vector retention)
};
struct OsdnChunkArgs {
    const void* q; const void* k; const void* k_tilde; const void* v; osdn_dtype dtype;
    const float* beta; const float* S0; void* o; float* S_out;
    int B, T, H, K, V, chunk; float scale;
    const float* alpha;  // [B,T,H] OSGDN state gate (Appendix B.1), or null: no gate
    int alpha_per_key;   // 1: alpha [B,T,H,K], one gate per key channel (OSKDA, Appendix B.2)
};
struct OsdnDecodeArgs {
    const void* q; const void* k; const void* v; osdn_dtype dtype; const float* beta;
    const float* r; float* S; float* d; void* o;
    int B, H, K, V; float eta, d_min, d_max, eps, scale; int beta_aware;
    int r_per_key;  // 1: r [B,H,K], one retention per key coordinate (vector retention)
    const float* alpha;  // [B,H] OSGDN state gate (Appendix B.1), or null: no gate
    int alpha_per_key;   // 1: alpha [B,H,K], one gate per key channel (OSKDA, Appendix B.2)
};

// Phase-1 scan.  16-bit keys with K = 128 use the blocked kernel; with a workspace of at least
// osdn_scan_block_workspace_bytes(a) bytes its write keys come from a separate parallel kernel.
cudaError_t osdn_launch_scan(const OsdnScanArgs& a, void* ws, size_t ws_bytes, cudaStream_t s);
cudaError_t osdn_launch_scan_block(const OsdnScanArgs& a, void* ws, size_t ws_bytes, cudaStream_t s);
size_t osdn_scan_block_workspace_bytes(const OsdnScanArgs& a);
cudaError_t osdn_launch_chunk_simt(const OsdnChunkArgs& a, cudaStream_t s);
// Tensor-core path.  With a workspace of at least osdn_chunk_tc_workspace_bytes(a) bytes it runs
// the parallel prep kernel and the serial chain kernel; otherwise one fused kernel.  Returns
// cudaErrorNotSupported when the tensor-core kernels do not cover the arguments.
cudaError_t osdn_launch_chunk_tc(const OsdnChunkArgs& a, void* ws, size_t ws_bytes, cudaStream_t s);
size_t osdn_chunk_tc_workspace_bytes(const OsdnChunkArgs& a);
// The same path's scratch without the segment split of the state pass (the prep images only).
size_t osdn_chunk_tc_plain_workspace_bytes(const OsdnChunkArgs& a);
cudaError_t osdn_launch_decode(const OsdnDecodeArgs& a, cudaStream_t s);
// Argument checks of osdn_chunk_fwd (all but the workspace); fills `out`, or sets `empty` when B
// or H is zero.  Scratch the chunk dispatch uses for validated arguments (0: none).
osdn_status osdn_chunk_validate(const void* q, const void* k, const void* k_tilde, const void* v, osdn_dtype dtype,
                                const float* beta, const float* alpha, int alpha_per_key, const float* S0, void* o,
                                float* S_out, int B, int T, int H, int K, int V, int chunk, float scale,
                                OsdnChunkArgs* out, bool* empty);
size_t osdn_chunk_scratch_bytes(const OsdnChunkArgs& a);
// Packed variable-length sequences: scatter into an [N, Tp, H, .] batch and gather back.
struct OsdnVarlenShape {
    int N, Tp, H, K, V;
    long long total;  // packed tokens
    int elt;          // bytes per q/k/v/o/k~ element
    int r_mode;       // 0 no retention, 1 one per head, 2 one per key coordinate
    int gated;        // 0 no state gate, 1 one per head, 2 one per key channel
};
struct OsdnVarlenIo {
    const int* cu;                                        // [N + 1] sequence offsets
    const void* q; const void* k; const void* v;          // packed inputs [total, H, .]
    const float* beta; const float* r; const float* alpha;
    void* k_tilde; void* o;                               // packed outputs
    const float* d0; float* d_out;                        // [N, H, K]
    void* pq; void* pk; void* pv; float* pbeta; float* pr; float* palpha; void* pkt; void* po;  // padded
};
size_t osdn_varlen_pad_bytes(const OsdnVarlenShape& v);
cudaError_t osdn_launch_varlen_pack(const OsdnVarlenIo& io, const OsdnVarlenShape& v, cudaStream_t s);
cudaError_t osdn_launch_varlen_unpack(const OsdnVarlenIo& io, const OsdnVarlenShape& v, cudaStream_t s);
cudaError_t osdn_varlen_read_and_clear_flag(unsigned int* flag);
// Layer backward (token-recurrent fp32 reverse sweeps of both phases).
struct OsdnBwdArgs {
    const void* q; const void* k; const void* v; osdn_dtype dtype;
    const float* beta; const float* r; int r_per_key; const float* d0; const float* S0;
    const float* dout;  // [B,T,H,V] fp32
    const float* dS;    // [B,H,V,K] fp32 or null
    const float* dd;    // [B,H,K] fp32 or null
    float* dq; float* dk; float* dv; float* dbeta; float* dr; float* dd0; float* dS0;
    int B, T, H, K, V; float eta, d_min, d_max, eps, scale; int beta_aware;
};
size_t osdn_bwd_workspace_bytes(int B, int T, int H, int K, int V);
cudaError_t osdn_launch_bwd(const OsdnBwdArgs& a, void* ws, cudaStream_t s);
// Fused layer forward (phase 1 + chunk prep in one cooperative launch, then the chain kernel).
cudaError_t osdn_launch_layer(const OsdnScanArgs& sa, const OsdnChunkArgs& ca, void* ws, size_t ws_bytes,
                              cudaStream_t s);
size_t osdn_layer_workspace_bytes(const OsdnScanArgs& sa, const OsdnChunkArgs& ca);
// Reads and clears the device-side word set when a 16-bit tensor-core kernel produced a non-finite
// output (call after the stream is synchronised).
cudaError_t osdn_read_and_clear_range(unsigned int* flag);
// Reads and clears the device-side timeout word (synchronous on the given stream).
cudaError_t osdn_read_and_clear_timeout(unsigned int* flag, cudaStream_t s);
