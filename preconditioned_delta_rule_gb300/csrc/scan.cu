// scan.cu -- phase 1 of OSDN: the online preconditioner sweep.
//
// "OSDN: Improving Delta Rule with Provable Online Preconditioning in Linear Attention",
// Section 4.2, Algorithm 1 and Eq. (4); the APF retention gate of Section 4.4, Eq. (7).
// Per (batch, head), for t = 0..T-1 (serial in t):
//   k~_t = d_t . k_t                                   (emitted with the OLD d)
//   s = k_t . k_t;  n = max(sum(s), eps);  a = <d_t, s>
//   g = eta * b * (1 - b * a) / n,  b = beta_t (beta-aware) or 1
//   d_{t+1} = clip(r_t * d_t + g * s, d_min, d_max)
//
// Mapping: one warp per (batch, head); lane l owns key coordinates [l*E, l*E+E), E = K/32.
// The two K-wide reductions (|k|^2 and <d, s>) are warp butterflies.  Keys, gates and
// retentions are staged 32 tokens at a time into shared memory with cp.async, double buffered,
// so the serial chain only waits on shared memory.  d is carried as an unevaluated fp32 pair
// (hi + lo): a long stream of O(eta / K) increments on d ~ 1 would otherwise lose ~1e-5 of
// relative accuracy over 10^4 tokens.
#include "common.cuh"

namespace osdn {
namespace {

constexpr int kStageTokens = 32;

__device__ __forceinline__ void cp_async_16(void* smem, const void* gmem) {
    uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_4(void* smem, const void* gmem) {
    uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_1() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_0() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

// One projected, compensated step on a coordinate: (hi, lo) <- clip(r (hi + lo) + g s).
__device__ __forceinline__ void d_step(float& hi, float& lo, float r, float g, float s,
                                       float dmin, float dmax) {
    float p = r * hi;
    float ep = fmaf(r, hi, -p);        // exact rounding error of r * hi
    float q = g * s;
    float x = p + q;                   // TwoSum(p, q)
    float z = x - p;
    float ex = (p - (x - z)) + (q - z);
    float l = fmaf(r, lo, ep + ex);
    float h2 = x + l;                  // renormalise (|l| << |x|)
    float l2 = l - (h2 - x);
    if (h2 < dmin || (h2 == dmin && l2 < 0.f)) { h2 = dmin; l2 = 0.f; }
    if (h2 > dmax || (h2 == dmax && l2 > 0.f)) { h2 = dmax; l2 = 0.f; }
    hi = h2;
    lo = l2;
}

// RMODE: 0 no retention, 1 one retention per head and token (Eq. (7)), 2 one per key coordinate
// (vector retention diag(r_t), Appendix A.5), staged with the keys, 16 tokens at a time.
template <int K, typename TIn, typename TOut, int RMODE>
__global__ void __launch_bounds__(32) scan_warp_kernel(OsdnScanArgs a) {
    constexpr bool HAS_R = RMODE != 0;
    constexpr int NST = RMODE == 2 ? kStageTokens / 2 : kStageTokens;
    constexpr int E = K / 32;
    constexpr int ROWB = K * (int)sizeof(TIn);
    constexpr int PIECES = ROWB / 16;
    constexpr int RROW = RMODE == 2 ? K : 1;  // retention floats per token
    __shared__ __align__(16) unsigned char kbuf[2][NST * ROWB];
    __shared__ float bbuf[2][NST];
    __shared__ __align__(16) float rbuf[2][NST * RROW];

    const int lane = threadIdx.x;
    const int bh = blockIdx.x;
    const int b = bh / a.H, h = bh % a.H;
    const int T = a.T, H = a.H;
    const TIn* kg = static_cast<const TIn*>(a.k);
    TOut* ktg = static_cast<TOut*>(a.k_tilde);
    const size_t row0 = (size_t)b * T * H + h;  // row of token 0; token t is row0 + t*H

    float dh[E], dl[E];
#pragma unroll
    for (int i = 0; i < E; ++i) {
        dh[i] = a.d0 ? a.d0[(size_t)bh * K + lane * E + i] : 1.f;
        dl[i] = 0.f;
    }

    auto stage = [&](int buf, int t0) {
        const int nt = min(NST, T - t0);
        for (int i = lane; i < nt * PIECES; i += 32) {
            const int tt = i / PIECES, c = i - tt * PIECES;
            const unsigned char* src =
                reinterpret_cast<const unsigned char*>(kg + (row0 + (size_t)(t0 + tt) * H) * K) + c * 16;
            cp_async_16(&kbuf[buf][tt * ROWB + c * 16], src);
        }
        if (RMODE == 2) {  // K fp32 per token, 16-byte pieces
            for (int i = lane; i < nt * (K / 4); i += 32) {
                const int tt = i / (K / 4), c = i - tt * (K / 4);
                cp_async_16(&rbuf[buf][tt * K + c * 4], a.r + (row0 + (size_t)(t0 + tt) * H) * K + c * 4);
            }
        }
        if (lane < nt) {
            cp_async_4(&bbuf[buf][lane], a.beta + row0 + (size_t)(t0 + lane) * H);
            if (RMODE == 1) cp_async_4(&rbuf[buf][lane], a.r + row0 + (size_t)(t0 + lane) * H);
        }
        cp_async_commit();
    };

    if (T > 0) stage(0, 0);
    for (int t0 = 0, it = 0; t0 < T; t0 += NST, ++it) {
        const int buf = it & 1;
        if (t0 + NST < T) stage(buf ^ 1, t0 + NST);
        else cp_async_commit();
        cp_async_wait_1();
        __syncwarp();
        const int nt = min(NST, T - t0);
#pragma unroll 2
        for (int tt = 0; tt < nt; ++tt) {
            float kv[E];
            VecIO<TIn, E>::load(reinterpret_cast<const TIn*>(&kbuf[buf][tt * ROWB]) + lane * E, kv);
            const float bt = bbuf[buf][tt];
            float rv[E];
#pragma unroll
            for (int i = 0; i < E; ++i)
                rv[i] = RMODE == 2 ? rbuf[buf][tt * RROW + lane * E + i] : (HAS_R ? rbuf[buf][tt] : 1.f);
            float s[E], n = 0.f, al = 0.f, ko[E];
#pragma unroll
            for (int i = 0; i < E; ++i) {
                s[i] = kv[i] * kv[i];
                n += s[i];
                al = fmaf(dh[i], s[i], al);
                ko[i] = fmaf(dl[i], kv[i], dh[i] * kv[i]);  // write key with the old d
            }
            VecIO<TOut, E>::store(ktg + (row0 + (size_t)(t0 + tt) * H) * K + lane * E, ko);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                n += __shfl_xor_sync(0xffffffffu, n, o);
                al += __shfl_xor_sync(0xffffffffu, al, o);
            }
            const float nbar = fmaxf(n, a.eps);
            const float bp = a.beta_aware ? bt : 1.f;
            const float g = a.eta * bp * (1.f - bp * al) / nbar;
#pragma unroll
            for (int i = 0; i < E; ++i) d_step(dh[i], dl[i], rv[i], g, s[i], a.d_min, a.d_max);
        }
        __syncwarp();
    }
    cp_async_wait_0();
#pragma unroll
    for (int i = 0; i < E; ++i) a.d_out[(size_t)bh * K + lane * E + i] = dh[i] + dl[i];
}

template <int K, typename TIn, typename TOut>
cudaError_t launch_k(const OsdnScanArgs& a, cudaStream_t s) {
    dim3 grid((unsigned)(a.B * a.H)), block(32);
    if (a.r && a.r_per_key) scan_warp_kernel<K, TIn, TOut, 2><<<grid, block, 0, s>>>(a);
    else if (a.r) scan_warp_kernel<K, TIn, TOut, 1><<<grid, block, 0, s>>>(a);
    else scan_warp_kernel<K, TIn, TOut, 0><<<grid, block, 0, s>>>(a);
    return cudaGetLastError();
}

template <int K, typename TIn>
cudaError_t launch_out(const OsdnScanArgs& a, cudaStream_t s) {
    switch (a.kt_dtype) {
        case OSDN_F32: return launch_k<K, TIn, float>(a, s);
        case OSDN_BF16: return launch_k<K, TIn, __nv_bfloat16>(a, s);
        case OSDN_F16: return launch_k<K, TIn, __half>(a, s);
    }
    return cudaErrorInvalidValue;
}

template <int K>
cudaError_t launch_in(const OsdnScanArgs& a, cudaStream_t s) {
    switch (a.k_dtype) {
        case OSDN_F32: return launch_out<K, float>(a, s);
        case OSDN_BF16: return launch_out<K, __nv_bfloat16>(a, s);
        case OSDN_F16: return launch_out<K, __half>(a, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace
}  // namespace osdn

cudaError_t osdn_launch_scan(const OsdnScanArgs& a, void* ws, size_t ws_bytes, cudaStream_t s) {
    if (a.K == 128) {
        cudaError_t e = osdn_launch_scan_block(a, ws, ws_bytes, s);  // 16-bit keys: blocked scan
        if (e != cudaErrorNotSupported) return e;
        return osdn::launch_in<128>(a, s);
    }
    if (a.K == 64) return osdn::launch_in<64>(a, s);
    return cudaErrorInvalidValue;
}
