// decode.cu -- one recurrent OSDN token for every (batch, head), in place on S and d.
//
// "OSDN: Improving Delta Rule with Provable Online Preconditioning in Linear Attention":
// Algorithm 2 (parts 2a and 2b for a single token) with the APF gate of Eq. (7); the pages'
// own decode path is a fused single-token kernel (Appendix L).  For one head:
//   k~ = d . k (old d);  d <- clip(r d + eta b (1 - b <d, k.k>) / max(|k|^2, eps) * k.k)
//   u_i = v_i - <S_i, k>;  S_i <- S_i + beta u_i k~;  o_i = <S_i_new, q'> = <S_i, q'> + beta u_i <k~, q'>
// with q' = scale * q, for every row i of S (rows are independent given k, k~, q).  With the OSGDN
// state gate (Appendix B.1, post-gate residual) S is first scaled by alpha: S <- alpha S, then the
// same step (alpha = 1 without the gate: an exact no-op); with one gate per key channel (OSKDA,
// Appendix B.2, the state stored as the transpose of its K x V convention) column i of S is scaled
// by alpha_i.
//
// The step is HBM-bound: S (V x K fp32) is read once and written once.  One CTA of 256 threads
// per head; 8 lanes per row, each lane holding 4-float pieces interleaved so that every load
// and store instruction of a warp covers four full 128-byte row segments.  All rows of a
// thread are loaded before any is used, and before the phase-1 step is computed (only that step's
// own operands are requested earlier), so that each thread keeps its loads in flight together and
// their latency overlaps the step's.  k and q (with the
// gate folded in) are held in registers; k~ and the gate are read from shared memory in the store
// loop, which keeps the kernel within the 128 registers a thread that two resident CTAs per SM
// allow.
#include "common.cuh"

namespace osdn {
namespace {

constexpr int kThreads = 256;
constexpr int kLanesPerRow = 8;

__device__ __forceinline__ float4 ld_stream(const float* p) {
    float4 v;
    asm volatile("ld.global.cs.v4.f32 {%0,%1,%2,%3}, [%4];\n"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ void st_stream(float* p, float4 v) {
    asm volatile("st.global.cs.v4.f32 [%0], {%1,%2,%3,%4};\n" ::"l"(p), "f"(v.x), "f"(v.y),
                 "f"(v.z), "f"(v.w) : "memory");
}

// RMODE: 0 no retention, 1 one per head (Eq. (7)), 2 one per key coordinate (diag(r_t), Appendix A.5)
template <int K, int V, typename TIn, int RMODE>
__global__ void __launch_bounds__(kThreads, 2) decode_kernel(OsdnDecodeArgs a) {
    constexpr int P4 = K / 4 / kLanesPerRow;        // float4 pieces per lane per row (4 or 2)
    constexpr int ROWS_PER_PASS = kThreads / kLanesPerRow;  // 32
    constexpr int PASSES = V / ROWS_PER_PASS;        // 4 or 2
    constexpr int E = K / 32;
    // sk, sq: k and scale * q with the state gate of their column folded in (<alpha o S_i, k> =
    // <S_i, alpha o k>); sga: the gate of each column (1 without one); skt: k~
    __shared__ __align__(16) float sk[K], skt[K], sq[K], sga[K];
    __shared__ float scoef[2];

    const int tid = threadIdx.x;
    const size_t bh = blockIdx.x;
    float* S = a.S + bh * (size_t)V * K;
    const int sub = tid % kLanesPerRow;
    const int rg = tid / kLanesPerRow;

    // Warp 0's operands of the phase-1 step are loaded first, then every thread's slice of the
    // state (which does not depend on the step), so that the step's loads do not queue behind the
    // state's and its latency overlaps theirs.
    float kv[E], qv[E], dv[E], gv[E], rv[E], bt0 = 0.f;
    if (tid < 32) {
        VecIO<TIn, E>::load(static_cast<const TIn*>(a.k) + bh * K + tid * E, kv);
        VecIO<TIn, E>::load(static_cast<const TIn*>(a.q) + bh * K + tid * E, qv);
        VecIO<float, E>::load(a.d + bh * K + tid * E, dv);
        if (a.alpha && a.alpha_per_key) {
            VecIO<float, E>::load(a.alpha + bh * K + tid * E, gv);
        } else {
            const float g1 = a.alpha ? a.alpha[bh] : 1.f;
#pragma unroll
            for (int i = 0; i < E; ++i) gv[i] = g1;
        }
        if (RMODE == 2) {
            VecIO<float, E>::load(a.r + bh * K + tid * E, rv);
        } else {
            const float r1 = RMODE == 1 ? a.r[bh] : 1.f;
#pragma unroll
            for (int i = 0; i < E; ++i) rv[i] = r1;
        }
        bt0 = a.beta[bh];
    }
    float4 Sr[PASSES][P4];
#pragma unroll
    for (int ps = 0; ps < PASSES; ++ps) {
        const int row = ps * ROWS_PER_PASS + rg;
#pragma unroll
        for (int c = 0; c < P4; ++c) Sr[ps][c] = ld_stream(S + (size_t)row * K + (c * kLanesPerRow + sub) * 4);
    }

    if (tid < 32) {  // warp 0: phase-1 step of this head, and the shared vectors
        float n = 0.f, al = 0.f, ktq = 0.f, s[E];
#pragma unroll
        for (int i = 0; i < E; ++i) {
            s[i] = kv[i] * kv[i];
            n += s[i];
            al = fmaf(dv[i], s[i], al);
            const float kt = dv[i] * kv[i];
            const float qs = a.scale * qv[i];
            ktq = fmaf(kt, qs, ktq);
            sk[tid * E + i] = gv[i] * kv[i];
            skt[tid * E + i] = kt;
            sq[tid * E + i] = gv[i] * qs;
            sga[tid * E + i] = gv[i];
        }
        n = warp_sum(n);
        al = warp_sum(al);
        ktq = warp_sum(ktq);
        const float bp = a.beta_aware ? bt0 : 1.f;
        const float g = a.eta * bp * (1.f - bp * al) / fmaxf(n, a.eps);
        float dn[E];
#pragma unroll
        for (int i = 0; i < E; ++i) dn[i] = fminf(fmaxf(fmaf(g, s[i], rv[i] * dv[i]), a.d_min), a.d_max);
        VecIO<float, E>::store(a.d + bh * K + tid * E, dn);
        if (tid == 0) {
            scoef[0] = bt0;
            scoef[1] = bt0 * ktq;
        }
    }
    __syncthreads();

    const float bt = scoef[0], bktq = scoef[1];
    float4 kr[P4], qr[P4];
#pragma unroll
    for (int c = 0; c < P4; ++c) {
        const int col = (c * kLanesPerRow + sub) * 4;
        kr[c] = *reinterpret_cast<const float4*>(sk + col);
        qr[c] = *reinterpret_cast<const float4*>(sq + col);
    }
    const TIn* vp = static_cast<const TIn*>(a.v) + bh * V;
    TIn* op = static_cast<TIn*>(a.o) + bh * V;
#pragma unroll
    for (int ps = 0; ps < PASSES; ++ps) {
        const int row = ps * ROWS_PER_PASS + rg;
        float dk = 0.f, dq = 0.f;
#pragma unroll
        for (int c = 0; c < P4; ++c) {
            const float4 x = Sr[ps][c];
            const float4 kk = kr[c];
            const float4 qq = qr[c];
            dk = fmaf(x.x, kk.x, fmaf(x.y, kk.y, fmaf(x.z, kk.z, fmaf(x.w, kk.w, dk))));
            dq = fmaf(x.x, qq.x, fmaf(x.y, qq.y, fmaf(x.z, qq.z, fmaf(x.w, qq.w, dq))));
        }
#pragma unroll
        for (int o = kLanesPerRow / 2; o > 0; o >>= 1) {
            dk += __shfl_xor_sync(0xffffffffu, dk, o);
            dq += __shfl_xor_sync(0xffffffffu, dq, o);
        }
        const float u = to_f32(vp[row]) - dk;
        const float bu = bt * u;
#pragma unroll
        for (int c = 0; c < P4; ++c) {
            const int col = (c * kLanesPerRow + sub) * 4;
            const float4 kt = *reinterpret_cast<const float4*>(skt + col);
            const float4 ga = *reinterpret_cast<const float4*>(sga + col);
            float4 x = Sr[ps][c];
            x.x = fmaf(bu, kt.x, ga.x * x.x);
            x.y = fmaf(bu, kt.y, ga.y * x.y);
            x.z = fmaf(bu, kt.z, ga.z * x.z);
            x.w = fmaf(bu, kt.w, ga.w * x.w);
            st_stream(S + (size_t)row * K + col, x);
        }
        if (sub == 0) op[row] = from_f32<TIn>(fmaf(bktq, u, dq));
    }
}

template <int K, int V, typename TIn>
cudaError_t launch3(const OsdnDecodeArgs& a, cudaStream_t s) {
    dim3 grid((unsigned)(a.B * a.H)), block(kThreads);
    if (a.r && a.r_per_key) decode_kernel<K, V, TIn, 2><<<grid, block, 0, s>>>(a);
    else if (a.r) decode_kernel<K, V, TIn, 1><<<grid, block, 0, s>>>(a);
    else decode_kernel<K, V, TIn, 0><<<grid, block, 0, s>>>(a);
    return cudaGetLastError();
}

template <int K, int V>
cudaError_t launch2(const OsdnDecodeArgs& a, cudaStream_t s) {
    switch (a.dtype) {
        case OSDN_F32: return launch3<K, V, float>(a, s);
        case OSDN_BF16: return launch3<K, V, __nv_bfloat16>(a, s);
        case OSDN_F16: return launch3<K, V, __half>(a, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace
}  // namespace osdn

cudaError_t osdn_launch_decode(const OsdnDecodeArgs& a, cudaStream_t s) {
    if (a.K == 128 && a.V == 128) return osdn::launch2<128, 128>(a, s);
    if (a.K == 128 && a.V == 64) return osdn::launch2<128, 64>(a, s);
    if (a.K == 64 && a.V == 128) return osdn::launch2<64, 128>(a, s);
    if (a.K == 64 && a.V == 64) return osdn::launch2<64, 64>(a, s);
    return cudaErrorInvalidValue;
}
