// chunk_simt.cu -- fp32 CUDA-core kernel for phase 2 of OSDN (the preconditioned delta rule).
//
// "OSDN: Improving Delta Rule with Provable Online Preconditioning in Linear Attention",
// Section 4.1 Eq. (2) / Section 4.3 Eq. (5):
//   u_t = v_t - S_{t-1} k_t   (original key: read side)
//   S_t = S_{t-1} + beta_t u_t k~_t^T   (write key)
//   o_t = scale * S_t q_t   (readout after the write)
// With the OSGDN state gate (Appendix B.1, post-gate residual) S_{t-1} is first scaled by
// alpha_t (alpha = 1 without the gate: an exact no-op), or each column i by alpha_{t,i} with one
// gate per key channel (OSKDA, Appendix B.2, in the transpose of its K x V convention).
// This kernel evaluates the recurrence token by token in fp32 (FFMA only), which is exact up to
// fp32 rounding for any input dtype.  It serves fp32 inputs (where bf16/f16 tensor-core
// operands could not meet a 1e-4 tolerance) and the head sizes the tensor-core kernel is not
// built for.  Mapping: one CTA per (batch, head, 32 rows of S); each warp owns 4 rows; a row's
// K entries are spread over the 32 lanes (E = K/32 each).  Per token the dot products <S_i, k>,
// <S_i, q> of every row and <k~, q> share one warp butterfly, and o_t = S_t q is formed as
// <Sbar_i, q> + beta u_i <k~, q>.  Token t+1's operands are loaded while token t is processed.
#include "common.cuh"

namespace osdn {
namespace {

constexpr int kRowsPerCta = 32;
constexpr int kRowsPerWarp = 4;

template <int K, typename TIn>
__global__ void __launch_bounds__(256) chunk_recurrent_kernel(OsdnChunkArgs a) {
    constexpr int E = K / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int bh = blockIdx.x;
    const int b = bh / a.H, h = bh % a.H;
    const int T = a.T, H = a.H, V = a.V;
    const int row_base = blockIdx.y * kRowsPerCta + warp * kRowsPerWarp;
    const TIn* qg = static_cast<const TIn*>(a.q);
    const TIn* kg = static_cast<const TIn*>(a.k);
    const TIn* ktg = static_cast<const TIn*>(a.k_tilde);
    const TIn* vg = static_cast<const TIn*>(a.v);
    TIn* og = static_cast<TIn*>(a.o);

    float S[kRowsPerWarp][E];
#pragma unroll
    for (int j = 0; j < kRowsPerWarp; ++j) {
        const size_t off = ((size_t)bh * V + row_base + j) * K + lane * E;
#pragma unroll
        for (int i = 0; i < E; ++i) S[j][i] = a.S0 ? a.S0[off + i] : 0.f;
    }

    const size_t row0 = (size_t)b * T * H + h;
    float kv[E], ktv[E], qv[E], vv[kRowsPerWarp], bt = 0.f, al[E];
    auto load = [&](int t) {
        const size_t r = row0 + (size_t)t * H;
        VecIO<TIn, E>::load(kg + r * K + lane * E, kv);
        VecIO<TIn, E>::load(ktg + r * K + lane * E, ktv);
        VecIO<TIn, E>::load(qg + r * K + lane * E, qv);
#pragma unroll
        for (int j = 0; j < kRowsPerWarp; ++j) vv[j] = to_f32(vg[r * V + row_base + j]);
        bt = a.beta[r];
        if (a.alpha && a.alpha_per_key) {
            VecIO<float, E>::load(a.alpha + r * K + lane * E, al);
        } else {
#pragma unroll
            for (int i = 0; i < E; ++i) al[i] = a.alpha ? a.alpha[r] : 1.f;
        }
    };
    if (T > 0) load(0);
    for (int t = 0; t < T; ++t) {
        float ck[E], ckt[E], cq[E], cv[kRowsPerWarp];
#pragma unroll
        for (int i = 0; i < E; ++i) { ck[i] = kv[i]; ckt[i] = ktv[i]; cq[i] = qv[i]; }
#pragma unroll
        for (int j = 0; j < kRowsPerWarp; ++j) cv[j] = vv[j];
        const float cb = bt;
        float ca[E];
#pragma unroll
        for (int i = 0; i < E; ++i) ca[i] = al[i];
        if (t + 1 < T) load(t + 1);
        const size_t r = row0 + (size_t)t * H;
        // <S_i, k>, <S_i, q> of the gated state and <k~, q> in one butterfly (independent sums);
        // then S_t q = Sbar q + beta u <k~, q>, so the readout needs no second pass over S
        float sk[kRowsPerWarp], sq[kRowsPerWarp], ktq = 0.f;
#pragma unroll
        for (int i = 0; i < E; ++i) ktq = fmaf(ckt[i], cq[i], ktq);
#pragma unroll
        for (int j = 0; j < kRowsPerWarp; ++j) {
            sk[j] = 0.f;
            sq[j] = 0.f;
#pragma unroll
            for (int i = 0; i < E; ++i) {
                S[j][i] *= ca[i];
                sk[j] = fmaf(S[j][i], ck[i], sk[j]);
                sq[j] = fmaf(S[j][i], cq[i], sq[j]);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            ktq += __shfl_xor_sync(0xffffffffu, ktq, o);
#pragma unroll
            for (int j = 0; j < kRowsPerWarp; ++j) {
                sk[j] += __shfl_xor_sync(0xffffffffu, sk[j], o);
                sq[j] += __shfl_xor_sync(0xffffffffu, sq[j], o);
            }
        }
#pragma unroll
        for (int j = 0; j < kRowsPerWarp; ++j) {
            const float bu = cb * (cv[j] - sk[j]);
#pragma unroll
            for (int i = 0; i < E; ++i) S[j][i] = fmaf(bu, ckt[i], S[j][i]);
            if (lane == 0) og[r * V + row_base + j] = from_f32<TIn>(a.scale * fmaf(bu, ktq, sq[j]));
        }
    }
#pragma unroll
    for (int j = 0; j < kRowsPerWarp; ++j) {
        const size_t off = ((size_t)bh * V + row_base + j) * K + lane * E;
#pragma unroll
        for (int i = 0; i < E; ++i) a.S_out[off + i] = S[j][i];
    }
}

template <int K, typename TIn>
cudaError_t launch_t(const OsdnChunkArgs& a, cudaStream_t s) {
    dim3 grid((unsigned)(a.B * a.H), (unsigned)(a.V / kRowsPerCta)), block(256);
    chunk_recurrent_kernel<K, TIn><<<grid, block, 0, s>>>(a);
    return cudaGetLastError();
}

template <int K>
cudaError_t launch_k(const OsdnChunkArgs& a, cudaStream_t s) {
    switch (a.dtype) {
        case OSDN_F32: return launch_t<K, float>(a, s);
        case OSDN_BF16: return launch_t<K, __nv_bfloat16>(a, s);
        case OSDN_F16: return launch_t<K, __half>(a, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace
}  // namespace osdn

cudaError_t osdn_launch_chunk_simt(const OsdnChunkArgs& a, cudaStream_t s) {
    if (a.V % osdn::kRowsPerCta != 0) return cudaErrorInvalidValue;
    if (a.K == 128) return osdn::launch_k<128>(a, s);
    if (a.K == 64) return osdn::launch_k<64>(a, s);
    return cudaErrorInvalidValue;
}
