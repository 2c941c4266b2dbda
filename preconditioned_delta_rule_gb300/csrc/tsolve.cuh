// tsolve.cuh -- the UT transform of the chunkwise delta rule in fp32 on the CUDA cores.
//
// "OSDN: Improving Delta Rule with Provable Online Preconditioning in Linear Attention",
// Appendix A.2, Eq. (8): T = (I + A)^-1 with A strictly lower triangular (64 x 64),
// A_ij = beta_i <k_i, k~_j> for j < i.  Blocked on 16 x 16 tiles:
//   T_ii = (I + A_ii)^-1                       (forward substitution, one column per thread)
//   T_ij = -T_ii * sum_{m=j}^{i-1} A_im T_mj    (i > j; levels i - j = 1, 2, 3)
// The ten lower-triangular tiles of A and T are stored packed (tile (i, j) at index
// i(i+1)/2 + j), each 16 rows of kTileStride floats (an even stride, so that pairs of columns
// load as float2, and rows fall on distinct banks).  Every loop has compile-time bounds.
// Must be called by 128 threads that share named barrier `bar` (bar 0 with a 128-thread CTA is
// __syncthreads()); it synchronises internally on that barrier.
#pragma once

namespace osdn {

__device__ __forceinline__ void bar_sync128(int bar) { asm volatile("bar.sync %0, 128;\n" ::"r"(bar) : "memory"); }

constexpr int kTileStride = 18;
constexpr int kTile = 16 * kTileStride;  // floats per packed tile

__device__ __forceinline__ constexpr int tile_index(int i, int j) { return i * (i + 1) / 2 + j; }

template <int LAM>
__device__ __forceinline__ void tsolve_level(const float* __restrict__ AM, float* __restrict__ TM,
                                             float* __restrict__ PM, int tid, int bar) {
    constexpr int NB = 4 - LAM;  // tiles on this sub-diagonal
    const int ii = tid >> 3, jj = (tid & 7) * 2;
    float acc[NB][2];
#pragma unroll
    for (int blk = 0; blk < NB; ++blk) {
        acc[blk][0] = 0.f;
        acc[blk][1] = 0.f;
#pragma unroll
        for (int mu = 0; mu < LAM; ++mu) {
            const float* Ar = AM + tile_index(blk + LAM, blk + mu) * kTile + ii * kTileStride;
            const float* Tc = TM + tile_index(blk + mu, blk) * kTile + jj;
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) {
                const float a = Ar[kk];
                const float2 t = *reinterpret_cast<const float2*>(Tc + kk * kTileStride);
                acc[blk][0] = fmaf(a, t.x, acc[blk][0]);
                acc[blk][1] = fmaf(a, t.y, acc[blk][1]);
            }
        }
    }
#pragma unroll
    for (int blk = 0; blk < NB; ++blk)
        *reinterpret_cast<float2*>(PM + blk * kTile + ii * kTileStride + jj) = make_float2(acc[blk][0], acc[blk][1]);
    bar_sync128(bar);
#pragma unroll
    for (int blk = 0; blk < NB; ++blk) {
        const float* Tr = TM + tile_index(blk + LAM, blk + LAM) * kTile + ii * kTileStride;
        const float* Pc = PM + blk * kTile + jj;
        float r0 = 0.f, r1 = 0.f;
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {  // T_ii is lower triangular; its upper half is stored as 0
            const float t = Tr[kk];
            const float2 p = *reinterpret_cast<const float2*>(Pc + kk * kTileStride);
            r0 = fmaf(t, p.x, r0);
            r1 = fmaf(t, p.y, r1);
        }
        *reinterpret_cast<float2*>(TM + tile_index(blk + LAM, blk) * kTile + ii * kTileStride + jj) =
            make_float2(-r0, -r1);
    }
    bar_sync128(bar);
}

// AM: packed strictly-lower A (the diagonal tiles' upper parts may hold anything; only entries
// below the diagonal are read).  TM receives T.  PM is scratch of 3 tiles.  Callers must
// synchronise on `bar` between writing AM and calling this.
__device__ __forceinline__ void ut_inverse_64(const float* __restrict__ AM, float* __restrict__ TM,
                                              float* __restrict__ PM, int tid, int bar = 0) {
    if (tid < 64) {
        const int blk = tid >> 4, c = tid & 15;
        const float* Ab = AM + tile_index(blk, blk) * kTile;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = (i == c) ? 1.f : 0.f;
#pragma unroll
        for (int m = 0; m < 16; ++m)
#pragma unroll
            for (int i = m + 1; i < 16; ++i) x[i] = fmaf(-Ab[i * kTileStride + m], x[m], x[i]);
        float* Tb = TM + tile_index(blk, blk) * kTile;
#pragma unroll
        for (int i = 0; i < 16; ++i) Tb[i * kTileStride + c] = x[i];
    }
    bar_sync128(bar);
    tsolve_level<1>(AM, TM, PM, tid, bar);
    tsolve_level<2>(AM, TM, PM, tid, bar);
    tsolve_level<3>(AM, TM, PM, tid, bar);
}

}  // namespace osdn
