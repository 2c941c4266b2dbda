// tsolve.cuh -- the UT transform of the chunkwise delta rule in fp32 on the CUDA cores.
//
// "OSDN: Improving Delta Rule with Provable Online Preconditioning in Linear Attention",
// Appendix A.2, Eq. (8): T = (I + A)^-1 with A strictly lower triangular (64 x 64),
// A_ij = beta_i <k_i, k~_j> for j < i.  Blocked on 16 x 16 tiles:
//   T_ii = (I + A_ii)^-1                       (forward substitution, one column per thread)
//   A'_im = T_ii A_im                          (i > m; the six tiles at once)
//   T_ij = -sum_{m=j}^{i-1} A'_im T_mj         (i > j; levels i - j = 1, 2, 3)
// (the same T as T_ij = -T_ii sum_m A_im T_mj, with the T_ii product taken out of the levels so
// that each level is one independent pass).
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
constexpr int kUtScratchTiles = 6;       // tiles of scratch ut_inverse_64 needs

__device__ __forceinline__ constexpr int tile_index(int i, int j) { return i * (i + 1) / 2 + j; }
// scratch slot of A'_im (i > m): (1,0) (2,0) (2,1) (3,0) (3,1) (3,2) -> 0 .. 5
__device__ __forceinline__ constexpr int prime_index(int i, int m) { return tile_index(i, m) - i; }

// Level LAM: T_{b+LAM, b} = -sum_{mu < LAM} A'_{b+LAM, b+mu} T_{b+mu, b} for the 4 - LAM tiles of
// the sub-diagonal; thread (ii, jj) forms row ii, columns jj and jj + 1 of each.
template <int LAM>
__device__ __forceinline__ void tsolve_level(const float* __restrict__ PM, float* __restrict__ TM, int tid, int bar) {
    constexpr int NB = 4 - LAM;
    const int ii = tid >> 3, jj = (tid & 7) * 2;
    float acc[NB][2];
#pragma unroll
    for (int blk = 0; blk < NB; ++blk) {
        acc[blk][0] = 0.f;
        acc[blk][1] = 0.f;
#pragma unroll
        for (int mu = 0; mu < LAM; ++mu) {
            const float* Ar = PM + prime_index(blk + LAM, blk + mu) * kTile + ii * kTileStride;
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
        *reinterpret_cast<float2*>(TM + tile_index(blk + LAM, blk) * kTile + ii * kTileStride + jj) =
            make_float2(-acc[blk][0], -acc[blk][1]);
    bar_sync128(bar);
}

// AM: packed strictly-lower A (the diagonal tiles' upper parts may hold anything; only entries
// below the diagonal are read).  TM receives T.  PM is scratch of kUtScratchTiles tiles.  Callers
// must synchronise on `bar` between writing AM and calling this.
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
    {  // A'_im = T_ii A_im for the six off-diagonal tiles (T_ii is lower triangular, zeros above)
        const int ii = tid >> 3, jj = (tid & 7) * 2;
        float acc[6][2];
#pragma unroll
        for (int t = 0; t < 6; ++t) {
            acc[t][0] = 0.f;
            acc[t][1] = 0.f;
        }
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            const float t1 = TM[tile_index(1, 1) * kTile + ii * kTileStride + kk];
            const float t2 = TM[tile_index(2, 2) * kTile + ii * kTileStride + kk];
            const float t3 = TM[tile_index(3, 3) * kTile + ii * kTileStride + kk];
            const float2 a10 = *reinterpret_cast<const float2*>(AM + tile_index(1, 0) * kTile + kk * kTileStride + jj);
            const float2 a20 = *reinterpret_cast<const float2*>(AM + tile_index(2, 0) * kTile + kk * kTileStride + jj);
            const float2 a21 = *reinterpret_cast<const float2*>(AM + tile_index(2, 1) * kTile + kk * kTileStride + jj);
            const float2 a30 = *reinterpret_cast<const float2*>(AM + tile_index(3, 0) * kTile + kk * kTileStride + jj);
            const float2 a31 = *reinterpret_cast<const float2*>(AM + tile_index(3, 1) * kTile + kk * kTileStride + jj);
            const float2 a32 = *reinterpret_cast<const float2*>(AM + tile_index(3, 2) * kTile + kk * kTileStride + jj);
            acc[0][0] = fmaf(t1, a10.x, acc[0][0]);
            acc[0][1] = fmaf(t1, a10.y, acc[0][1]);
            acc[1][0] = fmaf(t2, a20.x, acc[1][0]);
            acc[1][1] = fmaf(t2, a20.y, acc[1][1]);
            acc[2][0] = fmaf(t2, a21.x, acc[2][0]);
            acc[2][1] = fmaf(t2, a21.y, acc[2][1]);
            acc[3][0] = fmaf(t3, a30.x, acc[3][0]);
            acc[3][1] = fmaf(t3, a30.y, acc[3][1]);
            acc[4][0] = fmaf(t3, a31.x, acc[4][0]);
            acc[4][1] = fmaf(t3, a31.y, acc[4][1]);
            acc[5][0] = fmaf(t3, a32.x, acc[5][0]);
            acc[5][1] = fmaf(t3, a32.y, acc[5][1]);
        }
#pragma unroll
        for (int t = 0; t < 6; ++t)
            *reinterpret_cast<float2*>(PM + t * kTile + ii * kTileStride + jj) = make_float2(acc[t][0], acc[t][1]);
    }
    bar_sync128(bar);
    tsolve_level<1>(PM, TM, tid, bar);
    tsolve_level<2>(PM, TM, tid, bar);
    tsolve_level<3>(PM, TM, tid, bar);
}

// ---- the same inverse with T's off-diagonal tiles stored over A's --------------------------------
// A's off-diagonal tiles are dead once A'_im = T_ii A_im is formed, so T_ij (i > j) overwrites A_ij
// and only T's four diagonal tiles need room of their own (TD, 4 tiles).  After the call, tile
// (i, j) of T is ut_tile(AM, TD, i, j).  Same arithmetic, order and barriers as ut_inverse_64.
__device__ __forceinline__ float* ut_tile(float* AM, float* TD, int i, int j) {
    return i == j ? TD + i * kTile : AM + tile_index(i, j) * kTile;
}
template <int LAM>
__device__ __forceinline__ void tsolve_level_aliased(const float* __restrict__ PM, float* AM, float* TD, int tid, int bar) {
    constexpr int NB = 4 - LAM;
    const int ii = tid >> 3, jj = (tid & 7) * 2;
    float acc[NB][2];
#pragma unroll
    for (int blk = 0; blk < NB; ++blk) {
        acc[blk][0] = 0.f;
        acc[blk][1] = 0.f;
#pragma unroll
        for (int mu = 0; mu < LAM; ++mu) {
            const float* Ar = PM + prime_index(blk + LAM, blk + mu) * kTile + ii * kTileStride;
            const float* Tc = ut_tile(AM, TD, blk + mu, blk) + jj;
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
        *reinterpret_cast<float2*>(ut_tile(AM, TD, blk + LAM, blk) + ii * kTileStride + jj) =
            make_float2(-acc[blk][0], -acc[blk][1]);
    bar_sync128(bar);
}
__device__ __forceinline__ void ut_inverse_64_aliased(float* AM, float* TD, float* __restrict__ PM, int tid, int bar) {
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
        float* Tb = TD + blk * kTile;
#pragma unroll
        for (int i = 0; i < 16; ++i) Tb[i * kTileStride + c] = x[i];
    }
    bar_sync128(bar);
    {  // A'_im = T_ii A_im for the six off-diagonal tiles
        const int ii = tid >> 3, jj = (tid & 7) * 2;
        float acc[6][2];
#pragma unroll
        for (int t = 0; t < 6; ++t) {
            acc[t][0] = 0.f;
            acc[t][1] = 0.f;
        }
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            const float t1 = TD[1 * kTile + ii * kTileStride + kk];
            const float t2 = TD[2 * kTile + ii * kTileStride + kk];
            const float t3 = TD[3 * kTile + ii * kTileStride + kk];
            const float2 a10 = *reinterpret_cast<const float2*>(AM + tile_index(1, 0) * kTile + kk * kTileStride + jj);
            const float2 a20 = *reinterpret_cast<const float2*>(AM + tile_index(2, 0) * kTile + kk * kTileStride + jj);
            const float2 a21 = *reinterpret_cast<const float2*>(AM + tile_index(2, 1) * kTile + kk * kTileStride + jj);
            const float2 a30 = *reinterpret_cast<const float2*>(AM + tile_index(3, 0) * kTile + kk * kTileStride + jj);
            const float2 a31 = *reinterpret_cast<const float2*>(AM + tile_index(3, 1) * kTile + kk * kTileStride + jj);
            const float2 a32 = *reinterpret_cast<const float2*>(AM + tile_index(3, 2) * kTile + kk * kTileStride + jj);
            acc[0][0] = fmaf(t1, a10.x, acc[0][0]);
            acc[0][1] = fmaf(t1, a10.y, acc[0][1]);
            acc[1][0] = fmaf(t2, a20.x, acc[1][0]);
            acc[1][1] = fmaf(t2, a20.y, acc[1][1]);
            acc[2][0] = fmaf(t2, a21.x, acc[2][0]);
            acc[2][1] = fmaf(t2, a21.y, acc[2][1]);
            acc[3][0] = fmaf(t3, a30.x, acc[3][0]);
            acc[3][1] = fmaf(t3, a30.y, acc[3][1]);
            acc[4][0] = fmaf(t3, a31.x, acc[4][0]);
            acc[4][1] = fmaf(t3, a31.y, acc[4][1]);
            acc[5][0] = fmaf(t3, a32.x, acc[5][0]);
            acc[5][1] = fmaf(t3, a32.y, acc[5][1]);
        }
#pragma unroll
        for (int t = 0; t < 6; ++t)
            *reinterpret_cast<float2*>(PM + t * kTile + ii * kTileStride + jj) = make_float2(acc[t][0], acc[t][1]);
    }
    bar_sync128(bar);
    tsolve_level_aliased<1>(PM, AM, TD, tid, bar);
    tsolve_level_aliased<2>(PM, AM, TD, tid, bar);
    tsolve_level_aliased<3>(PM, AM, TD, tid, bar);
}

}  // namespace osdn
