// chunk_tc.cu -- tensor-core kernel for phase 2 of OSDN: the chunkwise preconditioned delta rule.
//
// "OSDN: Improving Delta Rule with Provable Online Preconditioning in Linear Attention",
// Section 4.3 (Eqs. (5)-(6)) and Appendix A.2 (Eqs. (8)-(11)).  For one chunk of C = 64 tokens
// with keys K, write keys K~ (C x K), values V (C x V), queries Q and gates beta:
//   A  = tril(diag(beta) K K~^T, -1)            (Gram with the write key, Eq. (6))
//   T  = (I + A)^-1,  T' = T diag(beta)          (UT transform, Eq. (8); fp32 forward substitution)
//   W  = T' K,  U = T' V                         (Eq. (9): the read key stays in W)
//   X  = U - W S^T                               (the chunk's scaled residuals)
//   O  = scale * (Q S^T + tril(Q K~^T, 0) X)     (readout after each write: the diagonal is kept)
//   S <- S + X^T K~                              (Eq. (11))
// with S carried across chunks in fp32.
//
// Design (one CTA per (batch, head, 64 rows of S); rows of S evolve independently given K, K~,
// beta, so the V dimension splits across CTAs with no exchange):
//   * TMA (128-byte swizzle) brings the K, Q, K~, V tiles of chunk n+1 into the other of two
//     shared-memory stages while chunk n is processed.
//   * Operands are fp16 (10-bit mantissa): bf16 inputs are converted in place (exact for
//     normal-range values); computed operands (T', W, S, X, L) are rounded to fp16.  All
//     products accumulate in fp32 in tensor memory.  fp16 rather than bf16 operands keep the
//     o/S error ~8x smaller at no extra tensor-core work.
//   * Every product is one tcgen05.mma group with M = 128, stacking two 64-row operands:
//       [K; Q] K~^T            -> lanes 0-63: K K~^T (Gram),  lanes 64-127: Q K~^T (scores)
//       [0; T'] K, [0; T'] V   -> lanes 64-127: W, U
//       [Q; -W] S^T   (+= U)   -> lanes 0-63: Q S^T,        lanes 64-127: X = U - W S^T
//       [L; 0] X      (+=)     -> lanes 0-63: O
//       K~^T X        (+= S^T) -> S^T accumulated in tensor memory (fp32, lanes = key dim)
//   * The triangular inverse is blocked (16 x 16 diagonal blocks by forward substitution, then
//     three levels of block products) in fp32 on the CUDA cores.
// All waits on mbarriers are bounded; on expiry the kernel records a timeout (reported by
// osdn_check), drains what it issued and exits.
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "scan_block_body.cuh"
#include "tc_ptx.cuh"
#include "tmap.cuh"
#include "tsolve.cuh"

namespace osdn {
// Set by any kernel of this library whose bounded device-side wait gave up.
__device__ unsigned int g_timeout_flag = 0;
// Set by the 16-bit tensor-core kernels when an output (o or the final S) is not finite: an fp16
// operand (input, state copy or intermediate) left fp16's range, and the call's results are invalid.
__device__ unsigned int g_range_flag = 0;

namespace {

constexpr int C = 64;          // chunk length
constexpr int KD = 128;        // key dim
constexpr int VS = 64;         // rows of S (value dims) per CTA
constexpr int NTHREADS = 128;
constexpr uint32_t kMaxPolls = 1u << 22;

namespace fused {
// shared memory map (byte offsets from a 1024-byte-aligned base)
constexpr uint32_t KQW_KB = 3 * 8192;                 // per 64-wide key block: K | Q | -W
constexpr uint32_t ST_KQW = 0;
constexpr uint32_t ST_KT = 2 * KQW_KB;                // 49152: K~, 2 key blocks
constexpr uint32_t ST_V = ST_KT + 2 * 8192;           // 65536: V slice
constexpr uint32_t STAGE = ST_V + (VS / 64) * 8192;   // 73728
constexpr uint32_t OFF_LZT = 2 * STAGE;               // L | zeros | T'  (8 KB each)
constexpr uint32_t OFF_X = OFF_LZT + 3 * 8192;
constexpr uint32_t OFF_SS = OFF_X + (VS / 64) * 8192;  // fp16 copy of S (MN-major B operand)
constexpr uint32_t OFF_AM = OFF_SS + (VS / 64) * KD * 128;
constexpr uint32_t OFF_TM = OFF_AM + 10 * kTile * 4;   // 10 packed lower-triangular tiles
constexpr uint32_t OFF_PM = OFF_TM + 10 * kTile * 4;
constexpr uint32_t OFF_BETA = OFF_PM + kUtScratchTiles * kTile * 4;
constexpr uint32_t OFF_BAR = OFF_BETA + 2 * C * 4;
constexpr uint32_t SMEM_USED = OFF_BAR + 64;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;
static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
static_assert(OFF_LZT % 1024 == 0 && OFF_X % 1024 == 0 && OFF_SS % 1024 == 0, "swizzle atoms");
constexpr uint32_t TMA_BYTES = 2 * 2 * 8192 + 2 * 8192 + (VS / 64) * 8192;

// tensor-memory columns
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_G = 0, COL_W = 64, COL_R = 192, COL_ST = 256;
}  // namespace fused

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// True when any of the 32 values is inf or NaN (one pass of compares, no branches).
__device__ __forceinline__ bool any_nonfinite32(const float (&v)[32]) {
    bool bad = false;
#pragma unroll
    for (int j = 0; j < 32; ++j) bad |= !isfinite(v[j]);
    return bad;
}
// Write 8 consecutive values as fp16 into chunk `c` of row `r` of a swizzled atom stack.
__device__ __forceinline__ void st_row_chunk(unsigned char* base, uint32_t r, uint32_t c,
                                             const float* v) {
    uint4 u;
    u.x = pack_h2(v[0], v[1]);
    u.y = pack_h2(v[2], v[3]);
    u.z = pack_h2(v[4], v[5]);
    u.w = pack_h2(v[6], v[7]);
    *reinterpret_cast<uint4*>(base + tc::sw128_off(r, c)) = u;
}

template <typename TIn>
__global__ void __launch_bounds__(NTHREADS, 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmKT, const __grid_constant__ CUtensorMap tmV,
                const float* __restrict__ beta, const float* S0, TIn* __restrict__ out,
                float* S_out, int T, int H, int V, float scale) {
    using namespace fused;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int tid = threadIdx.x, warp = tid >> 5;
    const int bh = blockIdx.x, b = bh / H, h = bh % H;
    const int v0 = blockIdx.y * VS;
    const int N = T / C;

    float* AM = reinterpret_cast<float*>(sm + OFF_AM);
    float* TM = reinterpret_cast<float*>(sm + OFF_TM);
    float* PM = reinterpret_cast<float*>(sm + OFF_PM);
    float* sbeta = reinterpret_cast<float*>(sm + OFF_BETA);
    const uint32_t bar_tma0 = tc::smem_u32(sm + OFF_BAR);
    const uint32_t bar_mma = tc::smem_u32(sm + OFF_BAR + 16);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_BAR + 24);
    const uint32_t sbase = tc::smem_u32(sm);
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;

    // ---- set-up: barriers, zero block, tensor memory, initial state ------------------------
    if (tid == 0) {
        tc::mbar_init(bar_tma0, 1);
        tc::mbar_init(bar_tma0 + 8, 1);
        tc::mbar_init(bar_mma, 1);
        tc::mbar_init_fence();
        tc::prefetch_tmap(&tmQ);
        tc::prefetch_tmap(&tmK);
        tc::prefetch_tmap(&tmKT);
        tc::prefetch_tmap(&tmV);
    }
    for (int e = tid; e < 8192 / 16; e += NTHREADS)
        reinterpret_cast<uint4*>(sm + OFF_LZT + 8192)[e] = make_uint4(0, 0, 0, 0);
    __syncthreads();
    if (warp == 0) tc::tmem_alloc(tc::smem_u32(tmem_slot), TMEM_COLS);

    auto issue_tma = [&](int m, int s) {
        const uint32_t bar = bar_tma0 + 8 * s;
        const uint32_t st = sbase + s * STAGE;
        const int row = b * T + m * C;
        tc::mbar_expect_tx(bar, TMA_BYTES);
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
            tc::tma_load_3d(st + ST_KQW + kb * KQW_KB, &tmK, bar, kb * 64, h, row);
            tc::tma_load_3d(st + ST_KQW + kb * KQW_KB + 8192, &tmQ, bar, kb * 64, h, row);
            tc::tma_load_3d(st + ST_KT + kb * 8192, &tmKT, bar, kb * 64, h, row);
        }
#pragma unroll
        for (int vb = 0; vb < VS / 64; ++vb)
            tc::tma_load_3d(st + ST_V + vb * 8192, &tmV, bar, v0 + vb * 64, h, row);
    };
    if (tid == 0 && N > 0) issue_tma(0, 0);
    if (tid < C && N > 0) sbeta[tid] = beta[(static_cast<size_t>(b) * T + tid) * H + h];

    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tbase = *tmem_slot;

    {  // S0 slice -> S^T in tensor memory (lane = key coordinate) and its fp16 operand copy
        const int k = tid;
        float sv[32];
#pragma unroll
        for (int half = 0; half < VS / 32; ++half) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int v = half * 32 + j;
                sv[j] = S0 ? S0[(static_cast<size_t>(bh) * V + v0 + v) * KD + k] : 0.f;
            }
            tc::tmem_st32(tbase + lane_base + COL_ST + half * 32, sv);
#pragma unroll
            for (int c = 0; c < 4; ++c)
                st_row_chunk(sm + OFF_SS + ((half * 32) / 64) * (KD * 128), k, ((half * 32) % 64) / 8 + c,
                             sv + 8 * c);
        }
        tc::tmem_st_wait();
    }
    tc::fence_proxy_async();
    tc::tc_fence_before();
    __syncthreads();

    uint32_t mph = 0;
    bool aborted = false;
    bool nonfinite = false;  // an output of this thread was inf or NaN
    bool tma_pending[2] = {N > 0, false};
    int tma_chunk[2] = {0, 0};  // chunk index of the load last issued into each stage
    bool mma_pending = false;
    auto wait_mma = [&]() -> bool {
        const bool ok = tc::mbar_wait(bar_mma, mph, kMaxPolls);
        const bool all = __syncthreads_and(ok);
        if (all) {
            mph ^= 1u;
            mma_pending = false;
            tc::tc_fence_after();
        }
        return all;
    };

    const uint32_t id_gram = tc::idesc_f16_f32(128, C, false, false);
    const uint32_t id_wk = tc::idesc_f16_f32(128, KD, false, true);
    const uint32_t id_uv = tc::idesc_f16_f32(128, VS, false, true);
    const uint32_t id_chain = tc::idesc_f16_f32(128, VS, false, true);
    const uint32_t id_state = tc::idesc_f16_f32(128, VS, true, true);

    for (int n = 0; n < N; ++n) {
        const int s = n & 1;
        unsigned char* stg = sm + s * STAGE;
        const uint32_t stg_a = sbase + s * STAGE;
        // 1. prefetch chunk n+1 (its stage was last read by chunk n-1, fully retired)
        if (tid == 0 && n + 1 < N) issue_tma(n + 1, s ^ 1);
        if (n + 1 < N) {
            tma_pending[s ^ 1] = true;
            tma_chunk[s ^ 1] = n + 1;
        }
        float beta_next = 0.f;
        if (tid < C && n + 1 < N)
            beta_next = beta[(static_cast<size_t>(b) * T + (n + 1) * C + tid) * H + h];

        // 2. wait for this chunk's tiles
        {
            const bool ok = tc::mbar_wait(bar_tma0 + 8 * s, (n >> 1) & 1, kMaxPolls);
            if (!__syncthreads_and(ok)) { aborted = true; break; }
            tma_pending[s] = false;
        }
        // 3. bf16 -> fp16 in place (K, Q, K~, V)
        if constexpr (!std::is_same<TIn, __half>::value) {
            for (int e = tid; e < 3584; e += NTHREADS) {
                uint32_t off;
                if (e < 2048) off = ST_KQW + (e >> 10) * KQW_KB + (e & 1023) * 16;
                else if (e < 3072) off = ST_KT + (e - 2048) * 16;
                else off = ST_V + (e - 3072) * 16;
                uint4* p = reinterpret_cast<uint4*>(stg + off);
                uint4 u = *p;
                uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    w[i] = pack_h2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
                *p = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
        tc::fence_proxy_async();
        __syncthreads();

        // 4. [K; Q] K~^T
        if (tid == 0) {
            tc::tc_fence_after();
#pragma unroll
            for (int st = 0; st < KD / 16; ++st) {
                const uint64_t a = tc::sdesc_sw128(stg_a + ST_KQW + (st >> 2) * KQW_KB + (st & 3) * 32, 16, 1024);
                const uint64_t bd = tc::sdesc_sw128(stg_a + ST_KT + (st >> 2) * 8192 + (st & 3) * 32, 16, 1024);
                tc::mma_f16(tbase + COL_G, a, bd, id_gram, st > 0);
            }
            tc::mma_commit(bar_mma);
        }
        mma_pending = true;
        if (!wait_mma()) { aborted = true; break; }

        // 5. A rows (lanes 0-63) to fp32 blocks; score rows L (lanes 64-127) to fp16
        {
            float g[64];
            tc::tmem_ld32(tbase + lane_base + COL_G, *reinterpret_cast<float(*)[32]>(g));
            tc::tmem_ld32(tbase + lane_base + COL_G + 32, *reinterpret_cast<float(*)[32]>(g + 32));
            tc::tmem_ld_wait();
            if (tid < C) {
                const int i = tid, bi = i >> 4, r = i & 15;
                const float bt = sbeta[s * C + i];
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    const int bj = j >> 4;
                    if (bj <= bi) AM[tile_index(bi, bj) * kTile + r * kTileStride + (j & 15)] = (j < i) ? bt * g[j] : 0.f;
                }
            } else {
                const int i = tid - C;
#pragma unroll
                for (int j = 0; j < 64; ++j) g[j] = (j <= i) ? g[j] : 0.f;
#pragma unroll
                for (int c = 0; c < 8; ++c) st_row_chunk(sm + OFF_LZT, i, c, g + 8 * c);
            }
        }
        tc::tc_fence_before();
        __syncthreads();

        // 6. T = (I + A)^-1 in fp32 (blocked forward substitution)
        ut_inverse_64(AM, TM, PM, tid);
        // T' = T diag(beta) -> fp16 rows of the [0; T'] operand
        {
            const int i = tid >> 1, half = tid & 1, bi = i >> 4, r = i & 15;
            float t[32];
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const int j = half * 32 + jj, bj = j >> 4;
                const float tv = (bj <= bi) ? TM[tile_index(bi, bj) * kTile + r * kTileStride + (j & 15)] : 0.f;
                t[jj] = tv * sbeta[s * C + j];
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) st_row_chunk(sm + OFF_LZT + 16384, i, half * 4 + c, t + 8 * c);
        }
        tc::fence_proxy_async();
        __syncthreads();

        // 7. W = T' K (lanes 64-127 of COL_W), U = T' V (lanes 64-127 of COL_R)
        if (tid == 0) {
            tc::tc_fence_after();
#pragma unroll
            for (int st = 0; st < C / 16; ++st) {
                const uint64_t a = tc::sdesc_sw128(sbase + OFF_LZT + 8192 + st * 32, 16, 1024);
                const uint64_t bk = tc::sdesc_sw128(stg_a + ST_KQW + st * 2048, KQW_KB, 1024);
                tc::mma_f16(tbase + COL_W, a, bk, id_wk, st > 0);
                const uint64_t bv = tc::sdesc_sw128(stg_a + ST_V + st * 2048, 8192, 1024);
                tc::mma_f16(tbase + COL_R, a, bv, id_uv, st > 0);
            }
            tc::mma_commit(bar_mma);
        }
        mma_pending = true;
        if (!wait_mma()) { aborted = true; break; }

        // 8. -W -> fp16 rows under Q in each key block
        if (tid >= C) {
            const int c = tid - C;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                float w[32];
                tc::tmem_ld32(tbase + lane_base + COL_W + q4 * 32, w);
                tc::tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) w[j] = -w[j];
                const int kb = q4 >> 1;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
                    st_row_chunk(stg + ST_KQW + kb * KQW_KB + 16384, c, (q4 & 1) * 4 + cc, w + 8 * cc);
            }
        }
        tc::fence_proxy_async();
        tc::tc_fence_before();
        __syncthreads();

        // 9. [Q; -W] S^T accumulated onto [0; U]
        if (tid == 0) {
            tc::tc_fence_after();
#pragma unroll
            for (int st = 0; st < KD / 16; ++st) {
                const uint64_t a = tc::sdesc_sw128(stg_a + ST_KQW + (st >> 2) * KQW_KB + 8192 + (st & 3) * 32, 16, 1024);
                const uint64_t bs = tc::sdesc_sw128(sbase + OFF_SS + st * 2048, KD * 128, 1024);
                tc::mma_f16(tbase + COL_R, a, bs, id_chain, 1);
            }
            tc::mma_commit(bar_mma);
        }
        mma_pending = true;
        if (!wait_mma()) { aborted = true; break; }

        // 10. X rows (lanes 64-127) -> fp16 operand
        if (tid >= C) {
            const int c = tid - C;
#pragma unroll
            for (int q2 = 0; q2 < VS / 32; ++q2) {
                float x[32];
                tc::tmem_ld32(tbase + lane_base + COL_R + q2 * 32, x);
                tc::tmem_ld_wait();
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
                    st_row_chunk(sm + OFF_X + ((q2 * 32) / 64) * 8192, c, ((q2 * 32) % 64) / 8 + cc, x + 8 * cc);
            }
        }
        tc::fence_proxy_async();
        tc::tc_fence_before();
        __syncthreads();

        // 11. O += L X (lanes 0-63 of COL_R);  S^T += K~^T X
        if (tid == 0) {
            tc::tc_fence_after();
#pragma unroll
            for (int st = 0; st < C / 16; ++st) {
                const uint64_t bx = tc::sdesc_sw128(sbase + OFF_X + st * 2048, 8192, 1024);
                const uint64_t al = tc::sdesc_sw128(sbase + OFF_LZT + st * 32, 16, 1024);
                tc::mma_f16(tbase + COL_R, al, bx, id_uv, 1);
                const uint64_t ak = tc::sdesc_sw128(stg_a + ST_KT + st * 2048, 8192, 1024);
                tc::mma_f16(tbase + COL_ST, ak, bx, id_state, 1);
            }
            tc::mma_commit(bar_mma);
        }
        mma_pending = true;
        if (!wait_mma()) { aborted = true; break; }

        // 12. outputs of the chunk; fp16 copy of the new S for the next chunk
        if (tid < C) {
            const int c = tid;
            TIn* orow = out + ((static_cast<size_t>(b) * T + n * C + c) * H + h) * V + v0;
#pragma unroll
            for (int q2 = 0; q2 < VS / 32; ++q2) {
                float o[32];
                tc::tmem_ld32(tbase + lane_base + COL_R + q2 * 32, o);
                tc::tmem_ld_wait();
                nonfinite |= any_nonfinite32(o);
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    float ov[4] = {scale * o[j], scale * o[j + 1], scale * o[j + 2], scale * o[j + 3]};
                    VecIO<TIn, 4>::store(orow + q2 * 32 + j, ov);
                }
            }
        }
        {
            const int k = tid;
#pragma unroll
            for (int q2 = 0; q2 < VS / 32; ++q2) {
                float sv[32];
                tc::tmem_ld32(tbase + lane_base + COL_ST + q2 * 32, sv);
                tc::tmem_ld_wait();
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
                    st_row_chunk(sm + OFF_SS + ((q2 * 32) / 64) * (KD * 128), k, ((q2 * 32) % 64) / 8 + cc, sv + 8 * cc);
            }
        }
        if (tid < C && n + 1 < N) sbeta[(s ^ 1) * C + tid] = beta_next;
        tc::fence_proxy_async();
        tc::tc_fence_before();
        __syncthreads();
    }

    if (aborted) {
        if (tid == 0) atomicExch(&g_timeout_flag, 1u);
        // drain whatever is still in flight (bounded), so the CTA leaves nothing behind
        for (int s = 0; s < 2; ++s)
            if (tma_pending[s]) tc::mbar_wait(bar_tma0 + 8 * s, (tma_chunk[s] >> 1) & 1, kMaxPolls >> 4);
        if (mma_pending) tc::mbar_wait(bar_mma, mph, kMaxPolls >> 4);
        tc::tc_fence_before();
        __syncthreads();
        tc::tc_fence_after();
    } else {
        // final state S_out[v0 + v][k] = S^T[k][v]
        const int k = tid;
#pragma unroll
        for (int q2 = 0; q2 < VS / 32; ++q2) {
            float sv[32];
            tc::tmem_ld32(tbase + lane_base + COL_ST + q2 * 32, sv);
            tc::tmem_ld_wait();
            nonfinite |= any_nonfinite32(sv);
#pragma unroll
            for (int j = 0; j < 32; ++j)
                S_out[(static_cast<size_t>(bh) * V + v0 + q2 * 32 + j) * KD + k] = sv[j];
        }
        if (nonfinite) atomicOr(&g_range_flag, 1u);
        tc::tc_fence_before();
        __syncthreads();
        tc::tc_fence_after();
    }
    if (warp == 0) tc::tmem_dealloc(tbase, TMEM_COLS);
}

// =============================================================================================
// Workspace path: a fully parallel prep kernel (everything that does not depend on S) and a
// serial chain kernel (everything that does).  Per chunk the workspace holds fp16 images, in
// the exact 128-byte-swizzled shared-memory layout, of T' (8 KB), -W (two key blocks, 16 KB)
// and L = tril(Q K~^T, 0) (8 KB).
// =============================================================================================
constexpr uint32_t WS_T = 0, WS_W = 8192, WS_L = 24576;
// gated (OSGDN) chunks also carry their decay factors: gamma_t = prod_{l <= t} alpha_l and
// rho_t = prod_{l > t} alpha_l as 32 fp16 pairs each (tokens 2i, 2i + 1), then gamma_C (fp32)
constexpr uint32_t WS_GATE = 32768, WS_GAM = 0, WS_RHO = 128, WS_GC = 256;
constexpr uint32_t WS_CHUNK = 33280;  // a multiple of 128 bytes
// One state gate per key channel (OSKDA): per chunk of a head T', -W and L as above (with the
// channel decay inside W and L), then Q . Gamma and K~ . Gamma_C / Gamma as fp16 images in the
// layout of a loaded tile, then Gamma_C (128 fp32).
constexpr uint32_t WS_QG = 32768, WS_KTS = 49152, WS_GCV = 65536;
constexpr uint32_t WS_CHUNK_KDA = 66048;

template <int NW>
__device__ __forceinline__ void convert_bf16_to_f16(unsigned char* base, int tid) {
    // NW uint4 (8 elements) per thread, contiguous region of NW * 128 * 16 bytes
#pragma unroll
    for (int r = 0; r < NW; ++r) {
        uint4* p = reinterpret_cast<uint4*>(base) + r * NTHREADS + tid;
        uint4 u = *p;
        uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
            w[i] = pack_h2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
        *p = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

namespace prep {
// One worker's shared memory (byte offsets from a 1024-aligned base), 72 KB so that three workers
// fit on an SM.  Buffers that die early host later ones:
constexpr uint32_t OFF_KQ = 0;         // per key block: K (64 rows) | Q (64 rows), 2 x 16 KB
constexpr uint32_t OFF_Q0 = 8192;      //   Q rows of key block 0; after the Gram: gated T' image
constexpr uint32_t OFF_PM = 24576;     //   Q rows of key block 1; after the Gram: UT scratch A'
constexpr uint32_t OFF_KT = 32768;     // K~ (two key blocks); after the Gram: A's packed tiles, then
                                       //   T's off-diagonal tiles over them; last the -W image
constexpr uint32_t OFF_ZT = 49152;     // [L | T'] (L rows 0-63: the score image and the rows 0-63
                                       //   of W's A operand; T' rows 64-127; gated: T'' there)
constexpr uint32_t OFF_AM = OFF_KT;
constexpr uint32_t OFF_TD = 65536;     // T's four diagonal tiles
constexpr uint32_t OFF_BETA = OFF_TD + 4 * kTile * 4;
constexpr uint32_t OFF_EMIT = OFF_BETA + C * 4;              // step sizes, retention, start state
constexpr uint32_t OFF_ALPHA = OFF_EMIT + (2 * C + 2 * KD) * 4;  // state gates of the chunk (+ pad)
constexpr uint32_t OFF_GAM = OFF_ALPHA + (C + 4) * 4;          // their prefix products gamma
constexpr uint32_t OFF_BAR = OFF_GAM + C * 4;
constexpr uint32_t REGION = ((OFF_BAR + 32 + 1023) / 1024) * 1024;  // one worker, 1024-aligned
constexpr uint32_t SMEM_ALLOC = OFF_BAR + 32 + 1024;
constexpr uint32_t TMEM_COLS = 128;
static_assert(10 * kTile * 4 <= 16384 && kUtScratchTiles * kTile * 4 <= 8192, "UT scratch in dead buffers");
static_assert(3 * SMEM_ALLOC <= 233472 && 3 * REGION + 1024 <= 232448, "three prep workers per SM");
}  // namespace prep

// bar.red.and over the 128 threads of named barrier `bar`.
__device__ __forceinline__ bool bar_and128(int bar, bool pred) {
    uint32_t r;
    asm volatile("{\n .reg .pred p, q;\n setp.ne.u32 p, %2, 0;\n bar.red.and.pred q, %1, 128, p;\n selp.u32 %0, 1, 0, q;\n}\n"
                 : "=r"(r)
                 : "r"(bar), "r"(static_cast<uint32_t>(pred))
                 : "memory");
    return r != 0;
}

// The per-chunk work of phase 2 that does not depend on S, for 128 threads sharing a named
// barrier, a 1024-aligned shared region of prep::REGION bytes and 128 tensor-memory columns.
// One tensor-core pass over the loaded tiles gives [K; Q] K~^T: the Gram K K~^T (rows 0-63, for
// A = tril(diag(beta) K K~^T, -1)) and the scores Q K~^T (rows 64-127, for L).  Then
// T = (I + A)^-1 in fp32, T' = T diag(beta) and W = T' K (tensor cores) -> fp16 images of T', -W
// and L in the workspace.  With the OSGDN state gate (Appendix B.1, Eqs. (13)-(15)) the Gram and
// score entries (i, j) carry the decay ratio gamma_i / gamma_j = prod_{j < l <= i} alpha_l (formed
// as a running product along each row, so a zero gate gives zeros, never 0/0), and W takes
// T diag(beta gamma) while the workspace's T' stays T diag(beta) (for U = T'V).  With EMIT the
// write keys of the chunk are formed here instead of
// loaded: phase 1's clipped recurrence replayed per key coordinate from the chunk's start state
// with the step sizes the scan fixed, k~_t = d_t k_t (the same arithmetic as the emission
// kernel), and written out as well.
// A workspace word written concurrently by another CTA: the workspace is filled with all-ones
// before the launch and the writer never stores that pattern, so the first load that differs is
// the value.  Relaxed GPU-scope loads (not cached in L1); bounded, clears `ok` on giving up.
// `limit` is the number of polls (kMaxPolls unless a failure-detection test lowered it); each
// poll is one L2 round trip plus a 64 ns back-off, so the default gives up after about 2-4 s.
__device__ __forceinline__ float poll_word(const float* p, bool& ok, uint32_t limit) {
    for (uint32_t i = 0; i < limit; ++i) {
        uint32_t v;
        asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
        if (v != 0xffffffffu) return __uint_as_float(v);
        __nanosleep(64);
    }
    ok = false;
    return 0.f;
}

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
    return pack_h2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
// Two 16-bit values as loaded (bf16 or fp16) converted to fp16 and multiplied by the fp16 pair s
// (one rounding of the product; the converted values are exact in the fp16 normal range).
template <bool kBf16In>
__device__ __forceinline__ uint32_t mul_f16x2(uint32_t w, uint32_t s) {
    const uint32_t h = kBf16In ? bf16x2_to_f16x2(w) : w;
    const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&h), *reinterpret_cast<const __half2*>(&s));
    return *reinterpret_cast<const uint32_t*>(&r);
}
// Gate products of one chunk from its 64 state gates, two per lane (tokens 2 lane, 2 lane + 1):
// prefix gamma_t = prod_{l <= t} alpha_l and suffix rho_t = prod_{l > t} alpha_l, by warp scans
// (no division: a zero gate gives zeros).  Returns gamma_C = gamma_63 in every lane.
__device__ __forceinline__ float chunk_gates(float a0, float a1, int lane, float& g0, float& g1, float& r0,
                                             float& r1) {
    const float p = a0 * a1;
    float incl = p, sufx = p;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl *= y;
        const float z = __shfl_down_sync(0xffffffffu, sufx, o);
        if (lane + o < 32) sufx *= z;
    }
    float excl = __shfl_up_sync(0xffffffffu, incl, 1);
    float sexc = __shfl_down_sync(0xffffffffu, sufx, 1);
    if (lane == 0) excl = 1.f;
    if (lane == 31) sexc = 1.f;
    g0 = excl * a0;
    g1 = g0 * a1;
    r1 = sexc;
    r0 = a1 * sexc;
    return __shfl_sync(0xffffffffu, incl, 31);
}

template <typename TIn>
struct PrepWorker {
    static constexpr bool kBf16 = std::is_same<TIn, __nv_bfloat16>::value;
    unsigned char* sm;
    uint32_t sbase, tbase, bar_tma, bar_mma, tph, mph;
    int tid, bar;
    bool tma_pending, mma_pending;

    __device__ void init(unsigned char* region, int t, int barrier_id) {
        sm = region;
        sbase = tc::smem_u32(sm);
        bar_tma = sbase + prep::OFF_BAR;
        bar_mma = sbase + prep::OFF_BAR + 8;
        tid = t;
        bar = barrier_id;
        tph = mph = 0;
        tma_pending = mma_pending = false;
        if (tid == 0) {
            tc::mbar_init(bar_tma, 1);
            tc::mbar_init(bar_mma, 1);
            tc::mbar_init_fence();
        }
    }

    // Chunk n of head (b, h) into workspace slot `slot`.  Emission inputs (EMIT only): g_src[64],
    // r_src (stride H, or null), d_src[2 * KD] (hi, lo); tmKTout: tensor map of the k~ output.
    template <bool EMIT>
    __device__ bool run(const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmKT,
                        const float* __restrict__ beta, const float* __restrict__ alpha,
                        unsigned char* __restrict__ ws, size_t slot, int b,
                        int h, int n, int T, int H, const float* g_src, const float* r_src, const float* d_src,
                        float dmin, float dmax, const CUtensorMap* tmKTout, uint32_t poll_limit = kMaxPolls) {
        using namespace prep;
        float* AM = reinterpret_cast<float*>(sm + OFF_AM);
        float* TD = reinterpret_cast<float*>(sm + OFF_TD);
        float* PM = reinterpret_cast<float*>(sm + OFF_PM);
        float* sbeta = reinterpret_cast<float*>(sm + OFF_BETA);
        float* semit = reinterpret_cast<float*>(sm + OFF_EMIT);
        float* salpha = reinterpret_cast<float*>(sm + OFF_ALPHA);
        float* sgam = reinterpret_cast<float*>(sm + OFF_GAM);
        const bool gated = alpha != nullptr;
        const uint32_t lane_base = static_cast<uint32_t>((tid >> 5) * 32) << 16;
        const uint32_t id_gram = kBf16 ? tc::idesc_bf16_f32(128, C, false, false) : tc::idesc_f16_f32(128, C, false, false);
        const uint32_t id_w = tc::idesc_f16_f32(128, KD, false, true);
        const int row = b * T + n * C;
        if (tid == 0) {
            // the previous chunk's images (in the K~, Q and T' regions) must have been read
            tc::bulk_wait_read_all();
            tc::mbar_expect_tx(bar_tma, (EMIT ? 4 : 6) * 8192);
#pragma unroll
            for (int kb = 0; kb < 2; ++kb) {
                tc::tma_load_3d(sbase + OFF_KQ + kb * 16384, tmK, bar_tma, kb * 64, h, row);
                tc::tma_load_3d(sbase + OFF_KQ + kb * 16384 + 8192, tmQ, bar_tma, kb * 64, h, row);
                if (!EMIT) tc::tma_load_3d(sbase + OFF_KT + kb * 8192, tmKT, bar_tma, kb * 64, h, row);
            }
        }
        tma_pending = true;
        if (tid < C) sbeta[tid] = beta[(static_cast<size_t>(row) + tid) * H + h];
        if (gated && tid < C) salpha[tid] = alpha[(static_cast<size_t>(row) + tid) * H + h];
        bool ready = true;
        if (EMIT) {  // the scan may still be writing these: poll until they are there (bounded)
            if (tid < C) {
                semit[tid] = poll_word(g_src + tid, ready, poll_limit);
                semit[C + tid] = r_src ? r_src[static_cast<size_t>(tid) * H] : 1.f;
            }
            semit[2 * C + tid] = poll_word(d_src + tid, ready, poll_limit);
            semit[2 * C + KD + tid] = poll_word(d_src + KD + tid, ready, poll_limit);
        }
        {
            const bool ok = tc::mbar_wait(bar_tma, tph, kMaxPolls) && ready;
            if (!bar_and128(bar, ok)) return false;
            tph ^= 1u;
            tma_pending = false;
        }
        if (gated && (tid >> 5) == 1) {  // warp 1 (warp 0 issues the Gram): the chunk's decay factors
            const int l = tid & 31;
            float g0, g1, r0, r1;
            const float gc = chunk_gates(salpha[2 * l], salpha[2 * l + 1], l, g0, g1, r0, r1);
            sgam[2 * l] = g0;
            sgam[2 * l + 1] = g1;
            uint32_t* wg = reinterpret_cast<uint32_t*>(ws + slot * WS_CHUNK + WS_GATE);
            wg[(WS_GAM >> 2) + l] = pack_h2(g0, g1);
            wg[(WS_RHO >> 2) + l] = pack_h2(r0, r1);
            if (l == 0) reinterpret_cast<float*>(wg)[WS_GC >> 2] = gc;
        }
        if (EMIT) {  // thread tid: key coordinate tid of the 64 tokens
            const int i = tid, kb = i >> 6, c = (i & 63) >> 3, e = i & 7;
            const unsigned char* kin = sm + OFF_KQ + kb * 16384 + 2 * e;
            unsigned char* kto = sm + OFF_KT + kb * 8192 + 2 * e;
            float d = semit[2 * C + i] + semit[2 * C + KD + i];
            // 32 tokens at a time: the keys first, then the serial steps, then the stores, so
            // that no load waits behind a store it might alias; the tile leaves by TMA
#pragma unroll
            for (int j0 = 0; j0 < C; j0 += 32) {
                float kv[32];
                TIn kt[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) kv[j] = to_f32(*reinterpret_cast<const TIn*>(kin + tc::sw128_off(j0 + j, c)));
                float inc[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) inc[j] = replay_inc(semit[j0 + j], kv[j]);
                if (r_src != nullptr) {
                    float rv[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) rv[j] = semit[C + j0 + j];
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        kt[j] = from_f32<TIn>(d * kv[j]);
                        d = replay_step(d, rv[j], inc[j], dmin, dmax);
                    }
                } else {  // no retention gates: r = 1 (the same value replay_step would compute)
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        kt[j] = from_f32<TIn>(d * kv[j]);
                        d = replay_step(d, 1.f, inc[j], dmin, dmax);
                    }
                }
#pragma unroll
                for (int j = 0; j < 32; ++j) *reinterpret_cast<TIn*>(kto + tc::sw128_off(j0 + j, c)) = kt[j];
            }
            tc::fence_proxy_async();
            bar_sync128(bar);
            if (tid == 0) {  // k~ of the chunk to HBM (read before the -W image reuses the tile)
                tc::tma_store_3d(tmKTout, sbase + OFF_KT, 0, h, row);
                tc::tma_store_3d(tmKTout, sbase + OFF_KT + 8192, 64, h, row);
                tc::bulk_commit();
            }
        }

        // [K; Q] K~^T on the 16-bit tiles (exact products, fp32 sums)
        if (tid == 0) {
            tc::tc_fence_after();
#pragma unroll
            for (int st = 0; st < KD / 16; ++st) {
                const uint64_t a = tc::sdesc_sw128(sbase + OFF_KQ + (st >> 2) * 16384 + (st & 3) * 32, 16, 1024);
                const uint64_t bd = tc::sdesc_sw128(sbase + OFF_KT + (st >> 2) * 8192 + (st & 3) * 32, 16, 1024);
                tc::mma_f16(tbase, a, bd, id_gram, st > 0);
            }
            tc::mma_commit(bar_mma);
        }
        mma_pending = true;
        {
            const bool ok = tc::mbar_wait(bar_mma, mph, kMaxPolls);
            if (!bar_and128(bar, ok)) return false;
            mph ^= 1u;
            mma_pending = false;
            tc::tc_fence_after();
        }
        // K becomes the fp16 B operand of W = T' K
        if constexpr (kBf16) {
            convert_bf16_to_f16<4>(sm + OFF_KQ, tid);
            convert_bf16_to_f16<4>(sm + OFF_KQ + 16384, tid);
        }
        if (EMIT) {  // A's tiles go over K~: the k~ store must have read it
            if (tid == 0) tc::bulk_wait_read_all();
            bar_sync128(bar);
        }
        {
            const int i = tid & 63;
            float g[64];
            tc::tmem_ld32(tbase + lane_base, *reinterpret_cast<float(*)[32]>(g));
            tc::tmem_ld32(tbase + lane_base + 32, *reinterpret_cast<float(*)[32]>(g + 32));
            tc::tmem_ld_wait();
            if (gated) {  // decay ratios gamma_i / gamma_j along row i, j descending from i
                float rr = 1.f;
#pragma unroll
                for (int j = 63; j >= 0; --j) {
                    if (j < i) {
                        rr *= salpha[j + 1];
                        g[j] *= rr;
                    }
                }
            }
            if (tid < C) {  // Gram rows -> strictly lower A = diag(beta) K K~^T
                const int bi = i >> 4, r = i & 15;
                const float bt = sbeta[i];
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    const int bj = j >> 4;
                    if (bj <= bi) AM[tile_index(bi, bj) * kTile + r * kTileStride + (j & 15)] = (j < i) ? bt * g[j] : 0.f;
                }
            } else {  // score rows -> L = tril(Q K~^T, 0), fp16 image
#pragma unroll
                for (int j = 0; j < 64; ++j) g[j] = (j <= i) ? g[j] : 0.f;
#pragma unroll
                for (int c = 0; c < 8; ++c) st_row_chunk(sm + OFF_ZT, i, c, g + 8 * c);
            }
        }
        tc::tc_fence_before();
        bar_sync128(bar);
        ut_inverse_64_aliased(AM, TD, PM, tid, bar);
        {
            const int i = tid >> 1, half = tid & 1, bi = i >> 4, r = i & 15;
            float t[32];
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const int j = half * 32 + jj, bj = j >> 4;
                const float tv = (bj <= bi) ? ut_tile(AM, TD, bi, bj)[r * kTileStride + (j & 15)] : 0.f;
                t[jj] = tv * sbeta[j];
            }
            if (gated) {  // T' = T diag(beta) for the workspace, T'' = T diag(beta gamma) for W
#pragma unroll
                for (int c = 0; c < 4; ++c) st_row_chunk(sm + OFF_Q0, i, half * 4 + c, t + 8 * c);
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) t[jj] *= sgam[half * 32 + jj];
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) st_row_chunk(sm + OFF_ZT + 8192, i, half * 4 + c, t + 8 * c);
        }
        tc::fence_proxy_async();
        bar_sync128(bar);

        // W = [L; T'] K, read from lanes 64-127 (128 columns; rows 0-63 of the operand are the L
        // image, whose products land in lanes 0-63 and are not read); K's key blocks are 16 KB
        // apart.  Gated: [L; T''] K
        if (tid == 0) {
            tc::tc_fence_after();
#pragma unroll
            for (int st = 0; st < C / 16; ++st) {
                const uint64_t a = tc::sdesc_sw128(sbase + OFF_ZT + st * 32, 16, 1024);
                const uint64_t bk = tc::sdesc_sw128(sbase + OFF_KQ + st * 2048, 16384, 1024);
                tc::mma_f16(tbase, a, bk, id_w, st > 0);
            }
            tc::mma_commit(bar_mma);
        }
        mma_pending = true;
        if (EMIT && tid == 0) tc::bulk_wait_read_all();  // the k~ store has read the tile
        {
            const bool ok = tc::mbar_wait(bar_mma, mph, kMaxPolls);
            if (!bar_and128(bar, ok)) return false;
            mph ^= 1u;
            mma_pending = false;
            tc::tc_fence_after();
        }
        if (tid >= C) {  // -W image into the K~ region (K~ is no longer needed)
            const int c = tid - C;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                float w[32];
                tc::tmem_ld32(tbase + lane_base + q4 * 32, w);
                tc::tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) w[j] = -w[j];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
                    st_row_chunk(sm + OFF_KT + (q4 >> 1) * 8192, c, (q4 & 1) * 4 + cc, w + 8 * cc);
            }
        }
        tc::fence_proxy_async();
        tc::tc_fence_before();
        bar_sync128(bar);
        if (tid == 0) {
            unsigned char* dst = ws + slot * WS_CHUNK;
            tc::bulk_store(dst + WS_T, sbase + (gated ? OFF_Q0 : OFF_ZT + 8192), 8192);
            tc::bulk_store(dst + WS_W, sbase + OFF_KT, 16384);
            tc::bulk_store(dst + WS_L, sbase + OFF_ZT, 8192);
            tc::bulk_commit();
        }
        return true;
    }

    // After the last chunk (or an abort): nothing may still be in flight.
    __device__ void finish(bool aborted) {
        if (aborted) {
            if (tid == 0) atomicExch(&g_timeout_flag, 1u);
            if (tma_pending) tc::mbar_wait(bar_tma, tph, kMaxPolls >> 4);
            if (mma_pending) tc::mbar_wait(bar_mma, mph, kMaxPolls >> 4);
        }
        if (tid == 0) tc::bulk_wait_all();
    }
};

// One CTA loops over chunks q = blockIdx.x, blockIdx.x + gridDim.x, ...  (q = (b*H + h)*N + n).
template <typename TIn>
__global__ void __launch_bounds__(NTHREADS, 3)
chunk_prep_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmKT, const float* __restrict__ beta,
                  const float* __restrict__ alpha, unsigned char* __restrict__ ws, int T, int H, int N,
                  int total) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int tid = threadIdx.x, warp = tid >> 5;
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");  // the chain kernel may set up
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + prep::OFF_BAR + 16);
    PrepWorker<TIn> w;
    w.init(sm, tid, 0);
    if (tid == 0) {
        tc::prefetch_tmap(&tmQ);
        tc::prefetch_tmap(&tmK);
        tc::prefetch_tmap(&tmKT);
    }
    __syncthreads();
    if (warp == 0) tc::tmem_alloc(tc::smem_u32(tmem_slot), prep::TMEM_COLS);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    w.tbase = *tmem_slot;
    bool aborted = false;
    for (int q = blockIdx.x; q < total; q += gridDim.x) {
        const int bh = q / N, n = q - bh * N, b = bh / H, h = bh - b * H;
        if (!w.template run<false>(&tmQ, &tmK, &tmKT, beta, alpha, ws, static_cast<size_t>(q), b, h, n, T, H, nullptr,
                                   nullptr, nullptr, 0.f, 0.f, nullptr)) {
            aborted = true;
            break;
        }
    }
    w.finish(aborted);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 0) tc::tmem_dealloc(w.tbase, prep::TMEM_COLS);
}


// =============================================================================================
// Prep for one state gate per key channel (OSKDA, Appendix B.2; the chunk form of Listing 3).
// With Gamma_t = prod_{l <= t} alpha_l (per channel, cumulative within the chunk):
//   A = tril(diag(beta) (K . Gamma) (K~ / Gamma)^T, -1),  T = (I + A)^-1,  T' = T diag(beta),
//   W = T' (K . Gamma),  L = tril((Q . Gamma) (K~ / Gamma)^T, 0),
// and for the chain Q . Gamma, K~ . Gamma_C / Gamma and Gamma_C.  K~ / Gamma grows as the decay
// falls (past fp16's range once a channel decays below ~1e-4 over a chunk), so the scaled tiles
// are split into bf16 high and low parts (bf16's exponent range, ~16 bits of mantissa together)
// and each product is formed as hi.hi^T + hi.lo^T + lo.hi^T on the tensor cores; T' enters W the
// same way.  Every image the chain reads is bounded by the unscaled inputs (the gates are <= 1)
// and is stored in fp16.  One 128-thread CTA per worker, two per SM, looping over chunks.
// =============================================================================================
namespace kdap {
constexpr uint32_t OFF_AH = 0;       // per key block (16 KB): K rows -> K.Gamma hi | Q rows -> Q.Gamma hi
                                     //   (after the Gram, the Q slots hold the -W image)
constexpr uint32_t OFF_AL = 32768;   // per key block: K.Gamma lo | Q.Gamma lo (then T' hi / T' lo)
constexpr uint32_t OFF_B = 65536;    // K~ -> (K~ / Gamma) hi (16 KB) | lo (16 KB); after the Gram:
                                     //   A's tiles, T's diagonal tiles, the UT scratch, the L image
constexpr uint32_t OFF_TD = OFF_B + 10 * kTile * 4;
constexpr uint32_t OFF_PM = OFF_TD + 4 * kTile * 4;
constexpr uint32_t OFF_L = OFF_B + 24576;
constexpr uint32_t OFF_BETA = 98304;
constexpr uint32_t OFF_BAR = OFF_BETA + C * 4;
constexpr uint32_t SMEM_ALLOC = OFF_BAR + 32 + 1024;
constexpr uint32_t TMEM_COLS = 128;
static_assert(OFF_PM + kUtScratchTiles * kTile * 4 <= OFF_L, "UT scratch below the L image");
static_assert(2 * SMEM_ALLOC <= 233472, "two workers per SM");
}  // namespace kdap

__device__ __forceinline__ uint16_t bf16_bits(float x) {
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<const uint16_t*>(&h);
}
__device__ __forceinline__ float bf16_val(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }
__device__ __forceinline__ uint16_t f16_bits(float x) {
    const __half h = __float2half_rn(x);
    return *reinterpret_cast<const uint16_t*>(&h);
}

template <typename TIn>
__global__ void __launch_bounds__(NTHREADS, 2)
chunk_prep_kda_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmKT, const float* __restrict__ beta,
                      const float* __restrict__ alpha, unsigned char* __restrict__ ws, int T, int H, int N, int total) {
    using namespace kdap;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int tid = threadIdx.x, warp = tid >> 5;
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");  // the chain kernel may set up
    const uint32_t sbase = tc::smem_u32(sm);
    const uint32_t bar_tma = sbase + OFF_BAR, bar_mma = sbase + OFF_BAR + 8;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_BAR + 16);
    float* AM = reinterpret_cast<float*>(sm + OFF_B);
    float* TD = reinterpret_cast<float*>(sm + OFF_TD);
    float* PM = reinterpret_cast<float*>(sm + OFF_PM);
    float* sbeta = reinterpret_cast<float*>(sm + OFF_BETA);
    if (tid == 0) {
        tc::mbar_init(bar_tma, 1);
        tc::mbar_init(bar_mma, 1);
        tc::mbar_init_fence();
        tc::prefetch_tmap(&tmQ);
        tc::prefetch_tmap(&tmK);
        tc::prefetch_tmap(&tmKT);
    }
    __syncthreads();
    if (warp == 0) tc::tmem_alloc(tc::smem_u32(tmem_slot), TMEM_COLS);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t id_gram = tc::idesc_bf16_f32(128, C, false, false);
    const uint32_t id_w = tc::idesc_bf16_f32(128, KD, false, true);
    // this thread's key channel and its place in a loaded 64-wide key-block tile
    const int ch = tid, kb = ch >> 6, cc = (ch & 63) >> 3, e = ch & 7;
    uint32_t tph = 0, mph = 0;
    bool ok = true;
    for (int q = blockIdx.x; ok && q < total; q += gridDim.x) {
        const int bh = q / N, n = q - bh * N, b = bh / H, h = bh - b * H;
        const int row = b * T + n * C;
        unsigned char* dst = ws + static_cast<size_t>(q) * WS_CHUNK_KDA;
        if (tid == 0) {
            tc::bulk_wait_read_all();  // the previous chunk's images have left shared memory
            tc::mbar_expect_tx(bar_tma, 6 * 8192);
#pragma unroll
            for (int k2 = 0; k2 < 2; ++k2) {
                tc::tma_load_3d(sbase + OFF_AH + k2 * 16384, &tmK, bar_tma, k2 * 64, h, row);
                tc::tma_load_3d(sbase + OFF_AH + k2 * 16384 + 8192, &tmQ, bar_tma, k2 * 64, h, row);
                tc::tma_load_3d(sbase + OFF_B + k2 * 8192, &tmKT, bar_tma, k2 * 64, h, row);
            }
        }
        if (tid < C) sbeta[tid] = beta[(static_cast<size_t>(row) + tid) * H + h];
        // the channel's cumulative decay over the chunk (fp32, a running product)
        float gam[C];
        {
            const float* ap = alpha + (static_cast<size_t>(row) * H + h) * KD + ch;
            float g = 1.f;
#pragma unroll
            for (int t = 0; t < C; ++t) {
                g *= ap[static_cast<size_t>(t) * H * KD];
                gam[t] = g;
            }
        }
        const float gC = gam[C - 1];
        reinterpret_cast<float*>(dst + WS_GCV)[ch] = gC;
        ok = tc::mbar_wait(bar_tma, tph, kMaxPolls);
        if (!__syncthreads_and(ok)) break;
        tph ^= 1u;
        // scale the channel's column of K, Q and K~ (64 tokens): bf16 hi / lo parts for the
        // tensor cores, Q . Gamma and K~ . Gamma_C / Gamma in fp16 for the chain
        {
            const uint32_t boff = 2u * e;
            unsigned char* kq = sm + OFF_AH + kb * 16384;
            unsigned char* kql = sm + OFF_AL + kb * 16384;
            unsigned char* kt = sm + OFF_B + kb * 8192;
            unsigned char* ktl = sm + OFF_B + 16384 + kb * 8192;
            unsigned char* gq = dst + WS_QG + kb * 8192;
            unsigned char* gk = dst + WS_KTS + kb * 8192;
#pragma unroll
            for (int t = 0; t < C; ++t) {
                const uint32_t o = tc::sw128_off(t, cc) + boff;
                const float g = gam[t];
                const float kx = to_f32(*reinterpret_cast<const TIn*>(kq + o)) * g;
                const float qx = to_f32(*reinterpret_cast<const TIn*>(kq + 8192 + o)) * g;
                const float kv = to_f32(*reinterpret_cast<const TIn*>(kt + o));
                const float zx = kv / fmaxf(g, 1e-30f);
                const uint16_t kh = bf16_bits(kx), qh = bf16_bits(qx), zh = bf16_bits(zx);
                *reinterpret_cast<uint16_t*>(kq + o) = kh;
                *reinterpret_cast<uint16_t*>(kql + o) = bf16_bits(kx - bf16_val(kh));
                *reinterpret_cast<uint16_t*>(kq + 8192 + o) = qh;
                *reinterpret_cast<uint16_t*>(kql + 8192 + o) = bf16_bits(qx - bf16_val(qh));
                *reinterpret_cast<uint16_t*>(kt + o) = zh;
                *reinterpret_cast<uint16_t*>(ktl + o) = bf16_bits(zx - bf16_val(zh));
                *reinterpret_cast<uint16_t*>(gq + o) = f16_bits(qx);
                *reinterpret_cast<uint16_t*>(gk + o) = f16_bits(kv * (gC / fmaxf(g, 1e-30f)));
            }
        }
        tc::fence_proxy_async();
        __syncthreads();
        // [K.G; Q.G] (K~/G)^T = hi.hi + hi.lo + lo.hi: lanes 0-63 the Gram, lanes 64-127 the scores
        if (tid == 0) {
            tc::tc_fence_after();
#pragma unroll
            for (int part = 0; part < 3; ++part) {
                const uint32_t abase = sbase + (part == 2 ? OFF_AL : OFF_AH);
                const uint32_t bbase = sbase + OFF_B + (part == 1 ? 16384 : 0);
#pragma unroll
                for (int st = 0; st < KD / 16; ++st) {
                    const uint64_t a = tc::sdesc_sw128(abase + (st >> 2) * 16384 + (st & 3) * 32, 16, 1024);
                    const uint64_t bd = tc::sdesc_sw128(bbase + (st >> 2) * 8192 + (st & 3) * 32, 16, 1024);
                    tc::mma_f16(tbase, a, bd, id_gram, (part > 0 || st > 0) ? 1u : 0u);
                }
            }
            tc::mma_commit(bar_mma);
        }
        ok = tc::mbar_wait(bar_mma, mph, kMaxPolls);
        if (!__syncthreads_and(ok)) break;
        mph ^= 1u;
        tc::tc_fence_after();
        {
            const int i = tid & 63;
            float gr[64];
            tc::tmem_ld32(tbase + lane_base, *reinterpret_cast<float(*)[32]>(gr));
            tc::tmem_ld32(tbase + lane_base + 32, *reinterpret_cast<float(*)[32]>(gr + 32));
            tc::tmem_ld_wait();
            if (tid < C) {  // Gram rows -> strictly lower A = diag(beta) (K.G) (K~/G)^T
                const int bi = i >> 4, r = i & 15;
                const float bt = sbeta[i];
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    const int bj = j >> 4;
                    if (bj <= bi) AM[tile_index(bi, bj) * kTile + r * kTileStride + (j & 15)] = (j < i) ? bt * gr[j] : 0.f;
                }
            } else {  // score rows -> L = tril(.., 0), fp16 image
#pragma unroll
                for (int j = 0; j < 64; ++j) gr[j] = (j <= i) ? gr[j] : 0.f;
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) st_row_chunk(sm + OFF_L, i, c8, gr + 8 * c8);
            }
        }
        tc::tc_fence_before();
        __syncthreads();
        ut_inverse_64_aliased(AM, TD, PM, tid, 0);
        {  // T' = T diag(beta): fp16 image to the workspace, bf16 hi / lo for W
            const int i = tid >> 1, half = tid & 1, bi = i >> 4, r = i & 15;
            float tv[32];
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const int j = half * 32 + jj, bj = j >> 4;
                tv[jj] = ((bj <= bi) ? ut_tile(AM, TD, bi, bj)[r * kTileStride + (j & 15)] : 0.f) * sbeta[j];
            }
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                const int c8 = half * 4 + c4;
                uint32_t w16[4], wh[4], wl[4];
#pragma unroll
                for (int p2 = 0; p2 < 4; ++p2) {
                    const float a0 = tv[c4 * 8 + 2 * p2], a1 = tv[c4 * 8 + 2 * p2 + 1];
                    w16[p2] = pack_h2(a0, a1);
                    const uint16_t h0 = bf16_bits(a0), h1 = bf16_bits(a1);
                    wh[p2] = static_cast<uint32_t>(h0) | (static_cast<uint32_t>(h1) << 16);
                    wl[p2] = static_cast<uint32_t>(bf16_bits(a0 - bf16_val(h0))) |
                             (static_cast<uint32_t>(bf16_bits(a1 - bf16_val(h1))) << 16);
                }
                *reinterpret_cast<uint4*>(dst + WS_T + tc::sw128_off(i, c8)) = make_uint4(w16[0], w16[1], w16[2], w16[3]);
                *reinterpret_cast<uint4*>(sm + OFF_AL + 8192 + tc::sw128_off(i, c8)) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
                *reinterpret_cast<uint4*>(sm + OFF_AL + 16384 + 8192 + tc::sw128_off(i, c8)) =
                    make_uint4(wl[0], wl[1], wl[2], wl[3]);
            }
        }
        tc::fence_proxy_async();
        tc::tc_fence_before();
        __syncthreads();
        // W = T' (K.G) = T'hi (K.G)hi + T'hi (K.G)lo + T'lo (K.G)hi, read from lanes 64-127: the A
        // operands are [K.G lo (kb); T' hi / lo], whose top rows only fill lanes 0-63
        if (tid == 0) {
            tc::tc_fence_after();
#pragma unroll
            for (int part = 0; part < 3; ++part) {
                const uint32_t abase = sbase + OFF_AL + (part == 2 ? 16384 : 0);
                const uint32_t bbase = sbase + (part == 1 ? OFF_AL : OFF_AH);
#pragma unroll
                for (int st = 0; st < C / 16; ++st) {
                    const uint64_t a = tc::sdesc_sw128(abase + st * 32, 16, 1024);
                    const uint64_t bk = tc::sdesc_sw128(bbase + st * 2048, 16384, 1024);
                    tc::mma_f16(tbase, a, bk, id_w, (part > 0 || st > 0) ? 1u : 0u);
                }
            }
            tc::mma_commit(bar_mma);
        }
        ok = tc::mbar_wait(bar_mma, mph, kMaxPolls);
        if (!__syncthreads_and(ok)) break;
        mph ^= 1u;
        tc::tc_fence_after();
        if (tid >= C) {  // -W image into the Q slots (Q is no longer needed)
            const int c = tid - C;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                float w[32];
                tc::tmem_ld32(tbase + lane_base + q4 * 32, w);
                tc::tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) w[j] = -w[j];
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4)
                    st_row_chunk(sm + OFF_AH + (q4 >> 1) * 16384 + 8192, c, (q4 & 1) * 4 + c4, w + 8 * c4);
            }
        }
        tc::fence_proxy_async();
        tc::tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc::bulk_store(dst + WS_W, sbase + OFF_AH + 8192, 8192);
            tc::bulk_store(dst + WS_W + 8192, sbase + OFF_AH + 16384 + 8192, 8192);
            tc::bulk_store(dst + WS_L, sbase + OFF_L, 8192);
            tc::bulk_commit();
        }
    }
    if (!ok && tid == 0) {  // a wait gave up: record it, let what was issued land, then leave
        atomicExch(&g_timeout_flag, 1u);
        tc::mbar_wait(bar_tma, tph, kMaxPolls >> 4);
        tc::mbar_wait(bar_mma, mph, kMaxPolls >> 4);
    }
    if (tid == 0) tc::bulk_wait_all();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 0) tc::tmem_dealloc(tbase, TMEM_COLS);
}

namespace chain {
// Twelve warps with fixed roles (one CTA per (batch, head, 64 rows of S)):
//   warps 0-3   S^T epilogue (fp32 S^T in tensor memory -> fp16 B operand in shared memory);
//               warps 0-1 also the X epilogue (X = U - W S^T -> fp16 B operand)
//   warps 4-7   operand staging: [-W; Q], [T'; 0], K~^T and [*; L] into tensor memory as fp16,
//               and the V tile to fp16 in place (the B operand of U = T'V)
//   warp 8      tcgen05.mma issue (one thread)
//   warp 9      TMA / bulk-copy producer (one thread)
//   warps 10-11 O readout (tensor memory -> shared memory -> TMA store)
// Every MMA takes its A operand from tensor memory; shared memory carries the loaded tiles, the
// B operands and the two epilogue tiles.  Only the S^T and X epilogues and the two S-dependent
// MMA groups lie on the serial path from one chunk to the next.
constexpr int NT = 384;
constexpr uint32_t ST_Q = 0;                           // Q, two 64-wide key blocks (as loaded)
constexpr uint32_t ST_W = 16384;                       // -W image (fp16)
constexpr uint32_t ST_KT = 32768;                      // K~ (as loaded)
constexpr uint32_t ST_V = 49152;                       // V slice (as loaded)
constexpr uint32_t ST_T = ST_V + (VS / 64) * 8192;     // T' image (fp16)
constexpr uint32_t ST_L = ST_T + 8192;                 // L image (fp16)
constexpr uint32_t STAGE = ST_L + 8192;
constexpr uint32_t OFF_X = 2 * STAGE;                  // X (64 tokens x VS values), fp16
constexpr uint32_t OFF_SS = OFF_X + (VS / 64) * 8192;  // S^T (128 key rows x VS values), fp16
constexpr uint32_t OFF_O = OFF_SS + (VS / 64) * KD * 128;  // O tile for the TMA store
constexpr uint32_t OFF_BAR = OFF_O + (VS / 64) * 8192;
constexpr uint32_t SMEM_ALLOC = OFF_BAR + 256 + 1024;
constexpr uint32_t LOAD_BYTES = 3 * 16384 + (VS / 64) * 8192 + 2 * 8192;
static_assert(SMEM_ALLOC <= 232448, "chain shared memory");
static_assert(STAGE % 1024 == 0 && OFF_X % 1024 == 0 && OFF_SS % 1024 == 0 && OFF_O % 1024 == 0,
              "swizzle atoms");
// tensor-memory columns (lanes 0-63 carry U / X, lanes 64-127 carry Q S^T / O)
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_R = 0;              // R[2] (fp32)
constexpr uint32_t COL_ST = 2 * VS;        // S^T (fp32, lane = key)
constexpr uint32_t COL_QW = COL_ST + VS;   // A: [-W; Q] fp16, two buffers of 64 columns
constexpr uint32_t COL_TH = COL_QW + 128;  // A: [T'; *] fp16, two buffers of 32 columns
constexpr uint32_t COL_KT = COL_TH + 64;   // A: K~^T fp16 (lane = key)
constexpr uint32_t COL_LH = COL_KT + 32;   // A: [*; L] fp16
static_assert(COL_LH + 32 <= TMEM_COLS, "tensor memory columns");
// mbarriers (byte offsets from OFF_BAR) and their arrival counts
constexpr uint32_t B_FULL = 0;      // [2] stage loaded                       (1 + tx bytes)
constexpr uint32_t B_FREE = 16;     // [2] stage no longer read               (U commit + 4 warps)
constexpr uint32_t B_CONVA = 32;    // [2] [-W; Q], T', fp16 V staged (buffer b) (4 warps)
constexpr uint32_t B_QS = 48;       // [2] [-W; Q] S^T done in R[b]           (commit)
constexpr uint32_t B_KT = 64;       // K~^T staged                            (4 warps)
constexpr uint32_t B_LH = 72;       // L staged                               (2 warps)
constexpr uint32_t B_XRDY = 80;     // fp16 X in shared memory                (2 warps)
constexpr uint32_t B_ST = 88;       // S^T update done                        (commit)
constexpr uint32_t B_SRDY = 96;     // fp16 S^T in shared memory              (4 warps)
constexpr uint32_t B_O = 104;       // [2] O accumulated in R[b]              (commit)
constexpr uint32_t B_RFREE = 120;   // [2] O read out of R[b]                 (2 warps)
constexpr uint32_t B_DRAIN = 136;   // final commit before tensor memory is released
constexpr uint32_t TMEM_SLOT = 144, ABORT = 148;
}  // namespace chain

// Bounded wait that also gives up as soon as another role has recorded an abort.  Every lane of
// the calling warp must call it; the result is the same in all lanes.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const volatile int* abort_flag) {
    bool ok = false;
    for (uint32_t i = 0; i < kMaxPolls; ++i) {
        if (tc::mbar_try_wait(bar, parity)) { ok = true; break; }
        if ((i & 63u) == 63u && *abort_flag) break;
    }
    return __all_sync(0xffffffffu, ok);
}
// Single-thread variant (MMA issuer, producer).
__device__ __forceinline__ bool thread_wait(uint32_t bar, uint32_t parity, const volatile int* abort_flag) {
    for (uint32_t i = 0; i < kMaxPolls; ++i) {
        if (tc::mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 63u && *abort_flag) return false;
    }
    return false;
}
__device__ __forceinline__ void record_abort(volatile int* abort_flag) {
    *abort_flag = 1;
    atomicExch(&g_timeout_flag, 1u);
}
// After a warp's writes for the tensor cores (shared memory through the async proxy, or tensor
// memory through tcgen05.st): make them visible, then one arrival per warp.
__device__ __forceinline__ void warp_publish(uint32_t bar, int lane) {
    tc::fence_proxy_async();
    tc::tc_fence_before();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(bar);
}
// Named barrier over the two readout warps; true when any thread passed `pred`.
__device__ __forceinline__ bool pair_any(bool pred) {
    uint32_t c;
    asm volatile("{\n .reg .pred p;\n setp.ne.u32 p, %1, 0;\n bar.red.popc.u32 %0, 1, 64, p;\n}\n"
                 : "=r"(c)
                 : "r"(static_cast<uint32_t>(pred))
                 : "memory");
    return c != 0;
}

// Segment-parallel state pass (Appendix A.2, Eq. (10): the chunk transition is affine in S,
// S^T_n = P_n S^T_{n-1} + Z_n with P_n = I - K~_n^T W_n).  The chunks of a head are cut into
// segments of n_seg chunks; segment 0 runs from S0, every later one from a zero state,
// and beside its value slices it runs as many transition slices: the same pass with
// zero values (U = 0) and the identity as its start (64 of its key columns per CTA).  Those carry
// Phi_n = P_n ... P_first, write G_n = scale (Q_n - L_n W_n) Phi_{n-1} (the readout of a transition
// slice) through tmG in fp16, and end in Phi of the segment.  With S_start of each segment known
// afterwards, S_end = S_start Phi^T-product + Z (seg_combine_kernel) and the outputs of a later
// segment gain G_n S_start^T (seg_correct_kernel).  Unsegmented: n_seg = N, no transition slices.
struct ChainSeg {
    int n_seg;    // chunks per segment
    int vslices;  // value slices per head (V / VS); slices from here on are transition slices
    float* Z;     // [G][B H][V][K]: end state of each segment's value slices (null: S_out directly)
    float* P;     // [G][B H][K][K]: end state of each later segment's transition slices
};

// One CTA per (batch, head, VS rows of S), serial over chunks.  Per chunk: U = T'V and
// [X; Q S^T] = [U; 0] + [-W; Q] S^T; then S^T += K~^T X and O = Q S^T + L X.  T', -W and L come
// from the workspace by bulk copy; Q, K~, V by TMA; O leaves by TMA.
// GATED (OSGDN, Appendix B.1, Eqs. (13)-(15)): with gamma_t / rho_t the gate products from the
// chunk start through t / after t (formed by the prep, read from the workspace a chunk ahead), the
// staging warps scale the rows of Q by gamma (O = diag(gamma) Q S^T + L X, the ratios being in L)
// and the tokens of K~ by rho (S^T <- gamma_C S^T + (rho . K~)^T X); the S^T epilogue stores the
// fp16 copy for the S-dependent products from the fp32 state it carries in registers, formed as
// gamma_C S^T + Y from the update product Y = (rho . K~)^T X that the tensor cores leave on its own.
template <typename TIn, bool GATED, bool SEG, bool KDA = false>
__device__ __forceinline__ void chain_body(const CUtensorMap& tmQ, const CUtensorMap& tmKT, const CUtensorMap& tmV,
                                           const CUtensorMap& tmO, const CUtensorMap& tmG, const ChainSeg& sg,
                                           const unsigned char* __restrict__ ws, const float* S0, float* S_out,
                                           int T, int H, int V, int N, float scale) {
    using namespace chain;
    static_assert(!KDA || GATED, "the channel-gated chain carries its state like the gated one");
    constexpr bool kBf16 = std::is_same<TIn, __nv_bfloat16>::value;
    constexpr uint32_t kSlot = KDA ? WS_CHUNK_KDA : WS_CHUNK;  // workspace bytes per chunk of a head
    // This CTA's segment of chunks [m0, m0 + NL) and slice (value rows, or key columns of Phi).
    // SEG: blockIdx.y enumerates the first segment's value slices, then for each later segment
    // its value slices and its transition slices (the first segment starts from S0 itself), so
    // that no CTA leaves early (an early exit here slows every CTA's loop); every segment is
    // non-empty.  SEG = false: one segment of value slices (the compiler drops the rest).
    const int ys = static_cast<int>(blockIdx.y) - sg.vslices;
    const int seg = (SEG && ys >= 0) ? 1 + ys / (2 * sg.vslices) : 0;
    const int slice = !SEG || ys < 0 ? static_cast<int>(blockIdx.y) : ys % (2 * sg.vslices);
    const bool phi = SEG && slice >= sg.vslices;
    const int m0 = SEG ? seg * sg.n_seg : 0;
    const int NL = SEG ? min(N - m0, sg.n_seg) : N;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x, b = bh / H, h = bh % H;
    const int v0 = (phi ? slice - sg.vslices : slice) * VS;
    const int BH = static_cast<int>(gridDim.x);
    // start state: S0 for the first segment's value slices, zero for later ones, the identity for
    // transition slices; end state: S_out, or the segment's slot in Z or P
    const float* S0c = (seg == 0) ? S0 : nullptr;
    float* S_end = !SEG ? S_out + static_cast<size_t>(bh) * V * KD
                   : phi ? sg.P + (static_cast<size_t>(seg) * BH + bh) * KD * KD
                         : sg.Z + (static_cast<size_t>(seg) * BH + bh) * V * KD;
    const CUtensorMap* tmOut = phi ? &tmG : &tmO;
    const uint32_t sbase = tc::smem_u32(sm);
    const uint32_t bars = sbase + OFF_BAR;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_BAR + TMEM_SLOT);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + OFF_BAR + ABORT);
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;

    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            tc::mbar_init(bars + B_FULL + 8 * s, 1);
            tc::mbar_init(bars + B_FREE + 8 * s, 5);
            tc::mbar_init(bars + B_CONVA + 8 * s, 4);
            tc::mbar_init(bars + B_QS + 8 * s, 1);
            tc::mbar_init(bars + B_O + 8 * s, 1);
            tc::mbar_init(bars + B_RFREE + 8 * s, 2);
        }
        tc::mbar_init(bars + B_KT, 4);
        tc::mbar_init(bars + B_LH, 2);
        tc::mbar_init(bars + B_XRDY, 2);
        tc::mbar_init(bars + B_ST, 1);
        tc::mbar_init(bars + B_SRDY, 4);
        tc::mbar_init(bars + B_DRAIN, 1);
        *abort_flag = 0;
        tc::mbar_init_fence();
        tc::prefetch_tmap(&tmQ);
        tc::prefetch_tmap(&tmKT);
        tc::prefetch_tmap(&tmV);
        tc::prefetch_tmap(&tmO);
    }
    __syncthreads();
    if (warp == 0) tc::tmem_alloc(tc::smem_u32(tmem_slot), TMEM_COLS);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    // Launched as a programmatic dependent of the kernel that writes the chunk images and k~
    // (the setup above overlaps that kernel's tail): wait until its results are visible.  A
    // no-op when launched without the attribute.
    asm volatile("griddepcontrol.wait;\n" ::: "memory");

    if (warp == 9) {
        // ================================ producer ============================================
        if (lane == 0) {
            int last[2] = {-1, -1};
            for (int m = 0; m < NL; ++m) {
                const int s = m & 1;
                if (m >= 2 && !thread_wait(bars + B_FREE + 8 * s, ((m - 2) >> 1) & 1, abort_flag)) {
                    record_abort(abort_flag);
                    break;
                }
                const uint32_t bar = bars + B_FULL + 8 * s;
                const uint32_t st = sbase + s * STAGE;
                const int row = b * T + (m0 + m) * C;
                const unsigned char* wsc = ws + (static_cast<size_t>(bh) * N + m0 + m) * kSlot;
                tc::mbar_expect_tx(bar, phi ? LOAD_BYTES - (VS / 64) * 8192 : LOAD_BYTES);
                if (KDA) {  // Q . Gamma and K~ . Gamma_C / Gamma, formed by the prep
                    tc::bulk_load(st + ST_Q, wsc + WS_QG, 16384, bar);
                    tc::bulk_load(st + ST_KT, wsc + WS_KTS, 16384, bar);
                } else {
#pragma unroll
                    for (int kb = 0; kb < 2; ++kb) {
                        tc::tma_load_3d(st + ST_Q + kb * 8192, &tmQ, bar, kb * 64, h, row);
                        tc::tma_load_3d(st + ST_KT + kb * 8192, &tmKT, bar, kb * 64, h, row);
                    }
                }
                if (!phi) {  // a transition slice has zero values
#pragma unroll
                    for (int vb = 0; vb < VS / 64; ++vb)
                        tc::tma_load_3d(st + ST_V + vb * 8192, &tmV, bar, v0 + vb * 64, h, row);
                }
                tc::bulk_load(st + ST_W, wsc + WS_W, 16384, bar);
                tc::bulk_load(st + ST_T, wsc + WS_T, 8192, bar);
                tc::bulk_load(st + ST_L, wsc + WS_L, 8192, bar);
                last[s] = m;
            }
            // nothing may still be landing in shared memory when the CTA exits
            for (int s = 0; s < 2; ++s)
                if (last[s] >= 0) tc::mbar_wait(bars + B_FULL + 8 * s, (last[s] >> 1) & 1, kMaxPolls >> 4);
        }
    } else if (warp == 8) {
        // ================================ MMA issuer ==========================================
        if (lane == 0) {
            const uint32_t id_h = tc::idesc_f16_f32(128, VS, false, true);  // fp16 A (tensor memory), MN-major B
            // Descriptors are built once; an operand k steps further is the same descriptor plus
            // its byte offset / 16 (shared memory stays below 2^18 bytes, so the 14-bit address
            // field never carries).
            const uint64_t d_v[2] = {tc::sdesc_sw128(sbase + ST_V, 8192, 1024),
                                     tc::sdesc_sw128(sbase + STAGE + ST_V, 8192, 1024)};
            const uint64_t d_ss = tc::sdesc_sw128(sbase + OFF_SS, KD * 128, 1024);
            const uint64_t d_x = tc::sdesc_sw128(sbase + OFF_X, 8192, 1024);
            auto off = [](uint32_t bytes) { return static_cast<uint64_t>(bytes >> 4); };
            auto issue_u = [&](int m) {  // R[m & 1] = [T'; 0] V  (a transition slice has U = 0)
                const int bb = m & 1;
                const uint32_t dR = tbase + COL_R + bb * VS;
                if (!phi) {
#pragma unroll
                    for (int k = 0; k < C / 16; ++k)
                        tc::mma_f16_ts(dR, tbase + COL_TH + bb * 32 + 8 * k, d_v[bb] + off(k * 2048), id_h, k > 0);
                }
                tc::mma_commit(bars + B_FREE + 8 * bb);
            };
            // U(m) needs chunk m staged and (from m = 2 on) R[m & 1] read out
            auto u_ready = [&](int m) -> bool {
                const uint32_t cb = bars + B_CONVA + 8 * (m & 1), cp = (m >> 1) & 1;
                const uint32_t rb = bars + B_RFREE + 8 * (m & 1), rp = ((m - 2) >> 1) & 1;
                return thread_wait(cb, cp, abort_flag) && (m < 2 || thread_wait(rb, rp, abort_flag));
            };
            bool ok = u_ready(0);
            if (ok) {
                tc::tc_fence_after();
                issue_u(0);
            }
            for (int n = 0; ok && n < NL; ++n) {
                const int bb = n & 1;
                const uint32_t dR = tbase + COL_R + bb * VS;
                // [X; Q S^T] += [-W; Q] S^T: needs the fp16 copy of S after chunk n - 1
                if (!(ok = thread_wait(bars + B_SRDY, n & 1, abort_flag))) break;
                tc::tc_fence_after();
#pragma unroll
                for (int k = 0; k < KD / 16; ++k)
                    tc::mma_f16_ts(dR, tbase + COL_QW + bb * 64 + 8 * k, d_ss + off(k * 2048), id_h,
                                   (phi && k == 0) ? 0u : 1u);
                tc::mma_commit(bars + B_QS + 8 * bb);
                // S^T += K~^T X  (gated: Y = (rho . K~)^T X on its own; the epilogue adds gamma_C S^T)
                if (!(ok = thread_wait(bars + B_XRDY, n & 1, abort_flag) && thread_wait(bars + B_KT, n & 1, abort_flag)))
                    break;
                tc::tc_fence_after();
#pragma unroll
                for (int k = 0; k < C / 16; ++k)
                    tc::mma_f16_ts(tbase + COL_ST, tbase + COL_KT + 8 * k, d_x + off(k * 2048), id_h,
                                   (GATED && k == 0) ? 0u : 1u);
                tc::mma_commit(bars + B_ST);
                // O = Q S^T + L X  (lanes 0-63 of the L operand only touch R rows already read)
                if (!(ok = thread_wait(bars + B_LH, n & 1, abort_flag))) break;
                tc::tc_fence_after();
#pragma unroll
                for (int k = 0; k < C / 16; ++k)
                    tc::mma_f16_ts(dR, tbase + COL_LH + 8 * k, d_x + off(k * 2048), id_h, 1);
                tc::mma_commit(bars + B_O + 8 * bb);
                if (n + 1 < NL) {  // the next chunk's U = T'V, off the serial path
                    if (!(ok = u_ready(n + 1))) break;
                    tc::tc_fence_after();
                    issue_u(n + 1);
                }
            }
            if (!ok) record_abort(abort_flag);
            // no MMA may be in flight when tensor memory is released: one more commit tracks all
            tc::mma_commit(bars + B_DRAIN);
            tc::mbar_wait(bars + B_DRAIN, 0, kMaxPolls >> 4);
        }
    } else if (warp >= 10) {
        // ========================== O readout: TMEM -> smem -> TMA ============================
        const int r = (warp - 10) * 32 + lane;  // token row; tensor-memory lane 64 + r
        const bool issuer = warp == 10 && lane == 0;
        bool ok = true, nonfinite = false;
        for (int n = 0; n < NL; ++n) {
            const int bb = n & 1;
            ok = warp_wait(bars + B_O + 8 * bb, (n >> 1) & 1, abort_flag);
            if (issuer) tc::bulk_wait_read_all();  // the previous tile has left shared memory
            if (pair_any(!ok)) { ok = false; break; }
            tc::tc_fence_after();
#pragma unroll
            for (int q2 = 0; q2 < VS / 32; ++q2) {
                float o[32];
                tc::tmem_ld32(tbase + lane_base + COL_R + bb * VS + q2 * 32, o);
                tc::tmem_ld_wait();
                nonfinite |= any_nonfinite32(o);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float ov[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) ov[j] = scale * o[8 * c + j];
                    uint4 u;
                    if (phi) {  // G_n in fp16
                        u = make_uint4(pack_h2(ov[0], ov[1]), pack_h2(ov[2], ov[3]), pack_h2(ov[4], ov[5]),
                                       pack_h2(ov[6], ov[7]));
                    } else {
                        VecIO<TIn, 4>::store(reinterpret_cast<TIn*>(&u), ov);
                        VecIO<TIn, 4>::store(reinterpret_cast<TIn*>(&u) + 4, ov + 4);
                    }
                    *reinterpret_cast<uint4*>(sm + OFF_O + ((q2 * 32) / 64) * 8192 +
                                              tc::sw128_off(r, ((q2 * 32) % 64) / 8 + c)) = u;
                }
            }
            tc::fence_proxy_async();
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(bars + B_RFREE + 8 * bb);
            pair_any(false);  // both warps' rows are in shared memory
            if (issuer) {
#pragma unroll
                for (int vb = 0; vb < VS / 64; ++vb)
                    tc::tma_store_3d(tmOut, sbase + OFF_O + vb * 8192, v0 + vb * 64, h, b * T + (m0 + n) * C);
                tc::bulk_commit();
            }
        }
        if (issuer) tc::bulk_wait_all();
        if (nonfinite) atomicOr(&g_range_flag, 1u);
        if (!ok) record_abort(abort_flag);
    } else if (warp >= 4) {
        // ======================== operand staging into tensor memory ==========================
        const int w4 = warp - 4;
        const bool low = w4 < 2;            // lanes 0-63: -W and T' rows; lanes 64-127: Q and L rows
        const int r = (w4 & 1) * 32 + lane;  // row 0..63 of the 64-row tiles
        if (!low) {  // [T'; 0]: the bottom 64 rows stay zero in both buffers
            uint32_t z[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) z[j] = 0u;
#pragma unroll
            for (int c = 0; c < 2; ++c) tc::tmem_st32u(tbase + lane_base + COL_TH + 32 * c, z);
            tc::tmem_st_wait();
        }
        bool ok = true;
        // gated: gamma and rho of tokens 2 lane, 2 lane + 1 of a chunk as fp16 pairs (formed by
        // the prep), read from the workspace one chunk ahead
        uint32_t gpair = 0, rpair = 0, gnext = 0, rnext = 0;
        auto gates_of = [&](int m) {  // (the gated chain is never segmented: m0 = 0)
            const uint32_t* wg = reinterpret_cast<const uint32_t*>(ws + (static_cast<size_t>(bh) * N + m) * kSlot + WS_GATE);
            gnext = wg[(WS_GAM >> 2) + lane];
            rnext = wg[(WS_RHO >> 2) + lane];
        };
        if (GATED && !KDA) {
            gates_of(0);
            gpair = gnext;
            rpair = rnext;
        }
        for (int m = 0; ok && m < NL; ++m) {
            const int s = m & 1, bb = m & 1;
            const unsigned char* stg = sm + s * STAGE;
            if (!(ok = warp_wait(bars + B_FULL + 8 * s, (m >> 1) & 1, abort_flag))) break;
            // buffer bb was last read by U and [-W; Q] S^T of chunk m - 2
            if (m >= 2 && !(ok = warp_wait(bars + B_QS + 8 * bb, ((m - 2) >> 1) & 1, abort_flag))) break;
            tc::tc_fence_after();
            if (low) {
                uint32_t wv[32];
#pragma unroll
                for (int kb = 0; kb < 2; ++kb) {
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint4 u = *reinterpret_cast<const uint4*>(stg + ST_W + kb * 8192 + tc::sw128_off(r, c));
                        wv[c * 4 + 0] = u.x;
                        wv[c * 4 + 1] = u.y;
                        wv[c * 4 + 2] = u.z;
                        wv[c * 4 + 3] = u.w;
                    }
                    tc::tmem_st32u(tbase + lane_base + COL_QW + bb * 64 + kb * 32, wv);
                }
                uint32_t th[32];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 u = *reinterpret_cast<const uint4*>(stg + ST_T + tc::sw128_off(r, c));
                    th[c * 4 + 0] = u.x;
                    th[c * 4 + 1] = u.y;
                    th[c * 4 + 2] = u.z;
                    th[c * 4 + 3] = u.w;
                }
                tc::tmem_st32u(tbase + lane_base + COL_TH + bb * 32, th);
            } else {
                uint32_t qh[32];
                uint32_t gq = 0;  // gated: row r of Q scaled by gamma_r (an fp16 pair of it)
                if (GATED && !KDA) {
                    const uint32_t gp = __shfl_sync(0xffffffffu, gpair, r >> 1);
                    const uint32_t g16 = (r & 1) ? (gp >> 16) : (gp & 0xffffu);
                    gq = g16 | (g16 << 16);
                }
#pragma unroll
                for (int kb = 0; kb < 2; ++kb) {
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint4 u = *reinterpret_cast<const uint4*>(stg + ST_Q + kb * 8192 + tc::sw128_off(r, c));
                        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            qh[c * 4 + j] = KDA ? w[j] : GATED ? mul_f16x2<kBf16>(w[j], gq) : (kBf16 ? bf16x2_to_f16x2(w[j]) : w[j]);
                    }
                    tc::tmem_st32u(tbase + lane_base + COL_QW + bb * 64 + kb * 32, qh);
                }
            }
            // V to fp16 in place (4 x 16 bytes per thread of the four staging warps)
            if (kBf16 && !phi) convert_bf16_to_f16<(VS / 64) * 4>(const_cast<unsigned char*>(stg) + ST_V, w4 * 32 + lane);
            tc::tmem_st_wait();
            warp_publish(bars + B_CONVA + 8 * bb, lane);
            if (GATED && !KDA && m + 1 < NL) gates_of(m + 1);
            // K~^T (lane = key); its buffer was last read by the S^T update of chunk m - 1
            if (m >= 1 && !(ok = warp_wait(bars + B_ST, (m - 1) & 1, abort_flag))) break;
            tc::tc_fence_after();
            {  // thread k gathers key coordinate k of the 64 tokens
                const int k = w4 * 32 + lane, kb = k >> 6, c = (k & 63) >> 3, e = k & 7;
                const unsigned char* kt = stg + ST_KT + kb * 8192 + 2 * e;
                uint32_t kw[32];
#pragma unroll
                for (int t2 = 0; t2 < 32; ++t2) {
                    const uint32_t a0 = *reinterpret_cast<const uint16_t*>(kt + tc::sw128_off(2 * t2, c));
                    const uint32_t a1 = *reinterpret_cast<const uint16_t*>(kt + tc::sw128_off(2 * t2 + 1, c));
                    const uint32_t pr = a0 | (a1 << 16);
                    if (KDA) {  // already scaled, fp16
                        kw[t2] = pr;
                    } else if (GATED) {  // tokens 2 t2, 2 t2 + 1 scaled by their rho
                        kw[t2] = mul_f16x2<kBf16>(pr, __shfl_sync(0xffffffffu, rpair, t2));
                    } else {
                        kw[t2] = kBf16 ? bf16x2_to_f16x2(pr) : pr;
                    }
                }
                tc::tmem_st32u(tbase + lane_base + COL_KT, kw);
                tc::tmem_st_wait();
                warp_publish(bars + B_KT, lane);
            }
            // L rows (lanes 64-127); the L operand was last read by O of chunk m - 1
            if (!low) {
                if (m >= 1 && !(ok = warp_wait(bars + B_O + 8 * ((m - 1) & 1), ((m - 1) >> 1) & 1, abort_flag))) break;
                tc::tc_fence_after();
                uint32_t lh[32];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 u = *reinterpret_cast<const uint4*>(stg + ST_L + tc::sw128_off(r, c));
                    lh[c * 4 + 0] = u.x;
                    lh[c * 4 + 1] = u.y;
                    lh[c * 4 + 2] = u.z;
                    lh[c * 4 + 3] = u.w;
                }
                tc::tmem_st32u(tbase + lane_base + COL_LH, lh);
                tc::tmem_st_wait();
                warp_publish(bars + B_LH, lane);
            }
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(bars + B_FREE + 8 * s);  // this warp's reads of stage s are done
            gpair = gnext;
            rpair = rnext;
        }
        if (!ok) record_abort(abort_flag);
    } else {
        // ============================ S^T and X epilogues =====================================
        const int k = tid;  // key coordinate = tensor-memory lane
        // gated: gamma_C of a chunk (the product of its 64 state gates, formed by the prep)
        auto gamma_c = [&](int m) -> float {  // channel-gated: this lane's (key channel's) Gamma_C
            if (KDA) return reinterpret_cast<const float*>(ws + (static_cast<size_t>(bh) * N + m) * kSlot + WS_GCV)[k];
            return *reinterpret_cast<const float*>(ws + (static_cast<size_t>(bh) * N + m) * kSlot + WS_GATE + WS_GC);
        };
        // gated: this lane's row of S^T (fp32) carried in registers; the update MMA leaves
        // Y = (rho . K~)^T X in tensor memory and S^T <- gamma_C S^T + Y is formed here
        float st[GATED ? VS : 1];
        {  // S0 slice -> S^T (tensor memory, or registers when gated) and its fp16 operand copy
            float sv[32];
#pragma unroll
            for (int half = 0; half < VS / 32; ++half) {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    sv[j] = phi ? (k == v0 + half * 32 + j ? 1.f : 0.f)
                                : (S0c ? S0c[(static_cast<size_t>(bh) * V + v0 + half * 32 + j) * KD + k] : 0.f);
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    st_row_chunk(sm + OFF_SS + ((half * 32) / 64) * (KD * 128), k, ((half * 32) % 64) / 8 + c, sv + 8 * c);
                if (GATED) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) st[half * 32 + j] = sv[j];
                } else {
                    tc::tmem_st32(tbase + lane_base + COL_ST + half * 32, sv);
                }
            }
            if (!GATED) tc::tmem_st_wait();
            warp_publish(bars + B_SRDY, lane);
        }
        bool ok = true;
        for (int n = 0; n < NL; ++n) {
            const int bb = n & 1;
            const float gcn = GATED ? gamma_c(n) : 1.f;  // gamma_C of this chunk, used after its update
            if (warp < 2) {  // X rows live in tensor-memory lanes 0-63
                if (!(ok = warp_wait(bars + B_QS + 8 * bb, (n >> 1) & 1, abort_flag))) break;
                tc::tc_fence_after();
#pragma unroll
                for (int q2 = 0; q2 < VS / 32; ++q2) {
                    float x[32];
                    tc::tmem_ld32(tbase + lane_base + COL_R + bb * VS + q2 * 32, x);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc)
                        st_row_chunk(sm + OFF_X + ((q2 * 32) / 64) * 8192, tid, ((q2 * 32) % 64) / 8 + cc, x + 8 * cc);
                }
                warp_publish(bars + B_XRDY, lane);
            }
            if (!(ok = warp_wait(bars + B_ST, n & 1, abort_flag))) break;
            tc::tc_fence_after();
            float sv[VS];
#pragma unroll
            for (int q2 = 0; q2 < VS / 32; ++q2)
                tc::tmem_ld32(tbase + lane_base + COL_ST + q2 * 32, *reinterpret_cast<float(*)[32]>(sv + q2 * 32));
            tc::tmem_ld_wait();
            if (GATED) {
#pragma unroll
                for (int j = 0; j < VS; ++j) {
                    st[j] = fmaf(gcn, st[j], sv[j]);
                    sv[j] = st[j];
                }
            }
            if (n + 1 < NL) {
#pragma unroll
                for (int cc = 0; cc < VS / 8; ++cc)
                    st_row_chunk(sm + OFF_SS + ((cc * 8) / 64) * (KD * 128), k, cc % 8, sv + 8 * cc);
                warp_publish(bars + B_SRDY, lane);
            } else {
                bool bad = false;
#pragma unroll
                for (int j = 0; j < VS; ++j) {
                    bad |= !isfinite(sv[j]);
                    S_end[static_cast<size_t>(v0 + j) * KD + k] = sv[j];
                }
                if (bad) atomicOr(&g_range_flag, 1u);
            }
        }
        if (!ok) record_abort(abort_flag);
    }

    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 0) tc::tmem_dealloc(tbase, TMEM_COLS);
}

template <typename TIn, bool GATED, bool KDA = false>
__global__ void __launch_bounds__(chain::NT, 1)
chunk_chain_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmKT,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                   const unsigned char* __restrict__ ws, const float* S0, float* S_out, int T, int H,
                   int V, int N, float scale) {
    chain_body<TIn, GATED, false, KDA>(tmQ, tmKT, tmV, tmO, tmO, ChainSeg{N, 0, nullptr, nullptr}, ws, S0, S_out, T, H, V,
                                  N, scale);
}
// The segmented pass: grid (B H, value slices x (2 G - 1)), see chain_body.
template <typename TIn>
__global__ void __launch_bounds__(chain::NT, 1)
chunk_chain_seg_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmKT,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                       const __grid_constant__ CUtensorMap tmG, ChainSeg sg, const unsigned char* __restrict__ ws,
                       const float* S0, float* S_out, int T, int H, int V, int N, float scale) {
    chain_body<TIn, false, true>(tmQ, tmKT, tmV, tmO, tmG, sg, ws, S0, S_out, T, H, V, N, scale);
}

// Start states of the segments and the final state.  Row v of S evolves on its own across a
// segment boundary: S_start(g + 1)[v][k] = sum_j S_start(g)[v][j] P_g[j][k] + Z_g[v][k] (P_g[j][k] =
// Phi_g[k][j], the transition slices' end state), so each CTA carries 16 rows of one head through
// all boundaries in fp32, with P_g staged in shared memory.  Sst[g] (g >= 1) receives S_start(g)
// for the output correction.  Grid (B H, V / 16), 256 threads, 72 KB of shared memory.
constexpr uint32_t COMBINE_SMEM = (KD * KD + 16 * KD) * 4;
__global__ void __launch_bounds__(256)
seg_combine_kernel(const float* __restrict__ Z, const float* __restrict__ P, float* __restrict__ Sst,
                   float* __restrict__ S_out, int G, int V) {
    extern __shared__ float cmb[];
    float* Ps = cmb;                   // P_g, [j][k]
    float(*cur)[KD] = reinterpret_cast<float(*)[KD]>(cmb + KD * KD);
    const int bh = blockIdx.x, BH = gridDim.x, r0 = blockIdx.y * 16, tid = threadIdx.x;
    const int k = tid & (KD - 1), rh = tid >> 7;  // column k, rows rh * 8 .. rh * 8 + 7
    auto row_of = [&](int g, int r) {  // offset of row r of head bh in slot g of a [G][BH][V][K] array
        return ((static_cast<size_t>(g) * BH + bh) * V + r0 + r) * KD;
    };
    for (int i = tid; i < 16 * KD; i += 256) cur[i / KD][i % KD] = Z[row_of(0, i / KD) + i % KD];
    for (int g = 1; g < G; ++g) {
        const float4* Pg = reinterpret_cast<const float4*>(P + (static_cast<size_t>(g) * BH + bh) * KD * KD);
        for (int i = tid; i < KD * KD / 4; i += 256) reinterpret_cast<float4*>(Ps)[i] = Pg[i];
        __syncthreads();
        for (int i = tid; i < 16 * KD; i += 256) Sst[row_of(g, i / KD) + i % KD] = cur[i / KD][i % KD];
        float acc[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) acc[r] = Z[row_of(g, rh * 8 + r) + k];
#pragma unroll 8
        for (int j = 0; j < KD; ++j) {
            const float pj = Ps[j * KD + k];
#pragma unroll
            for (int r = 0; r < 8; ++r) acc[r] = fmaf(cur[rh * 8 + r][j], pj, acc[r]);
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < 8; ++r) cur[rh * 8 + r][k] = acc[r];
    }
    __syncthreads();
    for (int i = tid; i < 16 * KD; i += 256)
        S_out[(static_cast<size_t>(bh) * V + r0 + i / KD) * KD + i % KD] = cur[i / KD][i % KD];
}

// Output correction of the later segments: o_n += G_n S_start(g)^T, G_n (64 tokens x K, fp16) from
// the transition slices.  One CTA per (head, segment g >= 1, group of chunk pairs): S_start(g) in
// fp16 as the K-major B operand (N = V = 128 rows), two chunks of G stacked as the M = 128 A
// operand, the same two chunks of o (TMA), fp32 accumulator in tensor memory; each thread adds its
// token row to the o tile in shared memory, which leaves by TMA.  128 threads, one pair at a time.
namespace segc {
constexpr uint32_t OFF_A = 0;          // per key block: chunk c rows | chunk c + 1 rows (16 KB)
constexpr uint32_t OFF_B = 32768;      // S_start^T operand: per key block 128 rows x 128 bytes
constexpr uint32_t OFF_O = 65536;      // o: per 64-wide value block, chunk c rows | chunk c + 1 rows
constexpr uint32_t OFF_BAR = 98304;
constexpr uint32_t SMEM_ALLOC = OFF_BAR + 64 + 1024;
}  // namespace segc
template <typename TIn>
__global__ void __launch_bounds__(128, 1)
seg_correct_kernel(const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmO,
                   const float* __restrict__ Sst, int T, int H, int V, int N, int n_seg) {
    using namespace segc;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int tid = threadIdx.x, warp = tid >> 5;
    const int bh = blockIdx.x, b = bh / H, h = bh % H, BH = gridDim.x;
    const int g = blockIdx.y + 1;
    const int m0 = g * n_seg, NL = min(N - m0, n_seg);
    const int npairs = (NL + 1) / 2;
    const uint32_t sbase = tc::smem_u32(sm);
    const uint32_t bar_tma = sbase + OFF_BAR, bar_mma = sbase + OFF_BAR + 8;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_BAR + 16);
    if (tid == 0) {
        tc::mbar_init(bar_tma, 1);
        tc::mbar_init(bar_mma, 1);
        tc::mbar_init_fence();
        tc::prefetch_tmap(&tmG);
        tc::prefetch_tmap(&tmO);
    }
    // S_start(g) -> fp16 K-major operand; unit u: row u / 16, eight columns 8 (u % 16), so that
    // sixteen threads read one 512-byte row
    {
        const float* S = Sst + (static_cast<size_t>(g) * BH + bh) * V * KD;
        for (int u = tid; u < V * 16; u += 128) {
            const int row = u >> 4, c16 = u & 15;
            const float4 x = *reinterpret_cast<const float4*>(S + row * KD + c16 * 8);
            const float4 y = *reinterpret_cast<const float4*>(S + row * KD + c16 * 8 + 4);
            const float v8[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
            st_row_chunk(sm + OFF_B + (c16 >> 3) * 16384, row, c16 & 7, v8);
        }
    }
    tc::fence_proxy_async();
    __syncthreads();
    if (warp == 0) tc::tmem_alloc(tc::smem_u32(tmem_slot), 128);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t idesc = tc::idesc_f16_f32(128, 128, false, false);
    const int r = tid & 63, half = tid >> 6;  // this thread's token row: chunk c + half, row r
    uint32_t ph = 0;
    bool ok = true;
    for (int p = blockIdx.z; ok && p < npairs; p += gridDim.z) {
        const int c = m0 + 2 * p;
        const bool two = 2 * p + 1 < NL;
        if (tid == 0) {
            tc::bulk_wait_read_all();  // the previous pair's o tile has left shared memory
            tc::mbar_expect_tx(bar_tma, (two ? 8 : 4) * 8192);
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
                if (hb == 1 && !two) break;
                const int row = b * T + (c + hb) * C;
#pragma unroll
                for (int kb = 0; kb < 2; ++kb) {
                    tc::tma_load_3d(sbase + OFF_A + kb * 16384 + hb * 8192, &tmG, bar_tma, kb * 64, h, row);
                    tc::tma_load_3d(sbase + OFF_O + kb * 16384 + hb * 8192, &tmO, bar_tma, kb * 64, h, row);
                }
            }
        }
        ok = tc::mbar_wait(bar_tma, ph, kMaxPolls);
        if (!__syncthreads_and(ok)) break;
        if (tid == 0) {
            tc::tc_fence_after();
#pragma unroll
            for (int k = 0; k < KD / 16; ++k) {
                const uint32_t koff = (k >> 2) * 16384 + (k & 3) * 32;
                tc::mma_f16(tbase, tc::sdesc_sw128(sbase + OFF_A + koff, 16, 1024),
                            tc::sdesc_sw128(sbase + OFF_B + koff, 16, 1024), idesc, k > 0);
            }
            tc::mma_commit(bar_mma);
        }
        ok = tc::mbar_wait(bar_mma, ph, kMaxPolls);
        if (!__syncthreads_and(ok)) break;
        ph ^= 1u;
        tc::tc_fence_after();
        if (half == 0 || two) {
#pragma unroll
            for (int q2 = 0; q2 < 4; ++q2) {  // 32 value columns at a time
                float acc[32];
                tc::tmem_ld32(tbase + lane_base + q2 * 32, acc);
                tc::tmem_ld_wait();
                unsigned char* tile = sm + OFF_O + (q2 >> 1) * 16384 + half * 8192;
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    uint4* pp = reinterpret_cast<uint4*>(tile + tc::sw128_off(r, (q2 & 1) * 4 + c8));
                    uint4 u = *pp;
                    float cur[8];
                    VecIO<TIn, 4>::load(reinterpret_cast<const TIn*>(&u), cur);
                    VecIO<TIn, 4>::load(reinterpret_cast<const TIn*>(&u) + 4, cur + 4);
#pragma unroll
                    for (int i = 0; i < 8; ++i) cur[i] += acc[c8 * 8 + i];
                    VecIO<TIn, 4>::store(reinterpret_cast<TIn*>(&u), cur);
                    VecIO<TIn, 4>::store(reinterpret_cast<TIn*>(&u) + 4, cur + 4);
                    *pp = u;
                }
            }
        }
        tc::fence_proxy_async();
        tc::tc_fence_before();
        __syncthreads();  // the o tile is complete; the A tiles and the accumulator are free again
        if (tid == 0) {
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
                if (hb == 1 && !two) break;
#pragma unroll
                for (int kb = 0; kb < 2; ++kb)
                    tc::tma_store_3d(&tmO, sbase + OFF_O + kb * 16384 + hb * 8192, kb * 64, h, b * T + (c + hb) * C);
            }
            tc::bulk_commit();
        }
    }
    if (!ok && tid == 0) {  // a wait gave up: record it, let what was issued land, then leave
        atomicExch(&g_timeout_flag, 1u);
        tc::mbar_wait(bar_tma, ph, kMaxPolls >> 4);
        tc::mbar_wait(bar_mma, ph, kMaxPolls >> 4);
    }
    if (tid == 0) tc::bulk_wait_all();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 0) tc::tmem_dealloc(tbase, 128);
}

// =============================================================================================
// Fused layer forward: phase 1 and the S-independent part of phase 2 in one cooperative launch.
// CTAs 0 .. BH-1 run the blocked scan of one (batch, head) each and store every 64-token block's
// step sizes and start state to the workspace as soon as it is solved; every other CTA runs two
// prep workers that take chunks in block-major order from a counter, poll (bounded) for their
// block's values, form the chunk's write keys from them and do the chunk prep.  Phase 1 keeps B*H
// SMs busy for its whole duration, so the prep of each chunk hides behind the scan of later
// blocks.  All CTAs are resident at once (cooperative launch), so the waits always end.  The
// workspace's scan part and the counter hold all-ones at launch (the counter's first increment
// wraps it to chunk 0).
// =============================================================================================
constexpr int LAYER_NT = 384;      // phase 1 on threads 0-255 of the first B*H CTAs; three prep workers
constexpr int LAYER_WORKERS = 3;

template <typename TIn, bool HAS_R>
__global__ void __launch_bounds__(LAYER_NT, 1)
layer_scan_prep_kernel(OsdnScanArgs sa, float* ws_g, float* ws_d, unsigned int* counter,
                       const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmKT, const float* __restrict__ alpha,
                       unsigned char* __restrict__ cws, int N, int BH, uint32_t poll_limit) {
    extern __shared__ unsigned char smem_raw[];
    const int tid = threadIdx.x, warp = tid >> 5, w = tid >> 7, wt = tid & 127;
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");  // the chain kernel may set up
    __shared__ uint32_t s_tmem;
    __shared__ int s_q[LAYER_WORKERS];
    constexpr uint32_t kCols = 512;  // >= the scan's 256 and the workers' 3 x 128, a power of two
    static_assert(kCols >= scanblk::TMEM_COLS && kCols >= LAYER_WORKERS * prep::TMEM_COLS, "tensor memory");
    if (warp == 0) tc::tmem_alloc(tc::smem_u32(&s_tmem), kCols);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tbase = s_tmem;
    // phase 1 for one (batch, head); afterwards this CTA joins the prep workers
    if (static_cast<int>(blockIdx.x) < BH && tid < scanblk::NT)
        scanblk::scan_block_body<TIn, TIn, HAS_R>(sa, ws_g, ws_d, blockIdx.x, smem_raw, tbase, &g_timeout_flag);
    __syncthreads();  // the scan's shared memory becomes the workers' regions
    unsigned char* base = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int T = sa.T, H = sa.H;
    PrepWorker<TIn> pw;
    pw.init(base + w * prep::REGION, wt, 1 + w);
    if (tid == 0) {
        tc::prefetch_tmap(&tmQ);
        tc::prefetch_tmap(&tmK);
        tc::prefetch_tmap(&tmKT);
    }
    __syncthreads();
    pw.tbase = tbase + w * prep::TMEM_COLS;
    const int total = BH * N;
    bool aborted = false;
    for (;;) {
        if (wt == 0) s_q[w] = static_cast<int>(atomicAdd(counter, 1u) + 1u);
        bar_sync128(1 + w);
        const int q = s_q[w];
        if (q >= total) break;
        const int m = q / BH, bh = q - m * BH, b = bh / H, h = bh - b * H;
        const size_t row0 = static_cast<size_t>(b) * T * H + h;
        const float* g_src = ws_g + static_cast<size_t>(bh) * T + m * C;
        const float* r_src = HAS_R ? sa.r + row0 + static_cast<size_t>(m) * C * H : nullptr;
        const float* d_src = ws_d + (static_cast<size_t>(bh) * N + m) * (2 * KD);
        if (!pw.template run<true>(&tmQ, &tmK, nullptr, sa.beta, alpha, cws, static_cast<size_t>(bh) * N + m, b, h, m, T, H,
                                   g_src, r_src, d_src, sa.d_min, sa.d_max, &tmKT, poll_limit)) {
            aborted = true;
            break;
        }
    }
    pw.finish(aborted);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 0) tc::tmem_dealloc(tbase, kCols);
}

// Poll limit of the fused layer's prep workers (0: the default kMaxPolls); lowered only by
// osdn_set_poll_limit, for failure-detection tests.
std::atomic<uint32_t> g_poll_limit{0};

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// [B*T rows of H heads of `inner` elements]: dims (inner, H, B*T), box (64, 1, 64).
bool make_map(CUtensorMap* m, const void* ptr, CUtensorMapDataType dt, int inner, int H, long long rows) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(H),
                          static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner) * 2, static_cast<cuuint64_t>(H) * inner * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, dt, 3, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() {
    static int n = 0;
    static std::once_flag once;
    std::call_once(once, [] {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            n = 148;
    });
    return n;
}

template <typename K>
cudaError_t set_smem(K kernel, uint32_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

// Segments of the state pass (see ChainSeg): more than one when a head's chain would leave most
// SMs idle, i.e. few heads and long sequences.  Each later segment adds as many transition-slice
// CTAs as value-slice CTAs; all CTAs must fit on the GPU at once, and segments keep >= 16 chunks.
int seg_count(int B, int H, int T, int V) {
    const int BH = B * H, N = T / C, vsl = V / VS;
    if (V != KD) return 1;
    int G = 1;
    for (int g = 2; g <= 8; ++g) {
        if (BH * (vsl + (g - 1) * 2 * vsl) > num_sms() || N < g * 16) break;
        G = g;
    }
    return G;
}
// Workspace of the segmented pass: [chunk images][G_n, fp16 rows like q][Z][P][S_start], 256-aligned.
struct SegWs {
    size_t gbuf, z, p, sst, total;
};
SegWs seg_ws(const OsdnChunkArgs& a, int G) {
    auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    const size_t BH = static_cast<size_t>(a.B) * a.H, N = static_cast<size_t>(a.T / C);
    SegWs s{};
    s.gbuf = up(BH * N * WS_CHUNK);
    s.z = s.gbuf + up(static_cast<size_t>(a.B) * a.T * a.H * KD * 2);
    s.p = s.z + up(static_cast<size_t>(G) * BH * a.V * KD * 4);
    s.sst = s.p + up(static_cast<size_t>(G) * BH * KD * KD * 4);
    s.total = s.sst + up(static_cast<size_t>(G) * BH * a.V * KD * 4);
    return s;
}

// With a workspace: the prep kernel (unless chain_only: the layer call's cooperative kernel did
// it) and the chain kernel, segmented when seg_count > 1 and the workspace holds the segment
// scratch, then the segment combine and the output correction.  Without: one fused kernel.
template <typename TIn>
cudaError_t launch_tc(const OsdnChunkArgs& a, void* ws, size_t ws_bytes, cudaStream_t s, bool chain_only = false) {
    const CUtensorMapDataType dt = std::is_same<TIn, __half>::value ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                                    : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const long long rows = static_cast<long long>(a.B) * a.T;
    CUtensorMap mq, mk, mkt, mv, mo, mg;
    if (!make_map(&mq, a.q, dt, a.K, a.H, rows) || !make_map(&mk, a.k, dt, a.K, a.H, rows) ||
        !make_map(&mkt, a.k_tilde, dt, a.K, a.H, rows) || !make_map(&mv, a.v, dt, a.V, a.H, rows) ||
        !make_map(&mo, a.o, dt, a.V, a.H, rows))
        return cudaErrorNotSupported;
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        cudaError_t e[9] = {set_smem(chunk_tc_kernel<TIn>, fused::SMEM_ALLOC),
                            set_smem(chunk_prep_kernel<TIn>, prep::SMEM_ALLOC),
                            set_smem(chunk_chain_kernel<TIn, false>, chain::SMEM_ALLOC),
                            set_smem(chunk_chain_kernel<TIn, true>, chain::SMEM_ALLOC),
                            set_smem(chunk_chain_seg_kernel<TIn>, chain::SMEM_ALLOC),
                            set_smem(seg_correct_kernel<TIn>, segc::SMEM_ALLOC),
                            set_smem(seg_combine_kernel, COMBINE_SMEM),
                            set_smem(chunk_prep_kda_kernel<TIn>, kdap::SMEM_ALLOC),
                            set_smem(chunk_chain_kernel<TIn, true, true>, chain::SMEM_ALLOC)};
        for (cudaError_t x : e)
            if (x != cudaSuccess && attr_err == cudaSuccess) attr_err = x;
    });
    if (attr_err != cudaSuccess) return attr_err;
    const int N = a.T / C;
    dim3 block(NTHREADS);
    if (a.alpha && a.alpha_per_key) {  // one gate per key channel: its prep, then the channel-gated chain
        const size_t need_kda = static_cast<size_t>(a.B) * a.H * N * WS_CHUNK_KDA;
        if (ws == nullptr || ws_bytes < need_kda || chain_only) return cudaErrorNotSupported;
        unsigned char* w = static_cast<unsigned char*>(ws);
        const int total = a.B * a.H * N;
        dim3 gp(static_cast<unsigned>(total < 2 * num_sms() ? total : 2 * num_sms()));
        chunk_prep_kda_kernel<TIn><<<gp, block, kdap::SMEM_ALLOC, s>>>(mq, mk, mkt, a.beta, a.alpha, w, a.T, a.H, N,
                                                                      total);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        dim3 gc(static_cast<unsigned>(a.B * a.H), static_cast<unsigned>(a.V / VS));
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = gc;
        cfg.blockDim = dim3(chain::NT);
        cfg.dynamicSmemBytes = chain::SMEM_ALLOC;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const unsigned char* wsc = w;
        e = cudaLaunchKernelEx(&cfg, chunk_chain_kernel<TIn, true, true>, mq, mkt, mv, mo, wsc, a.S0, a.S_out, a.T,
                               a.H, a.V, N, a.scale);
        if (e == cudaErrorNotSupported) {
            (void)cudaGetLastError();
            chunk_chain_kernel<TIn, true, true><<<gc, dim3(chain::NT), chain::SMEM_ALLOC, s>>>(
                mq, mkt, mv, mo, wsc, a.S0, a.S_out, a.T, a.H, a.V, N, a.scale);
            e = cudaGetLastError();
        }
        return e;
    }
    const size_t need = static_cast<size_t>(a.B) * a.H * N * WS_CHUNK;
    if (ws != nullptr && ws_bytes >= need) {
        unsigned char* w = static_cast<unsigned char*>(ws);
        const int BH = a.B * a.H;
        const int total = BH * N;
        int G = a.alpha ? 1 : seg_count(a.B, a.H, a.T, a.V);
        SegWs sw{};
        if (G > 1) {
            sw = seg_ws(a, G);
            if (ws_bytes < sw.total || !make_map(&mg, w + sw.gbuf, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, KD, a.H, rows)) G = 1;
        }
        if (G == 1) mg = mo;  // (unused)
        const int n_seg = (N + G - 1) / G;
        if (!chain_only) {
            dim3 gp(static_cast<unsigned>(total < 3 * num_sms() ? total : 3 * num_sms()));
            chunk_prep_kernel<TIn><<<gp, block, prep::SMEM_ALLOC, s>>>(mq, mk, mkt, a.beta, a.alpha, w, a.T, a.H, N,
                                                                      total);
            cudaError_t e = cudaGetLastError();
            if (e != cudaSuccess) return e;
        }
        ChainSeg sg{n_seg, a.V / VS, G > 1 ? reinterpret_cast<float*>(w + sw.z) : nullptr,
                    G > 1 ? reinterpret_cast<float*>(w + sw.p) : nullptr};
        static_assert(KD == 2 * 64, "transition slices: as many as value slices when V = K");
        dim3 gc(static_cast<unsigned>(BH), static_cast<unsigned>((a.V / VS) * (2 * G - 1)));
        // programmatic dependent launch: the chain CTAs take SMs as the previous kernel's CTAs
        // leave and wait (griddepcontrol.wait) for its results
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = gc;
        cfg.blockDim = dim3(chain::NT);
        cfg.dynamicSmemBytes = chain::SMEM_ALLOC;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const unsigned char* wsc = w;
        cudaError_t e;
        if (G > 1) {
            e = cudaLaunchKernelEx(&cfg, chunk_chain_seg_kernel<TIn>, mq, mkt, mv, mo, mg, sg, wsc, a.S0, a.S_out, a.T,
                                   a.H, a.V, N, a.scale);
        } else {
            auto chain_kernel = a.alpha ? chunk_chain_kernel<TIn, true> : chunk_chain_kernel<TIn, false>;
            e = cudaLaunchKernelEx(&cfg, chain_kernel, mq, mkt, mv, mo, wsc, a.S0, a.S_out, a.T, a.H, a.V, N, a.scale);
        }
        if (e == cudaErrorNotSupported) {  // no dependent launch here: an ordinary one
            (void)cudaGetLastError();
            if (G > 1) {
                chunk_chain_seg_kernel<TIn><<<gc, dim3(chain::NT), chain::SMEM_ALLOC, s>>>(
                    mq, mkt, mv, mo, mg, sg, wsc, a.S0, a.S_out, a.T, a.H, a.V, N, a.scale);
            } else {
                auto chain_kernel = a.alpha ? chunk_chain_kernel<TIn, true> : chunk_chain_kernel<TIn, false>;
                chain_kernel<<<gc, dim3(chain::NT), chain::SMEM_ALLOC, s>>>(mq, mkt, mv, mo, wsc, a.S0, a.S_out, a.T,
                                                                           a.H, a.V, N, a.scale);
            }
            e = cudaGetLastError();
        }
        if (e != cudaSuccess || G == 1) return e;
        // the segments' start states (and S_out), then the later segments' output correction
        float* sst = reinterpret_cast<float*>(w + sw.sst);
        seg_combine_kernel<<<dim3(static_cast<unsigned>(BH), static_cast<unsigned>(a.V / 16)), 256, COMBINE_SMEM, s>>>(
            sg.Z, sg.P, sst, a.S_out, G, a.V);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        const int per = (2 * num_sms() + BH * (G - 1) - 1) / (BH * (G - 1));  // about two CTAs per SM
        const int pairs = (n_seg + 1) / 2;
        dim3 gr(static_cast<unsigned>(BH), static_cast<unsigned>(G - 1),
                static_cast<unsigned>(per < pairs ? (per > 0 ? per : 1) : pairs));
        seg_correct_kernel<TIn><<<gr, 128, segc::SMEM_ALLOC, s>>>(mg, mo, sst, a.T, a.H, a.V, N, n_seg);
        return cudaGetLastError();
    }
    if (a.alpha) return cudaErrorNotSupported;  // the gate is carried by the two-kernel path only
    dim3 grid(static_cast<unsigned>(a.B * a.H), static_cast<unsigned>(a.V / VS));
    chunk_tc_kernel<TIn><<<grid, block, fused::SMEM_ALLOC, s>>>(mq, mk, mkt, mv, a.beta, a.S0, static_cast<TIn*>(a.o),
                                                        a.S_out, a.T, a.H, a.V, a.scale);
    return cudaGetLastError();
}

bool tc_covers(const OsdnChunkArgs& a) {
    // (one state gate per key channel: only with a workspace, through its own prep kernel)
    return a.K == KD && a.V % VS == 0 && a.chunk == C && a.T > 0 && a.T % C == 0 &&
           (a.dtype == OSDN_BF16 || a.dtype == OSDN_F16);
}

// Workspace of the fused layer: [scan: step sizes, block-start states][chunk counter][chunk
// images], each part 256-byte aligned.
struct LayerWs {
    size_t scan, counter, chunk, total;
};
LayerWs layer_ws(const OsdnScanArgs& sa, const OsdnChunkArgs& ca) {
    auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    LayerWs l{};
    const size_t nblk = static_cast<size_t>(ca.T / C);
    l.scan = 0;
    l.counter = up(osdn_scan_block_workspace_bytes(sa));
    l.chunk = l.counter + 256;
    l.total = l.chunk + up(osdn_chunk_tc_workspace_bytes(ca));
    (void)nblk;
    return l;
}

bool layer_covers(const OsdnScanArgs& sa, const OsdnChunkArgs& ca) {
    return tc_covers(ca) && !(ca.alpha && ca.alpha_per_key) && ca.V == KD && sa.K == KD && sa.k_dtype == ca.dtype && sa.kt_dtype == ca.dtype && !sa.r_per_key &&
           ca.B * ca.H < num_sms() && osdn_scan_block_workspace_bytes(sa) > 0;
}

template <typename TIn, bool HAS_R>
cudaError_t launch_layer_t(const OsdnScanArgs& sa, const OsdnChunkArgs& ca, unsigned char* ws, cudaStream_t s) {
    const CUtensorMapDataType dt = std::is_same<TIn, __half>::value ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                                    : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const long long rows = static_cast<long long>(ca.B) * ca.T;
    CUtensorMap mq, mk, mkt;
    if (!make_map(&mq, ca.q, dt, ca.K, ca.H, rows) || !make_map(&mk, ca.k, dt, ca.K, ca.H, rows) ||
        !make_map(&mkt, sa.k_tilde, dt, ca.K, ca.H, rows))
        return cudaErrorNotSupported;
    auto kernel = layer_scan_prep_kernel<TIn, HAS_R>;
    constexpr uint32_t kWorkSmem = LAYER_WORKERS * prep::REGION + 1024;
    const uint32_t smem = scanblk::SMEM_ALLOC > kWorkSmem ? scanblk::SMEM_ALLOC : kWorkSmem;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] { attr_err = set_smem(kernel, smem); });
    if (attr_err != cudaSuccess) return attr_err;
    // every CTA must be resident at once: one per SM, phase 1 on BH of them, prep on the rest
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, LAYER_NT, smem) != cudaSuccess || per_sm < 1)
        return cudaErrorNotSupported;
    const int grid = per_sm * num_sms();
    if (grid <= ca.B * ca.H) return cudaErrorNotSupported;
    const LayerWs l = layer_ws(sa, ca);
    // all-ones over the scan part (nothing published yet) and the counter
    cudaError_t e = cudaMemsetAsync(ws + l.scan, 0xff, l.counter + 4 - l.scan, s);
    if (e != cudaSuccess) return e;
    OsdnScanArgs sa2 = sa;
    float* ws_g = reinterpret_cast<float*>(ws + l.scan);
    float* ws_d = ws_g + static_cast<size_t>(sa.B) * sa.H * sa.T;
    unsigned int* counter = reinterpret_cast<unsigned int*>(ws + l.counter);
    unsigned char* cws = ws + l.chunk;
    int N = ca.T / C, BH = ca.B * ca.H;
    const float* alpha = ca.alpha;
    uint32_t poll_limit = g_poll_limit.load();
    if (poll_limit == 0) poll_limit = kMaxPolls;
    void* args[] = {&sa2, &ws_g, &ws_d, &counter, &mq, &mk, &mkt, &alpha, &cws, &N, &BH, &poll_limit};
    e = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kernel), dim3(static_cast<unsigned>(grid)),
                                    dim3(LAYER_NT), args, smem, s);
    if (e == cudaErrorCooperativeLaunchTooLarge) {  // fewer resident CTAs than expected: two calls
        (void)cudaGetLastError();
        return cudaErrorNotSupported;
    }
    if (e != cudaSuccess) return e;
    // the serial chain over the chunk images (same kernel as osdn_chunk_fwd's workspace path)
    return launch_tc<TIn>(ca, cws, l.total - l.chunk, s, /*chain_only=*/true);
}

}  // namespace

bool make_row_tmap(CUtensorMap* m, const void* ptr, CUtensorMapDataType dt, int inner, int H, long long rows) {
    return make_map(m, ptr, dt, inner, H, rows);
}
int device_sm_count() { return num_sms(); }

}  // namespace osdn

size_t osdn_layer_workspace_bytes(const OsdnScanArgs& sa, const OsdnChunkArgs& ca) {
    if (!osdn::layer_covers(sa, ca)) return 0;
    return osdn::layer_ws(sa, ca).total;
}

// Fused layer (scan + chunk prep in one cooperative launch, then the chain kernel);
// cudaErrorNotSupported when it does not apply (the caller then runs the two entry points).
cudaError_t osdn_launch_layer(const OsdnScanArgs& sa, const OsdnChunkArgs& ca, void* ws, size_t ws_bytes,
                              cudaStream_t s) {
    if (!osdn::layer_covers(sa, ca) || ws == nullptr || ws_bytes < osdn::layer_ws(sa, ca).total)
        return cudaErrorNotSupported;
    unsigned char* w = static_cast<unsigned char*>(ws);
    if (ca.dtype == OSDN_BF16)
        return sa.r ? osdn::launch_layer_t<__nv_bfloat16, true>(sa, ca, w, s)
                    : osdn::launch_layer_t<__nv_bfloat16, false>(sa, ca, w, s);
    return sa.r ? osdn::launch_layer_t<__half, true>(sa, ca, w, s) : osdn::launch_layer_t<__half, false>(sa, ca, w, s);
}

size_t osdn_chunk_tc_plain_workspace_bytes(const OsdnChunkArgs& a) {
    if (!osdn::tc_covers(a) || (a.alpha && a.alpha_per_key)) return 0;
    return static_cast<size_t>(a.B) * a.H * (a.T / osdn::C) * osdn::WS_CHUNK;
}

// With the segment scratch where the shape would use segments (whatever the gate: the size
// query does not see it).
size_t osdn_chunk_tc_workspace_bytes(const OsdnChunkArgs& a) {
    if (!osdn::tc_covers(a)) return 0;
    if (a.alpha && a.alpha_per_key) return static_cast<size_t>(a.B) * a.H * (a.T / osdn::C) * osdn::WS_CHUNK_KDA;
    const int G = osdn::seg_count(a.B, a.H, a.T, a.V);
    if (G > 1) return osdn::seg_ws(a, G).total;
    return osdn_chunk_tc_plain_workspace_bytes(a);
}

cudaError_t osdn_launch_chunk_tc(const OsdnChunkArgs& a, void* ws, size_t ws_bytes, cudaStream_t s) {
    if (!osdn::tc_covers(a)) return cudaErrorNotSupported;
    if (a.dtype == OSDN_BF16) return osdn::launch_tc<__nv_bfloat16>(a, ws, ws_bytes, s);
    return osdn::launch_tc<__half>(a, ws, ws_bytes, s);
}

cudaError_t osdn_scan_block_read_and_clear_timeout(unsigned int* flag);

cudaError_t osdn_read_and_clear_range(unsigned int* flag) {
    cudaError_t e = cudaMemcpyFromSymbol(flag, osdn::g_range_flag, sizeof(unsigned int));
    if (e != cudaSuccess || *flag == 0) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(osdn::g_range_flag, &zero, sizeof(unsigned int));
}

cudaError_t osdn_read_and_clear_timeout(unsigned int* flag, cudaStream_t s) {
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    unsigned int scan_flag = 0;
    e = osdn_scan_block_read_and_clear_timeout(&scan_flag);
    if (e != cudaSuccess) return e;

    e = cudaMemcpyFromSymbol(flag, osdn::g_timeout_flag, sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    if (*flag) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(osdn::g_timeout_flag, &zero, sizeof(unsigned int));
    }
    *flag |= scan_flag;
    return e;
}

extern "C" void osdn_set_poll_limit(unsigned int polls) { osdn::g_poll_limit.store(polls); }
