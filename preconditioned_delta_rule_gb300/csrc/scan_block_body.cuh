// scan_block_body.cuh -- the blocked phase-1 scan for one (batch, head), shared by the
// standalone scan kernel and the fused layer kernel.
//
// "OSDN: Improving Delta Rule with Provable Online Preconditioning in Linear Attention",
// Section 4.2 (Algorithm 1, Eq. (4)), Section 4.4 (APF, Eq. (7)), Appendix A.5 (Prop. A.3: the
// step is affine in d before the projection).  Per (batch, head), token by token:
//   k~_t = d_t . k_t;   a_t = <d_t, s_t>, s_t = k_t . k_t;   g_t = gamma_t (1 - b_t a_t),
//   gamma_t = eta b_t / max(|k_t|^2, eps);   d_{t+1} = clip(r_t d_t + g_t s_t, d_min, d_max).
//
// Blocked evaluation of the serial part.  Inside a block starting at token p with state d_p,
// suppose each coordinate is FREE (never clipped in the block) or PINNED at a bound b_i (clipped
// at every step).  For free coordinates the affine recurrence unrolls to
//   d_j = rho_j (d_p + sum_{l=p}^{j-1} h_l s_l),  rho_j = prod_{m=p}^{j-1} r_m,  h_l = g_l / rho_{l+1},
// so a_j = rho_j (cF_j + sum_{l<j} h_l M_jl) + cP_j with cF_j = <d_p, s_j>_free,
// cP_j = <b, s_j>_pinned and the Gram M_jl = <s_j, s_l>_free (tensor cores, computed ahead).  The
// g_j then solve a 64 x 64 unit-lower-triangular system: Jacobi sweeps until no g moves by more
// than an ulp (the coupling gamma b M is ~1e-3, so two or three sweeps).  The block end follows
// as d_64 = rho_64 (d_p + sum_l h_l s_l).  The assumption is checked per coordinate: a cheap
// sufficient bound on the free trajectory (d_p +- sum_l |h_l| s_l, scaled by the extreme rho),
// otherwise the exact trajectory; pinned coordinates must keep being clipped at every step.  At
// the first violation the tokens before it are accepted and the state after it is formed with
// the clip.  The rest of the block, and every block that starts with free and pinned coordinates
// together, is solved by Jacobi sweeps on the clipped recurrence itself: each coordinate runs its
// own clipped trajectory under a guess of the g's and the products d_j s_j, summed across the
// coordinates, give the next guess.  The clip is 1-Lipschitz, so the same coupling bound fixes
// the number of sweeps.  The result is the sequential algorithm's, up to reassociation.  d is
// carried across blocks as an unevaluated fp32 pair (hi + lo).
//
// Mapping: one CTA of 256 threads per (batch, head).  Warpgroup 0 ("chain") runs the serial part
// above, one key coordinate per thread, reading s = k.k straight from the staged keys (the square
// of a 16-bit key is exact in fp32).  Warpgroup 1 prepares block b+1 (cp.async staging of the keys
// three blocks ahead, the norms |k_t|^2 and gates; when the chain used a Gram in its latest block,
// power-of-two-scaled fp16 hi/lo copies of s and the Gram on the tensor cores, copied to shared
// memory as the chain's Jacobi rows; the fp32 s rows), writes the step sizes and start state of
// block b to the workspace when there is one, and otherwise emits the write keys of block b by
// replaying the clipped recurrence with the chain's g values.  The warpgroups hand blocks over
// through mbarriers.

#pragma once
#include <type_traits>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace osdn {
namespace scanblk {



constexpr int J = 64;              // tokens per block
constexpr int KD = 128;            // key dim (one coordinate per thread of each warpgroup)
constexpr int NT = 256;
constexpr int KROW = KD * 2 + 16;  // padded raw key row (16-bit elements), bytes
constexpr uint32_t kMaxPolls = 1u << 22;

constexpr uint32_t OFF_KT = 0;                             // 3 raw key tiles
constexpr uint32_t KT_BYTES = J * KROW;                    // 17408
// Two slots of fp16 copies of s = k.k scaled by a power of two, 128-byte swizzled.  Per key block
// (coordinates 0-63, 64-127) the 64 hi rows are followed by the 64 lo rows, so that one N = 128
// operand holds [hi; lo].
constexpr uint32_t OFF_SHL = 53248;
constexpr uint32_t SHL_SLOT = 32768, SHL_KB = 16384, SHL_LO = 8192;
// Two slots of s = k.k in fp32 (rows of SROW floats) for the chain.  SROW = 132: row j's 16-byte
// piece c sits in bank group (j + c) mod 8, which the chain's two-threads-per-row reads keep apart.
constexpr int SROW = KD + 4;
constexpr uint32_t OFF_SF = OFF_SHL + 2 * SHL_SLOT;
constexpr uint32_t SF_BYTES = J * SROW * 4;                // 33792
constexpr uint32_t OFF_F = OFF_SF + 2 * SF_BYTES;          // fp32 scratch
constexpr int F_GAM = 0;              // [2][64] gamma of the block in a slot
constexpr int F_BP = F_GAM + 128;     // [2][64] feedback beta
constexpr int F_RR = F_BP + 128;      // [2][64] retention (1 past the end of the sequence)
constexpr int F_RAWB = F_RR + 128;    // [3][64] cp.async destination for beta
constexpr int F_RAWR = F_RAWB + 192;  // [3][64] cp.async destination for r
constexpr int F_SIGS = F_RAWR + 192;  // [2] power-of-two scale of the fp16 s copies
constexpr int F_RHO = F_SIGS + 4;     // [65] (chain)
constexpr int F_G = F_RHO + 68;       // [64] g of the current sub-block (chain)
constexpr int F_H = F_G + 64;         // [2][64] h = g / rho, double-buffered across Jacobi sweeps
constexpr int F_CF = F_H + 128;       // [64]
constexpr int F_CP = F_CF + 64;       // [64]
constexpr int F_DF = F_CP + 64;       // [128] d of free coordinates (0 if pinned)
constexpr int F_BPV = F_DF + 128;     // [128] bound of pinned coordinates (0 if free)
constexpr int F_RED = F_BPV + 128;    // [8] chain reductions
constexpr int F_RED1 = F_RED + 8;     // [8] prep reductions
constexpr int F_INT = F_RED1 + 8;     // [8] int scratch (chain)
constexpr int F_GOUT = F_INT + 8;     // [2][64] final g of each token of a block (chain -> emit)
constexpr int F_DST = F_GOUT + 128;   // [2][128] state at the block start, hi part (chain -> emit)
constexpr int F_DSL = F_DST + 256;    // [2][128] state at the block start, lo part
constexpr int F_NU = F_DSL + 256;     // [2][4] coupling bound of the block in a slot (per copy warp)
constexpr int F_NRM = F_NU + 8;       // [2][64] |k_j|^2 of the block in a slot
constexpr int F_SMX = F_NRM + 128;    // [2][64] max_i k_{j,i}^2 of the block in a slot
constexpr int F_END = F_SMX + 128;
constexpr uint32_t OFF_BAR = OFF_F + ((F_END * 4 + 127) / 128) * 128;
constexpr uint32_t SMEM_BASE = OFF_BAR + 128;
// the all-free Gram of a block (two slots), scaled and masked to l < j, fp32 rows of MROW floats
// (the third gate slot of the vector-retention mode, which has no Gram)
constexpr int MROW = J + 4;
constexpr uint32_t MT_BYTES = J * MROW * 4;
constexpr uint32_t OFF_MT = ((SMEM_BASE + 127) / 128) * 128;
constexpr uint32_t SMEM_USED = OFF_MT + 2 * MT_BYTES;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;
// Vector retention (one gate per key coordinate, RM = 2): the gates of a block, J x KD fp32 rows,
// staged with its keys in three slots, in the space of the fp16 s copies and the Gram rows (that
// mode takes no Gram: every block runs the clipped sweeps).
constexpr uint32_t RV_BYTES = J * KD * 4;
__device__ __forceinline__ uint32_t rv_off(int slot) { return slot < 2 ? OFF_SHL + slot * SHL_SLOT : OFF_MT; }
static_assert(SHL_SLOT >= RV_BYTES && 2 * MT_BYTES >= RV_BYTES && OFF_MT % 16 == 0, "gate slots");
static_assert(3 * KT_BYTES <= OFF_SHL, "key tiles");
static_assert(OFF_SHL % 1024 == 0, "swizzle atoms");
static_assert(SMEM_ALLOC <= 232448, "shared memory");

constexpr uint32_t TMEM_COLS = 256;
constexpr uint32_t COL_G = 0;     // all-free Gram products of the block in slot q: columns 128 q ..

// mbarriers (offsets from OFF_BAR): gram[2], prep_ready[2], chain_done[2], Gram rows in shared
// memory[2]
constexpr uint32_t B_GRAM = 0, B_PREP = 16, B_CHAIN = 32, B_MRDY = 48;

__device__ __forceinline__ void cp_async_16z(void* smem, const void* gmem, bool valid) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    const int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_4z(void* smem, const void* gmem, bool valid) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    const int n = valid ? 4 : 0;
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(s), "l"(gmem), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

// Barrier over one warpgroup (128 threads) with hardware barrier `id` (1 or 2).
__device__ __forceinline__ void wg_sync(int id) { asm volatile("bar.sync %0, 128;\n" ::"r"(id) : "memory"); }
// All NT threads of the scan (a CTA may carry more threads that do not take part in the scan).
__device__ __forceinline__ void scan_sync() { asm volatile("bar.sync 4, 256;\n" ::: "memory"); }
// Barrier over one warpgroup that also counts the threads with `pred` set.
__device__ __forceinline__ int wg_count(int id, bool pred) {
    int c;
    asm volatile("{\n .reg .pred p;\n setp.ne.u32 p, %2, 0;\n bar.red.popc.u32 %0, %1, 128, p;\n}\n"
                 : "=r"(c)
                 : "r"(id), "r"(static_cast<int>(pred))
                 : "memory");
    return c;
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
}

template <typename TIn>
__device__ __forceinline__ float ld_key(const unsigned char* tile, int j, int i) {
    return to_f32(*reinterpret_cast<const TIn*>(tile + j * KROW + i * 2));
}

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = a + b;
    const float z = s - a;
    e = (a - (s - z)) + (b - z);
}
// (hi, lo) <- rho * (hi + lo + inc), renormalised.
__device__ __forceinline__ void pair_advance(float& hi, float& lo, float inc, float rho) {
    float s, e;
    two_sum(hi, inc, s, e);
    e += lo;
    float h2 = s + e;
    float l2 = e - (h2 - s);
    if (rho != 1.f) {
        const float p = rho * h2;
        const float ep = fmaf(rho, h2, -p);
        const float l3 = fmaf(rho, l2, ep);
        h2 = p + l3;
        l2 = l3 - (h2 - p);
    }
    hi = h2;
    lo = l2;
}
// min(max(a b + c, 0), 1) in one instruction (fma.rn.sat: NaN gives 0).
__device__ __forceinline__ float fma_sat(float a, float b, float c) {
    float r;
    asm("fma.rn.sat.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
__device__ __forceinline__ void pair_clip(float& hi, float& lo, float dmin, float dmax) {
    if (hi < dmin || (hi == dmin && lo < 0.f)) { hi = dmin; lo = 0.f; }
    if (hi > dmax || (hi == dmax && lo > 0.f)) { hi = dmax; lo = 0.f; }
}

// One halving step of a sum over the lanes of a warp of L values held by each lane: the lanes
// with bit O set keep the upper half, the others the lower half, each adding its partner's copy of
// the half it keeps.  After the steps for O = 16, 8, 4, 2, 1 (L = 64 .. 4) lane l holds in v[0],
// v[1] the warp sums of entries 2 l and 2 l + 1.
template <int L, int O>
__device__ __forceinline__ void rs_level(float (&v)[64], int lane) {
    const bool up = (lane & O) != 0;
#pragma unroll
    for (int t = 0; t < L / 2; ++t) {
        const float keep = up ? v[t + L / 2] : v[t];
        const float send = up ? v[t] : v[t + L / 2];
        v[t] = keep + __shfl_xor_sync(0xffffffffu, send, O);
    }
}

// The body of the blocked scan for one (batch, head) `bh`, run by 256 threads of a CTA whose
// dynamic shared memory starts at smem_raw (SMEM_ALLOC bytes) and which holds TMEM_COLS columns
// of tensor memory at `tbase` (allocated and released by the caller).  On return no asynchronous
// operation of the body is in flight and its mbarriers are retired, so the caller may reuse the
// shared and tensor memory.  A bounded wait that gives up sets *timeout_flag.  With a workspace
// (ws_g, ws_d) the step sizes and start state of every block are stored there as soon as the
// block is solved, each word with one relaxed GPU-scope store and never with the all-ones bit
// pattern, so a consumer running concurrently may poll for them.
// RM: 0 no retention, 1 one gate per token and head (Eq. (7)), 2 one gate per key coordinate
// (diag(r_t), Appendix A.5; no Gram: each block runs the clipped sweeps, whose trajectories take
// a gate per coordinate as they are, with the coupling bound from |gamma_j b_j| <s_j, sum_l s_l>).
template <typename TIn, typename TOut, int RM>
__device__ __forceinline__ void scan_block_body(const OsdnScanArgs& a, float* ws_g, float* ws_d, int bh,
                                                unsigned char* smem_raw, uint32_t tbase,
                                                unsigned int* timeout_flag) {
    unsigned char* sm = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    float* F = reinterpret_cast<float*>(sm + OFF_F);
    int* FI = reinterpret_cast<int*>(F + F_INT);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int b = bh / a.H, h = bh % a.H;
    const int T = a.T, H = a.H;
    constexpr bool HAS_R = RM == 1;  // per-token gates in F_RR
    constexpr bool VEC = RM == 2;    // per-coordinate gates in the slots at rv_off
    const TIn* kg = static_cast<const TIn*>(a.k);
    TOut* ktg = static_cast<TOut*>(a.k_tilde);
    const size_t row0 = static_cast<size_t>(b) * T * H + h;
    const int nblk = (T + J - 1) / J;
    const uint32_t sbase = tc::smem_u32(sm);
    const uint32_t bars = sbase + OFF_BAR;
    const float eta = a.eta, dmin = a.d_min, dmax = a.d_max, eps = a.eps;
    __shared__ int s_abort;
    // With per-head retention gates the Gram of a block is formed only when the chain used one in
    // its latest finished block (s_gram_want: every block of a head tends to take the same path;
    // APF gates hold d on d_min, and a block with every coordinate there needs no Gram).  Without
    // gates whole pinned blocks are rare and every block forms its Gram.  Per slot: whether this
    // block's Gram is formed (s_gon), the parity of its barrier phase (s_gpar) and the number of
    // Grams issued on the slot's barrier so far (s_gcnt).
    __shared__ int s_gram_want, s_gram_used, s_gon[2], s_gpar[2], s_gcnt[2];

    if (tid == 0) {
        for (int q = 0; q < 2; ++q) {
            tc::mbar_init(bars + B_GRAM + 8 * q, 1);
            tc::mbar_init(bars + B_PREP + 8 * q, 4);
            tc::mbar_init(bars + B_CHAIN + 8 * q, 128);
        }
        tc::mbar_init(bars + B_MRDY, 4);
        tc::mbar_init(bars + B_MRDY + 8, 4);
        tc::mbar_init_fence();
        s_abort = 0;
        s_gram_want = 1;
        s_gcnt[0] = s_gcnt[1] = 0;
    }
    scan_sync();
    const uint32_t id_hl = tc::idesc_f16_f32(J, 2 * J, false, false);  // M = 64, N = 128
    const uint32_t id_lh = tc::idesc_f16_f32(J, J, false, false);      // M = 64, N = 64

    // Gram products of the s copies in slot q into the 128 TMEM columns at `col`, M = 64: first
    // hi.[hi; lo]^T (N = 128), then lo.hi^T accumulated onto the first 64 columns, so that row j
    // of the Gram is M_j = D_j[0:64] + D_j[64:128] = hi.hi^T + lo.hi^T + hi.lo^T (lo.lo^T is
    // below fp32 rounding).  An M = 64 product puts row j in lane 32 (j / 16) + j % 16: rows
    // 16 w .. 16 w + 15 in the first 16 lanes of warp quadrant w.
    auto issue_gram = [&](int q, uint32_t col, uint32_t bar) {
        const uint32_t base = sbase + OFF_SHL + q * SHL_SLOT;
        tc::tc_fence_after();
#pragma unroll
        for (int st = 0; st < KD / 16; ++st) {
            const uint64_t d = tc::sdesc_sw128(base + (st >> 2) * SHL_KB + (st & 3) * 32, 16, 1024);
            tc::mma_f16(tbase + col, d, d, id_hl, st > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int st = 0; st < KD / 16; ++st) {
            const uint32_t a = base + (st >> 2) * SHL_KB + (st & 3) * 32;
            tc::mma_f16(tbase + col, tc::sdesc_sw128(a + SHL_LO, 16, 1024), tc::sdesc_sw128(a, 16, 1024), id_lh, 1u);
        }
        tc::mma_commit(bar);
    };
    // The Gram row of the calling lane of a warp of quadrant `lane_base` (row j = 16 w + lane for
    // lanes 0-15; the other lanes load what they load), scaled by 1 / sig^2 and masked to l < j.
    // Warp-collective: every lane of the warp must call it.
    auto load_gram_row = [&](uint32_t col, uint32_t lane_base, int j, float inv_sig2, float (&mrow)[64]) {
#pragma unroll
        for (int hv = 0; hv < 2; ++hv) {
            float x[32], y[32];
            tc::tmem_ld32(tbase + lane_base + col + hv * 32, x);
            tc::tmem_ld32(tbase + lane_base + col + 64 + hv * 32, y);
            tc::tmem_ld_wait();
#pragma unroll
            for (int l = 0; l < 32; ++l) mrow[hv * 32 + l] = (hv * 32 + l < j) ? (x[l] + y[l]) * inv_sig2 : 0.f;
        }
    };

    if (warp >= 4) {
        // =========================== warpgroup 1: staging, prep, emission ======================
        const int u = tid - 128;
        auto stage = [&](int m) {
            if (m < nblk) {
                unsigned char* dst = sm + OFF_KT + (m % 3) * KT_BYTES;
                const int t0 = m * J;
#pragma unroll
                for (int e = 0; e < (J * KD * 2 / 16) / 128; ++e) {
                    const int piece = e * 128 + u, j = piece >> 4, c = piece & 15;
                    const bool valid = t0 + j < T;
                    const size_t row = row0 + static_cast<size_t>(valid ? t0 + j : 0) * H;
                    cp_async_16z(dst + j * KROW + c * 16, reinterpret_cast<const unsigned char*>(kg + row * KD) + c * 16, valid);
                }
                if (u < J) {
                    const bool valid = t0 + u < T;
                    const size_t row = row0 + static_cast<size_t>(valid ? t0 + u : 0) * H;
                    cp_async_4z(F + F_RAWB + (m % 3) * J + u, a.beta + row, valid);
                    if (HAS_R) cp_async_4z(F + F_RAWR + (m % 3) * J + u, a.r + row, valid);
                }
                if (VEC) {  // the block's gates, row j = token (zeros past the end: never read)
                    float* dst = reinterpret_cast<float*>(sm + rv_off(m % 3));
#pragma unroll
                    for (int e = 0; e < (J * KD * 4 / 16) / 128; ++e) {
                        const int piece = e * 128 + u, j = piece >> 5, c = piece & 31;
                        const bool valid = t0 + j < T;
                        const size_t row = row0 + static_cast<size_t>(valid ? t0 + j : 0) * H;
                        cp_async_16z(dst + j * KD + c * 4, a.r + row * KD + c * 4, valid);
                    }
                }
            }
            cp_async_commit();
        };
        // block m: s = k.k in fp32 (slot m&1), scaled fp16 hi/lo copies, gates; then its Gram
        auto prepare = [&](int m) {
            const unsigned char* kt = sm + OFF_KT + (m % 3) * KT_BYTES;
            float* sf = reinterpret_cast<float*>(sm + OFF_SF + (m & 1) * SF_BYTES);
            const int j = u >> 1, hf = u & 1;
            float n = 0.f, mx = 0.f;
            float sv[64];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                float kv[8];
                VecIO<TIn, 4>::load(reinterpret_cast<const TIn*>(kt + j * KROW + hf * 128 + c * 16), kv);
                VecIO<TIn, 4>::load(reinterpret_cast<const TIn*>(kt + j * KROW + hf * 128 + c * 16 + 8), kv + 4);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    sv[c * 8 + e] = kv[e] * kv[e];
                    n += sv[c * 8 + e];
                    mx = fmaxf(mx, sv[c * 8 + e]);
                }
            }
            n += __shfl_xor_sync(0xffffffffu, n, 1);
            const float rowmx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            if ((u & 31) == 0) F[F_RED1 + (u >> 5)] = mx;
            if (hf == 0) {
                const int q = m & 1;
                const bool valid = m * J + j < T;
                const float bt = F[F_RAWB + (m % 3) * J + j];
                const float bp = a.beta_aware ? bt : 1.f;
                F[F_GAM + q * J + j] = valid ? eta * bp / fmaxf(n, eps) : 0.f;
                if (!VEC) {
                    F[F_NRM + q * J + j] = n;
                    F[F_SMX + q * J + j] = rowmx;
                }
                F[F_BP + q * J + j] = bp;
                F[F_RR + q * J + j] = (HAS_R && valid) ? F[F_RAWR + (m % 3) * J + j] : 1.f;
            }
            if constexpr (VEC) {
                // the fp32 s rows for the chain, then the coupling bound of the block
                __syncwarp();
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    float4* dst = reinterpret_cast<float4*>(sf + j * SROW + hf * 64 + c * 8);
                    dst[0] = make_float4(sv[c * 8], sv[c * 8 + 1], sv[c * 8 + 2], sv[c * 8 + 3]);
                    dst[1] = make_float4(sv[c * 8 + 4], sv[c * 8 + 5], sv[c * 8 + 6], sv[c * 8 + 7]);
                }
                __syncwarp();
                if ((u & 31) == 0) mbar_arrive(bars + B_PREP + 8 * (m & 1));
                wg_sync(2);
                // coordinate u: sum of s over the block's tokens, and whether a gate exceeds 1
                const float* rv = reinterpret_cast<const float*>(sm + rv_off(m % 3));
                const int jb = min(J, T - m * J);
                float cs = 0.f;
                bool rbad = false;
#pragma unroll 8
                for (int l = 0; l < J; ++l) {
                    cs += sf[l * SROW + u];
                    if (l < jb) rbad |= !(rv[l * KD + u] <= 1.f);
                }
                float* colsum = F + F_NRM;  // (the per-block norms of the Gram path: unused here)
                colsum[u] = cs;
                wg_sync(2);
                // sum_{l<j} M_jl <= <s_j, sum_l s_l> (s >= 0): the sweeps' contraction bound
                float dot = 0.f;
#pragma unroll
                for (int c = 0; c < 64; ++c) dot = fmaf(sv[c], colsum[hf * 64 + c], dot);
                dot += __shfl_xor_sync(0xffffffffu, dot, 1);
                const int q = m & 1;
                float tb = fabsf(F[F_GAM + q * J + j] * F[F_BP + q * J + j]) * dot;
                if (!(tb <= 3.0e38f)) tb = INFINITY;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) tb = fmaxf(tb, __shfl_xor_sync(0xffffffffu, tb, o));
                const bool bad = __any_sync(0xffffffffu, rbad);
                if ((u & 31) == 0) F[F_NU + 4 * q + (u >> 5)] = bad ? INFINITY : tb;
                __syncwarp();
                if ((u & 31) == 0) mbar_arrive(bars + B_MRDY + 8 * q);
                return;
            }
            if (u == 0) {  // form this block's Gram? (a hint from the chain; the decision is uniform)
                const int q = m & 1;
                s_gon[q] = HAS_R ? *static_cast<volatile int*>(&s_gram_want) : 1;
                s_gpar[q] = s_gcnt[q] & 1;
            }
            wg_sync(2);
            const float bmax = fmaxf(fmaxf(F[F_RED1], F[F_RED1 + 1]), fmaxf(F[F_RED1 + 2], F[F_RED1 + 3]));
            int ex = 0;
            if (bmax > 0.f) frexpf(bmax, &ex);
            const float sig = bmax > 0.f ? ldexpf(1.f, 14 - ex) : 1.f;  // max s * sig < 2^14
            if (u == 0) F[F_SIGS + (m & 1)] = sig;
            if (!HAS_R || s_gon[m & 1]) {
                unsigned char* sh = sm + OFF_SHL + (m & 1) * SHL_SLOT + hf * SHL_KB;
                unsigned char* sl = sh + SHL_LO;
                // hi: x rounded to 11 significant bits in fp32 (add half a unit of bit 13, clear the
                // 13 low bits; a carry moves into the exponent as it should), which fp16 holds exactly
                // in its normal range (x < 2^14 here); lo = x - hi is exact, |lo| <= 2^-11 |x|.  Two
                // packing conversions a pair instead of a round trip through fp16 per value.
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    float hi[8], lo[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float x = sv[c * 8 + e] * sig;
                        hi[e] = __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xffffe000u);
                        lo[e] = x - hi[e];
                    }
                    *reinterpret_cast<uint4*>(sh + tc::sw128_off(j, c)) =
                        make_uint4(pack_h2(hi[0], hi[1]), pack_h2(hi[2], hi[3]), pack_h2(hi[4], hi[5]), pack_h2(hi[6], hi[7]));
                    *reinterpret_cast<uint4*>(sl + tc::sw128_off(j, c)) =
                        make_uint4(pack_h2(lo[0], lo[1]), pack_h2(lo[2], lo[3]), pack_h2(lo[4], lo[5]), pack_h2(lo[6], lo[7]));
                }
                tc::fence_proxy_async();
                wg_sync(2);
                // The Gram goes first (its rows are what the chain waits for longest), issued from
                // warp 6.  (copy_gram waits for every formed Gram before the slot's next one, so no
                // wait on the barrier can mistake one phase for another.)
                if (u == 2 * 32) {
                    const int q = m & 1;
                    issue_gram(q, COL_G + q * 128, bars + B_GRAM + 8 * q);
                    s_gcnt[q] = s_gcnt[q] + 1;
                }
                __syncwarp();
            }
            // then the fp32 s tile for the chain, each warp releasing the block once its rows are
            // stored
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                float4* dst = reinterpret_cast<float4*>(sf + j * SROW + hf * 64 + c * 8);
                dst[0] = make_float4(sv[c * 8], sv[c * 8 + 1], sv[c * 8 + 2], sv[c * 8 + 3]);
                dst[1] = make_float4(sv[c * 8 + 4], sv[c * 8 + 5], sv[c * 8 + 6], sv[c * 8 + 7]);
            }
            __syncwarp();
            if ((u & 31) == 0) mbar_arrive(bars + B_PREP + 8 * (m & 1));
        };

        // Gram of block m (when formed), tensor memory -> shared memory slot m & 1 as the chain's
        // Jacobi rows (one row per thread of lanes 0-15 of each warp), scaled back by 1 / sig^2
        // (exact: powers of two) and masked to l < j, with the coupling bound nu of the block's
        // system for the chain's sweep count.  B_GRAM and B_MRDY of a slot complete one phase per
        // formed Gram, so both waits take the parity warpgroup 1 recorded for the block.
        auto copy_gram = [&](int m) {
            const int q = m & 1;
            const bool okg = tc::mbar_wait(bars + B_GRAM + 8 * q, static_cast<uint32_t>(s_gpar[q]), kMaxPolls);
            if (!__all_sync(0xffffffffu, okg)) {
                atomicExch(&s_abort, 1);
                return;
            }
            tc::tc_fence_after();
            const int lane = u & 31, j = ((u >> 5) << 4) | (lane & 15);
            const float isg = 1.f / F[F_SIGS + q];
            float g[64];
            load_gram_row(COL_G + q * 128, static_cast<uint32_t>((warp & 3) * 32) << 16, j, isg * isg, g);
            tc::tc_fence_before();
            float tb = 0.f;
            if (lane < 16) {
                float* row = reinterpret_cast<float*>(sm + OFF_MT + q * MT_BYTES) + j * MROW;
#pragma unroll
                for (int l = 0; l < 64; l += 4) *reinterpret_cast<float4*>(row + l) = make_float4(g[l], g[l + 1], g[l + 2], g[l + 3]);
                // max_j |gamma_j b_j| sum_l M_jl (M >= 0); infinite when it is not finite or a
                // retention gate exceeds 1
                float r4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int l = 0; l < 64; ++l) r4[l & 3] += g[l];
                tb = fabsf(F[F_GAM + q * J + j] * F[F_BP + q * J + j]) * ((r4[0] + r4[1]) + (r4[2] + r4[3]));
                if (!(tb <= 3.0e38f) || (HAS_R && F[F_RR + q * J + j] > 1.f)) tb = INFINITY;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) tb = fmaxf(tb, __shfl_xor_sync(0xffffffffu, tb, o));
            if (lane == 0) F[F_NU + 4 * q + (u >> 5)] = tb;
            __syncwarp();
            if (lane == 0) mbar_arrive(bars + B_MRDY + 8 * q);
        };
        // step sizes and start state of block m to the workspace (warps 6-7).  A reader in
        // another CTA polls each word until it differs from the all-ones pattern the workspace
        // was filled with, so no fence or flag is needed; a value with that pattern (a NaN) is
        // written as the canonical NaN.
        auto publish = [&](int m) {
            const int v = u - J, q = m & 1;
            auto put = [](float* p, float x) {
                uint32_t w = __float_as_uint(x);
                if (w == 0xffffffffu) w = 0x7fffffffu;
                asm volatile("st.relaxed.gpu.global.b32 [%0], %1;\n" ::"l"(p), "r"(w) : "memory");
            };
            if (m * J + v < T) put(ws_g + static_cast<size_t>(bh) * T + m * J + v, F[F_GOUT + q * J + v]);
            float* wd = ws_d + (static_cast<size_t>(bh) * nblk + m) * (2 * KD);
            put(wd + v, F[F_DST + q * KD + v]);
            put(wd + v + 64, F[F_DST + q * KD + v + 64]);
            put(wd + KD + v, F[F_DSL + q * KD + v]);
            put(wd + KD + v + 64, F[F_DSL + q * KD + v + 64]);
        };

        stage(0);
        stage(1);
        stage(2);
        if (nblk > 0) {
            cp_async_wait<2>();
            wg_sync(2);
            prepare(0);
            if (!VEC && (!HAS_R || s_gon[0])) copy_gram(0);
        }
        for (int m = 0; m < nblk; ++m) {
            if (m + 1 < nblk) {
                cp_async_wait<1>();  // groups 0..m+2 committed; block m+1's has landed
                wg_sync(2);
                prepare(m + 1);  // slot (m + 1) & 1: the chain finished block m - 1 with it
                if (!VEC && (!HAS_R || s_gon[(m + 1) & 1])) copy_gram(m + 1);
            }
            // block m once the chain has fixed its g values
            const bool ok = tc::mbar_wait(bars + B_CHAIN + 8 * (m & 1), (m >> 1) & 1, kMaxPolls);
            const bool bad = !ok || *static_cast<volatile int*>(&s_abort);
            if (wg_count(2, bad) != 0) {  // uniform decision across the warpgroup
                atomicExch(&s_abort, 1);
                break;
            }
            if (ws_g != nullptr && u >= J) publish(m);
            if (ws_g == nullptr) {  // emit here; with a workspace scan_emit_kernel does it
                const int q = m & 1;
                const unsigned char* kt = sm + OFF_KT + (m % 3) * KT_BYTES;
                const int t0 = m * J, jb = min(J, T - t0);
                float d = F[F_DST + q * KD + u] + F[F_DSL + q * KD + u];
                TOut* out = ktg + (row0 + static_cast<size_t>(t0) * H) * KD + u;
                const size_t stride = static_cast<size_t>(H) * KD;
                const float* rv = reinterpret_cast<const float*>(sm + rv_off(m % 3));
#pragma unroll 4
                for (int j = 0; j < jb; ++j) {
                    const float kj = ld_key<TIn>(kt, j, u);
                    out[j * stride] = from_f32<TOut>(d * kj);
                    const float rj = VEC ? rv[j * KD + u] : F[F_RR + q * J + j];
                    d = replay_step(d, rj, replay_inc(F[F_GOUT + q * J + j], kj), dmin, dmax);
                }
            }
            wg_sync(2);
            stage(m + 3);  // the key slot of block m is free: chain and emission are done with it
        }
    } else {
        // =========================== warpgroup 0: the serial chain =============================
        const int i = tid;
        float d_hi = a.d0 ? a.d0[static_cast<size_t>(bh) * KD + i] : 1.f, d_lo = 0.f;
        for (int blk = 0; blk < nblk; ++blk) {
            const int q = blk & 1;
            const uint32_t ph = (blk >> 1) & 1;
            const bool ok = tc::mbar_wait(bars + B_PREP + 8 * q, ph, kMaxPolls);
            const bool bad = !ok || *static_cast<volatile int*>(&s_abort);
            if (wg_count(1, bad) != 0) {  // uniform decision across the warpgroup
                atomicExch(&s_abort, 1);
                break;
            }
            tc::tc_fence_after();
            const float* sf = reinterpret_cast<const float*>(sm + OFF_SF + q * SF_BYTES);
            auto s_at = [&](int j, int c) -> float { return sf[j * SROW + c]; };
            // the 16-byte piece a chain thread reads in step c of a row: thread pairs split the
            // row so that the eight lanes of a shared-memory phase hit eight bank groups
            auto piece = [](int c, int hf) -> int { return hf ? 16 + ((c + 4) & 15) : c; };
            const float* gam = F + F_GAM + q * J;
            const float* bpv = F + F_BP + q * J;
            const float* rr = F + F_RR + q * J;
            float* gout = F + F_GOUT + q * J;
            F[F_DST + q * KD + i] = d_hi;
            F[F_DSL + q * KD + i] = d_lo;

            int p = 0;
            // vector gates: every block by the clipped sweeps (p = 0)
            bool abort_now = false, gram_rows_ready = false, clipped = VEC;
            bool have_rows = false;  // this block's Gram rows
            if (tid == 0) s_gram_used = 0;
            // vector gates of the block (tokens past the end keep d: gate 1)
            auto rvec = [&](int j) -> float {
                return j < min(J, T - blk * J) ? reinterpret_cast<const float*>(sm + rv_off(blk % 3))[j * KD + i] : 1.f;
            };
            // Waits for the all-free Gram rows of this block (copied by warpgroup 1 to shared
            // memory slot q) and the coupling bound nu = max_j |gamma_j b_j| sum_l M_jl (infinite
            // when it is not finite or a retention gate exceeds 1) for the sweep count; with one
            // gate per coordinate there is no Gram and warpgroup 1 forms nu from the s rows.
            // false: a wait gave up.  Otherwise have_rows says whether rows and bound are there:
            // with per-head gates warpgroup 1 skips a block's Gram when the chain did not use the
            // last one, and the block then runs the clipped sweeps until no step size moves, which
            // needs no bound.
            auto gram_ready = [&]() -> bool {
                if (tid == 0) s_gram_used = 1;
                if (gram_rows_ready) return true;
                if (VEC || !HAS_R || s_gon[q] != 0) {
                    const uint32_t par = VEC ? ph : static_cast<uint32_t>(s_gpar[q]);
                    const bool okr = tc::mbar_wait(bars + B_MRDY + 8 * q, par, kMaxPolls);
                    if (wg_count(1, okr && !*static_cast<volatile int*>(&s_abort)) != 128) return false;
                    have_rows = true;
                }
                gram_rows_ready = true;
                return true;
            };
            // Sweeps needed by the bound nu: each Jacobi sweep shrinks the error by nu (the largest
            // |gamma_j b_j| sum_l M_jl), so K more sweeps after an estimate within nu |g| leave
            // nu^(K+1) |g| <= 1e-7 |g|; -1: sweep until no g moves.
            auto sweeps_for_nu = [&]() -> int {
                const float nu = fmaxf(fmaxf(F[F_NU + 4 * q], F[F_NU + 4 * q + 1]), fmaxf(F[F_NU + 4 * q + 2], F[F_NU + 4 * q + 3]));
                const float nu2 = nu * nu;
                return nu <= 1e-7f ? 0 : nu2 <= 1e-7f ? 1 : nu2 * nu <= 1e-7f ? 2 : nu2 * nu2 <= 1e-7f ? 3 : -1;
            };
            while (p < J) {
                if (clipped) {
                    // ---- Jacobi sweeps on the clipped recurrence itself, tokens p..63 ----------
                    // From a guess of the g's every coordinate runs its own clipped trajectory
                    // d_{j+1} = clip(r_j d_j + g_j s_j) and the products d_j s_j summed over the
                    // coordinates give a_j and the next guess g_j = gamma_j (1 - b_j a_j).  Sweep n
                    // fixes g_p .. g_{p+n-1} exactly (the trajectory up to j needs only the g's
                    // before j); and since the clip is 1-Lipschitz and r <= 1, g's that are off by e
                    // move a_j by at most e sum_l M_jl, so each sweep shrinks the error by nu as on
                    // the unclipped system.  Starting from g = 0 (error |g|) K + 1 sweeps suffice.
                    if (!gram_ready()) {
                        abort_now = true;
                        break;
                    }
                    const int K = have_rows ? sweeps_for_nu() : -1;
                    const int nsw = K >= 0 ? min(K + 1, J - p) : J - p;
                    float* red = F + F_DF;  // [4][64] per-warp partial sums (F_DF, F_BPV: free here)
                    const int lane = tid & 31;
                    wg_sync(1);
                    if (tid < J) F[F_G + tid] = 0.f;  // tokens before p then leave d unchanged
                    wg_sync(1);
                    // With a finite box the trajectory runs in y = (d - d_min) / (d_max - d_min):
                    // y' = sat(r y + c), c = (g s + (r - 1) d_min) / (d_max - d_min) formed off the
                    // chain, one saturating fma per token on it instead of an fma, a max and a min.
                    // (Not with one gate per head, whose blocks seldom come here: its registers are
                    // the scarcest.)
                    const bool unit_box = !HAS_R && dmax > dmin && dmax - dmin < INFINITY;
                    const float bw = dmax - dmin, ibw = 1.f / bw;
                    for (int it = 0; it < nsw; ++it) {
                        float v[J];
                        float x = d_hi, y = (d_hi - dmin) * ibw;
#pragma unroll
                        for (int j4 = 0; j4 < J; j4 += 4) {
                            const float4 g4 = *reinterpret_cast<const float4*>(F + F_G + j4);
                            const float gg[4] = {g4.x, g4.y, g4.z, g4.w};
                            float r4[4] = {1.f, 1.f, 1.f, 1.f};
                            if (HAS_R) {
                                const float4 t4 = *reinterpret_cast<const float4*>(rr + j4);
                                r4[0] = t4.x;
                                r4[1] = t4.y;
                                r4[2] = t4.z;
                                r4[3] = t4.w;
                            }
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int j = j4 + e;
                                const float sj = s_at(j, i);
                                const float rj = VEC ? rvec(j) : (j >= p ? r4[e] : 1.f);
                                if (unit_box) {
                                    v[j] = fmaf(bw, y, dmin) * sj;
                                    y = fma_sat(rj, y, fmaf(gg[e], sj, (rj - 1.f) * dmin) * ibw);
                                } else {
                                    v[j] = x * sj;
                                    x = fminf(fmaxf(fmaf(rj, x, gg[e] * sj), dmin), dmax);
                                }
                            }
                        }
                        // sum over the warp: lane l keeps the sums for tokens 2 l and 2 l + 1
                        rs_level<64, 16>(v, lane);
                        rs_level<32, 8>(v, lane);
                        rs_level<16, 4>(v, lane);
                        rs_level<8, 2>(v, lane);
                        rs_level<4, 1>(v, lane);
                        *reinterpret_cast<float2*>(red + warp * J + 2 * lane) = make_float2(v[0], v[1]);
                        wg_sync(1);
                        bool changed = false;
                        if (tid >= p && tid < J) {
                            const float aj = (red[tid] + red[J + tid]) + (red[2 * J + tid] + red[3 * J + tid]);
                            const float gn = gam[tid] * (1.f - bpv[tid] * aj);
                            changed = fabsf(gn - F[F_G + tid]) > 5e-7f * fabsf(gn) + 1e-30f;
                            F[F_G + tid] = gn;
                        }
                        if (K >= 0) wg_sync(1);
                        else if (wg_count(1, changed) == 0) break;
                    }
                    if (tid >= p && tid < J) gout[tid] = F[F_G + tid];
                    // the block end with the final g's, carried as a (hi, lo) pair: hi takes one
                    // product and one sum per token, their rounding errors go to lo (off hi's
                    // dependency chain), the clip acts on the pair, and the pair is renormalised once
                    // (lo gathers at most ~64 ulps of d over the block).  Tokens before p leave it as
                    // it is (gate 1, step 0).
                    {
                        float hi = d_hi, lo = d_lo;
#pragma unroll 8
                        for (int j = 0; j < J; ++j) {
                            const bool act = j >= p;
                            const float sj = s_at(j, i), g = act ? F[F_G + j] : 0.f;
                            const float r = act ? (VEC ? rvec(j) : (HAS_R ? rr[j] : 1.f)) : 1.f;
                            const float p1 = r * hi, ep = fmaf(r, hi, -p1), q1 = g * sj;
                            float s1, e1;
                            two_sum(p1, q1, s1, e1);
                            // the clip decides on s1 + r lo (this step's rounding terms ep + e1, under
                            // an ulp, left out), so that lo's TwoSum stays off hi's chain
                            const float v = fmaf(r, lo, s1);
                            lo = fmaf(r, lo, ep + e1);
                            hi = s1;
                            if (v < dmin) { hi = dmin; lo = 0.f; }
                            if (v > dmax) { hi = dmax; lo = 0.f; }
                        }
                        d_hi = hi + lo;
                        d_lo = lo - (d_hi - hi);
                    }
                    p = J;
                    wg_sync(1);
                    break;
                }
                // ---- c_j = <d_p, s_j> over all coordinates, j >= p (2 threads per row) ----------
                // This is cF_j when every coordinate turns out free (the usual case); it also gives
                // the exact first step a_p = c_p.
                F[F_DF + i] = d_hi;
                wg_sync(1);
                {
                    const int j = tid >> 1, hf = tid & 1;
                    float cf = 0.f;
                    if (j >= p) {
                        const float* row = sf + j * SROW;
                        float c2 = 0.f;
#pragma unroll 4
                        for (int c = 0; c < 16; c += 2) {
                            const int i0 = piece(c, hf) * 4, i1 = piece(c + 1, hf) * 4;
                            const float4 s0 = *reinterpret_cast<const float4*>(row + i0);
                            const float4 d0 = *reinterpret_cast<const float4*>(F + F_DF + i0);
                            const float4 s1 = *reinterpret_cast<const float4*>(row + i1);
                            const float4 d1 = *reinterpret_cast<const float4*>(F + F_DF + i1);
                            cf = fmaf(d0.x, s0.x, fmaf(d0.y, s0.y, fmaf(d0.z, s0.z, fmaf(d0.w, s0.w, cf))));
                            c2 = fmaf(d1.x, s1.x, fmaf(d1.y, s1.y, fmaf(d1.z, s1.z, fmaf(d1.w, s1.w, c2))));
                        }
                        cf += c2;
                    }
                    cf += __shfl_xor_sync(0xffffffffu, cf, 1);
                    if (hf == 0) {
                        F[F_CF + j] = cf;
                        F[F_CP + j] = 0.f;
                    }
                }
                wg_sync(1);
                // ---- exact first step at p; classify -------------------------------------
                const float sp = s_at(p, i);
                const float gp = gam[p] * (1.f - bpv[p] * F[F_CF + p]);
                const float x = fmaf(gp, sp, rr[p] * d_hi);
                const int status = (x < dmin) ? 1 : ((x > dmax) ? 2 : 0);  // free, low, high
                const float bound = status == 1 ? dmin : dmax;
                const int nfree = wg_count(1, status == 0);
                if (tid == 0) {
                    F[F_G + p] = gp;
                    gout[p] = gp;
                }
                if (nfree > 0 && nfree < KD) {  // free and pinned coordinates: clipped sweeps
                    clipped = true;
                    continue;
                }
                bool all_low = false;  // every coordinate clipped at d_min
                if (nfree == 0) {  // every coordinate pinned: cF = 0, cP_j = <b, s_j>
                    const int nlow = wg_count(1, status == 1);
                    all_low = nlow == KD;
                    if (nlow == KD || nlow == 0) {  // all on one face: cP_j = b |k_j|^2
                        const float bd = nlow == KD ? dmin : dmax;
                        if (tid < J && tid > p) {
                            F[F_CF + tid] = 0.f;
                            F[F_CP + tid] = bd * F[F_NRM + q * J + tid];
                        }
                    } else {
                        F[F_BPV + i] = bound;
                        wg_sync(1);
                        const int j = tid >> 1, hf = tid & 1;
                        float cpv = 0.f;
                        if (j > p) {
                            const float* row = sf + j * SROW;
#pragma unroll 4
                            for (int c = 0; c < 16; ++c) {
                                const int ii = piece(c, hf) * 4;
                                const float4 s4 = *reinterpret_cast<const float4*>(row + ii);
                                const float4 b4 = *reinterpret_cast<const float4*>(F + F_BPV + ii);
                                cpv = fmaf(b4.x, s4.x, fmaf(b4.y, s4.y, fmaf(b4.z, s4.z, fmaf(b4.w, s4.w, cpv))));
                            }
                        }
                        cpv += __shfl_xor_sync(0xffffffffu, cpv, 1);
                        if (hf == 0 && j > p) {
                            F[F_CF + j] = 0.f;
                            F[F_CP + j] = cpv;
                        }
                    }
                }
                wg_sync(1);  // F_G / F_CF / F_CP are read by other chain threads below
                // ---- rho (APF) -------------------------------------------------------------
                if (HAS_R) {
                    if (warp == 0) {
                        const int lane = tid & 31;
                        const int j0 = 2 * lane, j1 = j0 + 1;
                        const float r0 = j0 >= p ? rr[j0] : 1.f;
                        const float r1 = j1 >= p ? rr[j1] : 1.f;
                        const float pr = r0 * r1;
                        float incl = pr;
#pragma unroll
                        for (int o = 1; o < 32; o <<= 1) {
                            const float y = __shfl_up_sync(0xffffffffu, incl, o);
                            if (lane >= o) incl *= y;
                        }
                        const float excl = incl / pr;
                        F[F_RHO + j0] = j0 > p ? excl : 1.f;
                        F[F_RHO + j1] = j1 > p ? excl * r0 : 1.f;
                        if (lane == 31) F[F_RHO + J] = incl;
                    }
                    wg_sync(1);
                    if (!(F[F_RHO + J] > 1e-30f)) {  // retention products too small: clipped sweeps
                        clipped = true;
                        continue;
                    }
                }
                auto rho = [&](int j) -> float { return HAS_R ? F[F_RHO + j] : 1.f; };
                // ---- g_{p+1..63}: Jacobi sweeps on the unit-lower-triangular system --------
                int hb = 0;  // which half of F_H holds the final h
                {
                    float m[64];
                    // row jr of the system on lanes 0-15 of each chain warp (the lanes of an M = 64 product)
                    const int jr = (warp << 4) | (tid & 15);
                    const bool row_thread = (tid & 31) < 16;
                    // this row's coefficients, read once for all sweeps
                    float ga = 0.f, gb = 0.f, rj = 1.f, cfj = 0.f, cpj = 0.f, ir1 = 1.f;
                    if (row_thread) {
                        ga = gam[jr];
                        gb = bpv[jr];
                        rj = rho(jr);
                        cfj = F[F_CF + jr];
                        cpj = F[F_CP + jr];
                        if (HAS_R) ir1 = 1.f / rho(jr + 1);
                    }
                    if (nfree == KD) {
                        if (!gram_ready()) {
                            abort_now = true;
                            break;
                        }
                        if (!have_rows) {  // no Gram formed for this block
                            clipped = true;
                            continue;
                        }
                        if (row_thread) {
                            const float* mrow = reinterpret_cast<const float*>(sm + OFF_MT + q * MT_BYTES) + jr * MROW;
#pragma unroll
                            for (int l = 0; l < 64; l += 4) {
                                const float4 v = *reinterpret_cast<const float4*>(mrow + l);
                                m[l] = v.x;
                                m[l + 1] = v.y;
                                m[l + 2] = v.z;
                                m[l + 3] = v.w;
                            }
                        }
                    }
                    float gj = 0.f;
                    if (row_thread) {
                        const int j = jr;
                        if (j > p) {
                            gj = ga * (1.f - gb * (rj * cfj + cpj));
                            F[F_G + j] = gj;
                        } else if (j == p) {
                            gj = F[F_G + j];
                        }
                        const float hj = j >= p ? gj * ir1 : 0.f;
                        F[F_H + j] = hj;
                        F[F_H + J + j] = hj;
                    }
                    if (nfree == KD) {
                        // from the estimate above (within nu |g|; the rho ratios are <= 1)
                        const int K = sweeps_for_nu();
                        wg_sync(1);
                        for (int it = 0; K < 0 ? it < J : it < K; ++it) {
                            const float* hc = F + F_H + hb * J;  // h of the previous sweep
                            bool changed = false;
                            if (row_thread && jr > p) {
                                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                                for (int l = 0; l < 64; l += 4) {
                                    const float4 h4 = *reinterpret_cast<const float4*>(hc + l);
                                    acc[0] = fmaf(h4.x, m[l], acc[0]);
                                    acc[1] = fmaf(h4.y, m[l + 1], acc[1]);
                                    acc[2] = fmaf(h4.z, m[l + 2], acc[2]);
                                    acc[3] = fmaf(h4.w, m[l + 3], acc[3]);
                                }
                                const float accs = (acc[0] + acc[1]) + (acc[2] + acc[3]);
                                const float gn = ga * (1.f - gb * (rj * (cfj + accs) + cpj));
                                // stop once no g moves by more than a few ulps: each sweep shrinks
                                // the remaining error by the coupling |gamma b M| (~1e-3 here), so
                                // what is left is below rounding; a 1-ulp test can cycle on noise
                                changed = fabsf(gn - gj) > 5e-7f * fabsf(gn) + 1e-30f;
                                gj = gn;
                                F[F_G + jr] = gj;
                                F[F_H + (hb ^ 1) * J + jr] = gj * ir1;
                            }
                            hb ^= 1;
                            if (K >= 0) wg_sync(1);
                            else if (wg_count(1, changed) == 0) break;
                        }
                    }
                    tc::tc_fence_before();
                    wg_sync(1);
                }
                // ---- block end and verification ------------------------------------------
                const float* Hf = F + F_H + hb * J;
                if (tid == 0) FI[0] = J;
                float inc = 0.f;  // sum_{l=p}^{63} h_l s_li  (free coordinates)
                int viol = J;     // first token whose update leaves the assumed regime
                if (status == 0) {
                    float bnd = 0.f, inc1 = 0.f, bnd1 = 0.f;
#pragma unroll 4
                    for (int l = 0; l < J; l += 4) {  // h_l = 0 for l < p
                        const float4 h4 = *reinterpret_cast<const float4*>(Hf + l);
                        const float hs0 = h4.x * s_at(l, i);
                        const float hs1 = h4.y * s_at(l + 1, i);
                        const float hs2 = h4.z * s_at(l + 2, i);
                        const float hs3 = h4.w * s_at(l + 3, i);
                        inc += hs0;
                        bnd += fabsf(hs0);
                        inc1 += hs1;
                        bnd1 += fabsf(hs1);
                        inc += hs2;
                        bnd += fabsf(hs2);
                        inc1 += hs3;
                        bnd1 += fabsf(hs3);
                    }
                    inc += inc1;
                    bnd += bnd1;
                    bnd = bnd * 1.0001f + fabsf(d_lo);  // margin for the fp32 sums
                    // retention gates lie in (0, 1]: rho_j stays within [rho_64, 1]
                    const float rmin = HAS_R ? F[F_RHO + J] : 1.f;
                    const bool safe = (d_hi - bnd) >= 0.f && rmin * (d_hi - bnd) >= dmin && (d_hi + bnd) <= dmax;
                    if (!safe) {  // exact trajectory
                        float part = 0.f;
                        for (int j = p; j < J; ++j) {
                            part += Hf[j] * s_at(j, i);
                            const float v = rho(j + 1) * (d_hi + (part + d_lo));
                            if (v < dmin || v > dmax) { viol = j; break; }
                        }
                    }
                } else if (all_low) {
                    // every coordinate on d_min: for g_j > 0 the step r_j d_min + g_j s_j is
                    // largest at the largest s_j (fmaf is monotone in s), so that coordinate decides
                    // exactly; for g_j <= 0 the step is at most r_j d_min (a gate above 1 counts as
                    // leaving; the sweeps then take the rest of the block).  The same for every
                    // thread: each lane checks two tokens, then a warp minimum.
                    const int lane = tid & 31;
                    int v = J;
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int j = 2 * lane + e;
                        const float g = F[F_G + j], c = rr[j] * dmin;
                        const bool off = j > p && (g > 0.f ? fmaf(g, F[F_SMX + q * J + j], c) > dmin : c > dmin);
                        v = off ? min(v, j) : v;
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
                    viol = v;
                } else {
                    // the first token after p whose step would leave the face: all 64 at once, no
                    // early exit (g and r four at a time, so the loads pipeline)
#pragma unroll 4
                    for (int j4 = 0; j4 < J; j4 += 4) {
                        const float4 g4 = *reinterpret_cast<const float4*>(F + F_G + j4);
                        const float4 r4 = *reinterpret_cast<const float4*>(rr + j4);
                        const float gg[4] = {g4.x, g4.y, g4.z, g4.w}, rv[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = j4 + e;
                            const float xn = fmaf(gg[e], s_at(j, i), rv[e] * bound);
                            const bool off = j > p && (status == 1 ? (xn > dmin) : (xn < dmax));
                            viol = off ? min(viol, j) : viol;
                        }
                    }
                }
                wg_sync(1);
                if (viol < J) atomicMin(FI, viol);
                wg_sync(1);
                const int jstar = FI[0];
                if (jstar == J) {
                    if (tid < J && tid > p) gout[tid] = F[F_G + tid];
                    if (status == 0) pair_advance(d_hi, d_lo, inc, rho(J));
                    else { d_hi = bound; d_lo = 0.f; }
                    p = J;
                } else {
                    if (tid < J && tid > p && tid <= jstar) gout[tid] = F[F_G + tid];
                    if (status == 0) {
                        float part = 0.f;
                        for (int l = p; l <= jstar; ++l) part += Hf[l] * s_at(l, i);
                        pair_advance(d_hi, d_lo, part, rho(jstar + 1));
                        pair_clip(d_hi, d_lo, dmin, dmax);
                    } else {
                        const float xn = fmaf(F[F_G + jstar], s_at(jstar, i), rr[jstar] * bound);
                        d_hi = fminf(fmaxf(xn, dmin), dmax);
                        d_lo = 0.f;
                    }
                    p = jstar + 1;
                    clipped = true;  // the rest of the block by clipped sweeps
                }
                wg_sync(1);
            }
            if (abort_now) {
                atomicExch(&s_abort, 1);
                break;
            }
            if (tid == 0) *static_cast<volatile int*>(&s_gram_want) = s_gram_used;
            mbar_arrive(bars + B_CHAIN + 8 * q);
        }
        a.d_out[static_cast<size_t>(bh) * KD + i] = d_hi + d_lo;
    }
    if (tid >= 128) cp_async_wait<0>();
    scan_sync();
    if (tid == 0 && s_abort) {
        atomicExch(timeout_flag, 1u);
        // let the last Gram of each slot land before tensor memory is released (each earlier one
        // was waited for before its barrier was reused)
        for (int q = 0; q < 2; ++q)
            if (s_gcnt[q] > 0) tc::mbar_wait(bars + B_GRAM + 8 * q, (s_gcnt[q] - 1) & 1, kMaxPolls >> 4);
    }
    tc::tc_fence_before();
    scan_sync();
    tc::tc_fence_after();
    if (tid == 0) {
        for (int q = 0; q < 2; ++q) {
            tc::mbar_inval(bars + B_GRAM + 8 * q);
            tc::mbar_inval(bars + B_PREP + 8 * q);
            tc::mbar_inval(bars + B_CHAIN + 8 * q);
        }
        tc::mbar_inval(bars + B_MRDY);
        tc::mbar_inval(bars + B_MRDY + 8);
    }
    scan_sync();
}

}  // namespace scanblk
}  // namespace osdn
