// scan_block.cu -- phase 1 of OSDN (the online preconditioner sweep) in 64-token blocks.
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
// the first violation the tokens before it are accepted, the state after it is formed with the
// clip, and the block restarts there with the new classification (after 8 restarts in a block
// the rest of the block runs token by token).  The result is the sequential algorithm's, up to
// reassociation.  d is carried across blocks as an unevaluated fp32 pair (hi + lo).
// With one gate per key coordinate (diag(r_t), Appendix A.5) the free trajectories no longer share
// one product of gates, so every block is solved by Jacobi sweeps on the clipped recurrence itself:
// each coordinate runs its own trajectory d_{j+1} = clip(r_{j,i} d_j + g_j s_j) under a guess of
// the g's, and the products d_j s_j summed over the coordinates give the next guess.  The gates
// are staged with the keys, in the space the Gram path uses for its fp16 s copies and Gram rows.
//
// Mapping: one CTA of 256 threads per (batch, head).  Warpgroup 0 ("chain") runs the serial part
// above, one key coordinate per thread.  Warpgroup 1 prepares block b+1 (cp.async staging of the
// keys three blocks ahead, s = k.k in fp32, power-of-two-scaled fp16 hi/lo copies and the Gram on
// the tensor cores) and emits the write keys of block b by replaying the clipped recurrence with
// the chain's g values.  The warpgroups hand blocks over through mbarriers.
#include <type_traits>

#include "common.cuh"
#include "scan_block_body.cuh"
#include "tc_ptx.cuh"

namespace osdn {
namespace {
using namespace scanblk;

// Set when a bounded wait of the scan kernel gave up (read and cleared by osdn_check).
__device__ unsigned int g_scan_timeout_flag = 0;

template <typename TIn, typename TOut, int RM>
__global__ void __launch_bounds__(NT, 1) scan_block_kernel(OsdnScanArgs a, float* ws_g, float* ws_d) {
    extern __shared__ unsigned char smem_raw[];
    __shared__ uint32_t s_tmem;
    if (threadIdx.x < 32) tc::tmem_alloc(tc::smem_u32(&s_tmem), TMEM_COLS);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tbase = s_tmem;
    scan_block_body<TIn, TOut, RM>(a, ws_g, ws_d, blockIdx.x, smem_raw, tbase, &g_scan_timeout_flag);
    if (threadIdx.x < 32) tc::tmem_dealloc(tbase, TMEM_COLS);
}

// Write keys of one 64-token block of one head, EC key coordinates per CTA: thread i replays
// coordinate c0 + i of the clipped recurrence d <- clip(r_t d + g_t k_t^2) from the block's start
// state with the step sizes g_t the scan fixed, emitting k~_t = d_t k_t.  Fully parallel over
// (head, block, coordinate slice); small CTAs keep many blocks in flight so that loads, the
// dependent 64-step loop and stores of different blocks overlap.  The key slice (64 rows of
// 2 EC bytes) moves through shared memory in 16-byte pieces; 16-bit write keys overwrite their key
// in the tile and leave the same way, fp32 write keys go straight out.  RM as in scan_block_body:
// with one gate per coordinate (RM = 2) each thread reads its coordinate's gates, 32 tokens ahead.
constexpr int EC = 32;
template <typename TIn, typename TOut, int RM>
__global__ void __launch_bounds__(EC) scan_emit_kernel(OsdnScanArgs a, const float* __restrict__ ws_g,
                                                       const float* __restrict__ ws_d) {
    static_assert(sizeof(TIn) == 2, "16-bit keys");
    constexpr int ROW_U4 = EC * 2 / 16;   // 16-byte pieces per key row slice
    __shared__ __align__(16) TIn tile[J * EC];
    __shared__ float sg[J], sr[J];
    const int m = blockIdx.x, bh = blockIdx.y, c0 = blockIdx.z * EC, i = threadIdx.x;
    const int b = bh / a.H, h = bh % a.H, T = a.T, H = a.H;
    const int nblk = gridDim.x, t0 = m * J, jb = min(J, T - t0);
    const size_t row0 = static_cast<size_t>(b) * T * H + h;
    const size_t stride = static_cast<size_t>(H) * KD;      // elements between consecutive tokens
    const TIn* kg = static_cast<const TIn*>(a.k) + (row0 + static_cast<size_t>(t0) * H) * KD + c0;
    TOut* og = static_cast<TOut*>(a.k_tilde) + (row0 + static_cast<size_t>(t0) * H) * KD + c0;
    uint4* t4 = reinterpret_cast<uint4*>(tile);
#pragma unroll
    for (int e = i; e < J * ROW_U4; e += EC) {
        const int j = e / ROW_U4, c = e % ROW_U4;
        if (j < jb) t4[e] = *reinterpret_cast<const uint4*>(kg + j * stride + c * 8);
    }
#pragma unroll
    for (int jj = i; jj < J; jj += EC) {
        const bool valid = jj < jb;
        sg[jj] = valid ? ws_g[static_cast<size_t>(bh) * T + t0 + jj] : 0.f;
        sr[jj] = (RM == 1 && valid) ? a.r[row0 + static_cast<size_t>(t0 + jj) * H] : 1.f;
    }
    const float* wd = ws_d + (static_cast<size_t>(bh) * nblk + m) * (2 * KD) + c0;
    float d = wd[i] + wd[KD + i];
    __syncthreads();
    const float dmin = a.d_min, dmax = a.d_max;
    // 32 tokens at a time: keys and increments first, then the serial steps, then the stores
#pragma unroll
    for (int j0 = 0; j0 < J; j0 += 32) {
        float kv[32], inc[32], kt[32], rv[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const bool valid = j0 + j < jb;
            kv[j] = valid ? to_f32(tile[(j0 + j) * EC + i]) : 0.f;
            inc[j] = replay_inc(sg[j0 + j], kv[j]);
            if constexpr (RM == 2) rv[j] = valid ? a.r[(row0 + static_cast<size_t>(t0 + j0 + j) * H) * KD + c0 + i] : 1.f;
            else rv[j] = sr[j0 + j];
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            kt[j] = d * kv[j];
            d = replay_step(d, rv[j], inc[j], dmin, dmax);
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            if (j0 + j < jb) {
                if constexpr (sizeof(TOut) == 2) reinterpret_cast<TOut*>(tile)[(j0 + j) * EC + i] = from_f32<TOut>(kt[j]);  // own slot
                else og[(j0 + j) * stride + i] = kt[j];
            }
        }
    }
    if constexpr (sizeof(TOut) == 2) {
        __syncthreads();
#pragma unroll
        for (int e = i; e < J * ROW_U4; e += EC) {
            const int j = e / ROW_U4, c = e % ROW_U4;
            if (j < jb) *reinterpret_cast<uint4*>(og + j * stride + c * 8) = t4[e];
        }
    }
}

template <typename TIn, typename TOut>
cudaError_t launch_b(const OsdnScanArgs& a, void* ws, size_t ws_bytes, cudaStream_t s) {
    static cudaError_t attr = [] {
        cudaError_t e[3] = {
            cudaFuncSetAttribute(scan_block_kernel<TIn, TOut, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC),
            cudaFuncSetAttribute(scan_block_kernel<TIn, TOut, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC),
            cudaFuncSetAttribute(scan_block_kernel<TIn, TOut, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC)};
        for (cudaError_t x : e)
            if (x != cudaSuccess) return x;
        return cudaSuccess;
    }();
    if (attr != cudaSuccess) return attr;
    dim3 grid(static_cast<unsigned>(a.B * a.H)), block(NT);
    const int nblk = (a.T + J - 1) / J;
    const size_t need = static_cast<size_t>(a.B) * a.H * (static_cast<size_t>(a.T) + static_cast<size_t>(nblk) * 2 * KD) * 4;
    float* ws_g = nullptr;
    float* ws_d = nullptr;
    if (ws != nullptr && ws_bytes >= need) {
        ws_g = static_cast<float*>(ws);
        ws_d = ws_g + static_cast<size_t>(a.B) * a.H * a.T;
    }
    const int rm = a.r ? (a.r_per_key ? 2 : 1) : 0;
    if (rm == 2) scan_block_kernel<TIn, TOut, 2><<<grid, block, SMEM_ALLOC, s>>>(a, ws_g, ws_d);
    else if (rm == 1) scan_block_kernel<TIn, TOut, 1><<<grid, block, SMEM_ALLOC, s>>>(a, ws_g, ws_d);
    else scan_block_kernel<TIn, TOut, 0><<<grid, block, SMEM_ALLOC, s>>>(a, ws_g, ws_d);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || ws_g == nullptr) return e;
    dim3 ge(static_cast<unsigned>(nblk), static_cast<unsigned>(a.B * a.H), KD / EC), be(EC);
    if (rm == 2) scan_emit_kernel<TIn, TOut, 2><<<ge, be, 0, s>>>(a, ws_g, ws_d);
    else if (rm == 1) scan_emit_kernel<TIn, TOut, 1><<<ge, be, 0, s>>>(a, ws_g, ws_d);
    else scan_emit_kernel<TIn, TOut, 0><<<ge, be, 0, s>>>(a, ws_g, ws_d);
    return cudaGetLastError();
}

template <typename TIn>
cudaError_t launch_bo(const OsdnScanArgs& a, void* ws, size_t ws_bytes, cudaStream_t s) {
    switch (a.kt_dtype) {
        case OSDN_F32: return launch_b<TIn, float>(a, ws, ws_bytes, s);
        case OSDN_BF16: return launch_b<TIn, __nv_bfloat16>(a, ws, ws_bytes, s);
        case OSDN_F16: return launch_b<TIn, __half>(a, ws, ws_bytes, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace
}  // namespace osdn

cudaError_t osdn_scan_block_read_and_clear_timeout(unsigned int* flag) {
    cudaError_t e = cudaMemcpyFromSymbol(flag, osdn::g_scan_timeout_flag, sizeof(unsigned int));
    if (e == cudaSuccess && *flag) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(osdn::g_scan_timeout_flag, &zero, sizeof(unsigned int));
    }
    return e;
}

bool osdn_scan_block_covers(const OsdnScanArgs& a) {
    return a.K == osdn::KD && a.T > 0 && (a.k_dtype == OSDN_BF16 || a.k_dtype == OSDN_F16);
}

size_t osdn_scan_block_workspace_bytes(const OsdnScanArgs& a) {
    if (!osdn_scan_block_covers(a)) return 0;
    const size_t nblk = (static_cast<size_t>(a.T) + osdn::J - 1) / osdn::J;
    return static_cast<size_t>(a.B) * a.H * (static_cast<size_t>(a.T) + nblk * 2 * osdn::KD) * 4;
}

// Blocked scan for 16-bit keys with K = 128 (cudaErrorNotSupported otherwise).  With a workspace
// of osdn_scan_block_workspace_bytes(a) bytes the write keys come from scan_emit_kernel.
cudaError_t osdn_launch_scan_block(const OsdnScanArgs& a, void* ws, size_t ws_bytes, cudaStream_t s) {
    if (!osdn_scan_block_covers(a)) return cudaErrorNotSupported;
    if (a.k_dtype == OSDN_BF16) return osdn::launch_bo<__nv_bfloat16>(a, ws, ws_bytes, s);
    return osdn::launch_bo<__half>(a, ws, ws_bytes, s);
}
