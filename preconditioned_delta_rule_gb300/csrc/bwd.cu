// bwd.cu -- the OSDN layer backward, token-recurrent in fp32 on the CUDA cores.
//
// "OSDN: Improving Delta Rule with Provable Online Preconditioning in Linear Attention".  The
// forward (Algorithm 1 / Eqs. (2), (4), (5), (7)): k~_t = d_t . k_t;
// d_{t+1} = clip(r_t d_t + g_t s_t), s_t = k_t . k_t, g_t = eta b (1 - b a_t) / max(|k_t|^2, eps),
// a_t = <d_t, s_t>, b = beta_t (or 1); u_t = v_t - S_{t-1} k_t; S_t = S_{t-1} + beta_t u_t k~_t^T;
// o_t = scale S_t q_t.  Given dL/do_t, dL/dS_T and dL/dd_T, the reverse sweeps are:
//
// Phase 2, t = T-1 .. 0, with G the gradient of S_t (dL/dS_T, then carried):
//   G += scale do_t q_t^T;  dq_t = scale S_t^T do_t;
//   gk = G k~_t;  du_t = beta_t gk;  dbeta_t += <u_t, gk>;  dv_t = du_t;  dk~_t = beta_t G^T u_t;
//   S_{t-1} = S_t - beta_t u_t k~_t^T;  dk_t += -S_{t-1}^T du_t;  G <- G - du_t k_t^T.
// Phase 1, t = T-1 .. 0, with e the gradient of d_{t+1} (dL/dd_T, then carried):
//   x = r d_t + g s;  e <- e . [d_min <= x <= d_max]  (the clip stops the gradient outside);
//   dd = r e + (dk~_t . k_t);  dr = <e, d_t> (or e . d_t per coordinate);  dg = <e, s>;
//   ds = g e;  with c = eta / max(n, eps), n = |k|^2:  da = -c b^2 dg,  db = c (1 - 2 b a) dg,
//   dn = -(g / max(n, eps)) dg where n > eps;  dd += da s;  ds += da d_t + dn;
//   dk_t += 2 k . ds + dk~_t . d_t;  dbeta_t += db (beta-aware);  e <- dd.
//
// Phase 2 runs one CTA per (batch, head, 32 rows of S): a forward pass stores S at the start of
// every 64-token chunk; then each chunk, last first, is recomputed from its checkpoint (keeping
// u_t in shared memory) and walked backward, S_{t-1} rebuilt from S_t.  Each chunk's inputs are
// staged in shared memory first.  Row-owned gradients (dv, the carried G) stay in the CTA; dq, dk,
// dk~ and dbeta sum over the rows of a CTA in shared memory (one barrier per token) and over the
// CTAs of a head by fp32 atomics into zeroed buffers.  Phase 1 runs one warp per (batch, head)
// and walks the 64-token blocks backward: for 16-bit keys with K = 128 from the forward scan's
// record (step sizes and block-start states, inputs staged a block ahead), otherwise from d
// checkpoints stored by its own forward pass.  Both are fp32 throughout; the d recurrence of the
// fallback is not compensated (its forward rounding is ~1e-7 relative per token).
#include "common.cuh"

namespace osdn {
namespace {

constexpr int kChunk = 64;
constexpr int kRows = 32;         // rows of S per phase-2 CTA
constexpr int kRowsPerWarp = 4;   // 8 warps x 4 rows
constexpr int kThreads2 = 256;

__device__ __forceinline__ void cp_async16(void* sdst, const void* gsrc) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(sdst))),
                 "l"(gsrc)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

// ---------------------------------------------------------------------------------------------
// Phase 2 with staged inputs: the same sweeps as bwd_phase2_kernel, but each 64-token chunk's
// q, k, k~, beta and this CTA's rows of v and dL/do are copied to shared memory (cp.async) before
// the chunk is processed, so no token waits on global memory, and the three column sums of a
// reverse step (dq_t, dk~_t, dk_t) are formed in one shared-memory pass with one barrier per token
// (their per-warp partials alternate between two buffers by token parity).
// ---------------------------------------------------------------------------------------------
template <int K, typename TIn>
struct P2Buf {
    TIn q[kChunk][K];
    TIn k[kChunk][K];
    float kt[kChunk][K];
    float dout[kChunk][kRows];
    TIn v[kChunk][kRows];
    float beta[kChunk];
    float su[kChunk][kRows];        // u_t of the chunk
    float red[2][3][8][K];          // per-warp partials of dq, dk~, dk
    float redb[2][8];
};

template <int K, typename TIn>
__global__ void __launch_bounds__(kThreads2, 2) bwd_phase2_st_kernel(OsdnBwdArgs a, const float* __restrict__ kt,
                                                                    float* __restrict__ ckpt, float* __restrict__ dkt) {
    constexpr int E = K / 32;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    P2Buf<K, TIn>& sb = *reinterpret_cast<P2Buf<K, TIn>*>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int bh = blockIdx.x, b = bh / a.H, h = bh % a.H;
    const int T = a.T, H = a.H, V = a.V;
    const int slice = blockIdx.y;
    const int rl = warp * kRowsPerWarp;           // this warp's first row within the slice
    const int r0 = slice * kRows + rl;            // ... of S
    const int nch = (T + kChunk - 1) / kChunk;
    const TIn* qg = static_cast<const TIn*>(a.q);
    const TIn* kg = static_cast<const TIn*>(a.k);
    const TIn* vg = static_cast<const TIn*>(a.v);
    const size_t row0 = static_cast<size_t>(b) * T * H + h;
    float* ck = ckpt + (static_cast<size_t>(bh) * gridDim.y + slice) * static_cast<size_t>(nch) * kRows * K;

    // chunk c's inputs -> shared memory (the backward sweep also needs q and dL/do)
    auto stage = [&](int c, bool bwd) {
        const int t0 = c * kChunk, jb = min(kChunk, T - t0);
        constexpr int KC = K * static_cast<int>(sizeof(TIn)) / 16;  // 16-byte pieces of a key row
        for (int e = tid; e < jb * KC; e += kThreads2) {
            const int j = e / KC, cc = e % KC;
            const size_t r = row0 + static_cast<size_t>(t0 + j) * H;
            cp_async16(reinterpret_cast<char*>(&sb.k[j][0]) + cc * 16, reinterpret_cast<const char*>(kg + r * K) + cc * 16);
            if (bwd) cp_async16(reinterpret_cast<char*>(&sb.q[j][0]) + cc * 16, reinterpret_cast<const char*>(qg + r * K) + cc * 16);
        }
        for (int e = tid; e < jb * (K / 4); e += kThreads2) {
            const int j = e / (K / 4), cc = e % (K / 4);
            cp_async16(&sb.kt[j][cc * 4], kt + (row0 + static_cast<size_t>(t0 + j) * H) * K + cc * 4);
        }
        if (bwd) {
            for (int e = tid; e < jb * (kRows / 4); e += kThreads2) {
                const int j = e / (kRows / 4), cc = e % (kRows / 4);
                cp_async16(&sb.dout[j][cc * 4], a.dout + (row0 + static_cast<size_t>(t0 + j) * H) * V + slice * kRows + cc * 4);
            }
        }
        cp_async_commit();
        for (int e = tid; e < jb * kRows; e += kThreads2) {
            const int j = e / kRows, cc = e % kRows;
            sb.v[j][cc] = vg[(row0 + static_cast<size_t>(t0 + j) * H) * V + slice * kRows + cc];
        }
        for (int j = tid; j < jb; j += kThreads2) sb.beta[j] = a.beta[row0 + static_cast<size_t>(t0 + j) * H];
        cp_async_wait<0>();
        __syncthreads();
    };
    float S[kRowsPerWarp][E];
    // one forward step on the slice from shared memory; u_t of the warp's rows into su (bwd) or dropped
    auto fwd_step = [&](int j) {
        float kv[E], ktv[E];
        VecIO<TIn, E>::load(&sb.k[j][lane * E], kv);
        VecIO<float, E>::load(&sb.kt[j][lane * E], ktv);
        const float bt = sb.beta[j];
        float sk[kRowsPerWarp];
#pragma unroll
        for (int jj = 0; jj < kRowsPerWarp; ++jj) {
            float x = 0.f;
#pragma unroll
            for (int i = 0; i < E; ++i) x = fmaf(S[jj][i], kv[i], x);
            sk[jj] = x;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int jj = 0; jj < kRowsPerWarp; ++jj) sk[jj] += __shfl_xor_sync(0xffffffffu, sk[jj], o);
#pragma unroll
        for (int jj = 0; jj < kRowsPerWarp; ++jj) {
            const float u = to_f32(sb.v[j][rl + jj]) - sk[jj];
            if (lane == jj) sb.su[j][rl + jj] = u;
            const float bu = bt * u;
#pragma unroll
            for (int i = 0; i < E; ++i) S[jj][i] = fmaf(bu, ktv[i], S[jj][i]);
        }
    };
#pragma unroll
    for (int jj = 0; jj < kRowsPerWarp; ++jj)
#pragma unroll
        for (int i = 0; i < E; ++i) {
            const size_t off = (static_cast<size_t>(bh) * V + r0 + jj) * K + lane * E + i;
            S[jj][i] = a.S0 ? a.S0[off] : 0.f;
        }
    // forward pass: checkpoints at chunk starts
    for (int c = 0; c < nch; ++c) {
#pragma unroll
        for (int jj = 0; jj < kRowsPerWarp; ++jj)
#pragma unroll
            for (int i = 0; i < E; ++i) ck[(static_cast<size_t>(c) * kRows + rl + jj) * K + lane * E + i] = S[jj][i];
        stage(c, false);
        const int jb = min(kChunk, T - c * kChunk);
        for (int j = 0; j < jb; ++j) fwd_step(j);
        __syncthreads();  // the next stage overwrites the tiles
    }
    float G[kRowsPerWarp][E];  // dL/dS of the warp's rows, carried backward
#pragma unroll
    for (int jj = 0; jj < kRowsPerWarp; ++jj)
#pragma unroll
        for (int i = 0; i < E; ++i) {
            const size_t off = (static_cast<size_t>(bh) * V + r0 + jj) * K + lane * E + i;
            G[jj][i] = a.dS ? a.dS[off] : 0.f;
        }
    int par = 0;
    for (int c = nch - 1; c >= 0; --c) {
        const int t0 = c * kChunk, jb = min(kChunk, T - t0);
#pragma unroll
        for (int jj = 0; jj < kRowsPerWarp; ++jj)
#pragma unroll
            for (int i = 0; i < E; ++i) S[jj][i] = ck[(static_cast<size_t>(c) * kRows + rl + jj) * K + lane * E + i];
        stage(c, true);
        for (int j = 0; j < jb; ++j) fwd_step(j);  // S back to the chunk's end, u_t recorded
        __syncthreads();
        for (int j = jb - 1; j >= 0; --j) {
            const size_t r = row0 + static_cast<size_t>(t0 + j) * H;
            float qv[E], kv[E], ktv[E], dov[kRowsPerWarp], u[kRowsPerWarp];
            VecIO<TIn, E>::load(&sb.q[j][lane * E], qv);
            VecIO<TIn, E>::load(&sb.k[j][lane * E], kv);
            VecIO<float, E>::load(&sb.kt[j][lane * E], ktv);
            const float bt = sb.beta[j];
#pragma unroll
            for (int jj = 0; jj < kRowsPerWarp; ++jj) {
                dov[jj] = sb.dout[j][rl + jj] * a.scale;
                u[jj] = sb.su[j][rl + jj];
            }
            float p1[E], p2[E], p3[E];
            // dq_t = scale S_t^T do_t
#pragma unroll
            for (int i = 0; i < E; ++i) {
                float x = 0.f;
#pragma unroll
                for (int jj = 0; jj < kRowsPerWarp; ++jj) x = fmaf(S[jj][i], dov[jj], x);
                p1[i] = x;
            }
            // G += scale do_t q_t^T;  gk = G k~
            float gk[kRowsPerWarp];
#pragma unroll
            for (int jj = 0; jj < kRowsPerWarp; ++jj) {
                float x = 0.f;
#pragma unroll
                for (int i = 0; i < E; ++i) {
                    G[jj][i] = fmaf(dov[jj], qv[i], G[jj][i]);
                    x = fmaf(G[jj][i], ktv[i], x);
                }
                gk[jj] = x;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                for (int jj = 0; jj < kRowsPerWarp; ++jj) gk[jj] += __shfl_xor_sync(0xffffffffu, gk[jj], o);
            // du = beta gk, dbeta += <u, gk>, dv = du;  dk~_t = beta G^T u
            float du[kRowsPerWarp], ub = 0.f;
#pragma unroll
            for (int jj = 0; jj < kRowsPerWarp; ++jj) {
                du[jj] = bt * gk[jj];
                ub = fmaf(u[jj], gk[jj], ub);
                if (lane == jj) a.dv[r * V + r0 + jj] = du[jj];
            }
#pragma unroll
            for (int i = 0; i < E; ++i) {
                float x = 0.f;
#pragma unroll
                for (int jj = 0; jj < kRowsPerWarp; ++jj) x = fmaf(G[jj][i], bt * u[jj], x);
                p2[i] = x;
            }
            // S_{t-1} = S_t - beta u k~^T;  dk_t += -S_{t-1}^T du;  G -= du k^T
#pragma unroll
            for (int jj = 0; jj < kRowsPerWarp; ++jj)
#pragma unroll
                for (int i = 0; i < E; ++i) S[jj][i] = fmaf(-bt * u[jj], ktv[i], S[jj][i]);
#pragma unroll
            for (int i = 0; i < E; ++i) {
                float x = 0.f;
#pragma unroll
                for (int jj = 0; jj < kRowsPerWarp; ++jj) x = fmaf(S[jj][i], -du[jj], x);
                p3[i] = x;
            }
#pragma unroll
            for (int jj = 0; jj < kRowsPerWarp; ++jj)
#pragma unroll
                for (int i = 0; i < E; ++i) G[jj][i] = fmaf(-du[jj], kv[i], G[jj][i]);
            // the three column sums over the CTA's rows, one barrier
#pragma unroll
            for (int i = 0; i < E; ++i) {
                sb.red[par][0][warp][lane * E + i] = p1[i];
                sb.red[par][1][warp][lane * E + i] = p2[i];
                sb.red[par][2][warp][lane * E + i] = p3[i];
            }
            if (lane == 0) sb.redb[par][warp] = ub;
            __syncthreads();
            for (int e = tid; e < 3 * K; e += kThreads2) {
                const int which = e / K, col = e % K;
                float x = 0.f;
#pragma unroll
                for (int w8 = 0; w8 < 8; ++w8) x += sb.red[par][which][w8][col];
                float* dst = which == 0 ? a.dq : (which == 1 ? dkt : a.dk);
                atomicAdd(dst + r * K + col, x);
            }
            if (tid == 0) {
                float x = 0.f;
#pragma unroll
                for (int w8 = 0; w8 < 8; ++w8) x += sb.redb[par][w8];
                atomicAdd(a.dbeta + r, x);
            }
            par ^= 1;
        }
        __syncthreads();  // the next stage overwrites the tiles
    }
    if (a.dS0) {
#pragma unroll
        for (int jj = 0; jj < kRowsPerWarp; ++jj)
#pragma unroll
            for (int i = 0; i < E; ++i) a.dS0[(static_cast<size_t>(bh) * V + r0 + jj) * K + lane * E + i] = G[jj][i];
    }
}

// ---------------------------------------------------------------------------------------------
// Phase 1: one warp per (batch, head)
// ---------------------------------------------------------------------------------------------
template <int K, typename TIn, int RMODE>
__global__ void __launch_bounds__(32) bwd_phase1_kernel(OsdnBwdArgs a, const float* __restrict__ dkt,
                                                        float* __restrict__ dck) {
    constexpr int E = K / 32;
    const int lane = threadIdx.x;
    const int bh = blockIdx.x, b = bh / a.H, h = bh % a.H;
    const int T = a.T, H = a.H;
    const int nch = (T + kChunk - 1) / kChunk;
    const TIn* kg = static_cast<const TIn*>(a.k);
    const size_t row0 = static_cast<size_t>(b) * T * H + h;
    float* ck = dck + static_cast<size_t>(bh) * nch * K;
    __shared__ float sd[kChunk][K];  // d_t of the block being walked

    float d[E];
#pragma unroll
    for (int i = 0; i < E; ++i) d[i] = a.d0 ? a.d0[static_cast<size_t>(bh) * K + lane * E + i] : 1.f;

    // a token's operands (key, gate inputs, and in the reverse sweep dL/dk~), loaded a token ahead
    struct In {
        float kv[E], bb, r[E], dkt[E];
    };
    auto load_in = [&](int t, In& f, bool with_dkt) {
        const size_t r = row0 + static_cast<size_t>(t) * H;
        VecIO<TIn, E>::load(kg + r * K + lane * E, f.kv);
        f.bb = a.beta_aware ? a.beta[r] : 1.f;
        if (RMODE == 2) {
            VecIO<float, E>::load(a.r + r * K + lane * E, f.r);
        } else {
#pragma unroll
            for (int i = 0; i < E; ++i) f.r[i] = RMODE == 1 ? a.r[r] : 1.f;
        }
        if (with_dkt) VecIO<float, E>::load(dkt + r * K + lane * E, f.dkt);
    };
    struct Step {
        float s[E], g, n, a_;
    };
    // the forward step's quantities at a token from d_t
    auto step_of = [&](const float (&dt)[E], const In& f, Step& st) {
        float n = 0.f, al = 0.f;
#pragma unroll
        for (int i = 0; i < E; ++i) {
            st.s[i] = f.kv[i] * f.kv[i];
            n += st.s[i];
            al = fmaf(dt[i], st.s[i], al);
        }
        n = warp_sum(n);
        al = warp_sum(al);
        st.n = n;
        st.a_ = al;
        st.g = a.eta * f.bb * (1.f - f.bb * al) / fmaxf(n, a.eps);
    };
    {
        In nx;
        if (T > 0) load_in(0, nx, false);
        for (int c = 0; c < nch; ++c) {
#pragma unroll
            for (int i = 0; i < E; ++i) ck[static_cast<size_t>(c) * K + lane * E + i] = d[i];
            const int t1 = min(T, (c + 1) * kChunk);
            for (int t = c * kChunk; t < t1; ++t) {
                const In cur = nx;
                if (t + 1 < T) load_in(t + 1, nx, false);
                Step st;
                step_of(d, cur, st);
#pragma unroll
                for (int i = 0; i < E; ++i) d[i] = fminf(fmaxf(fmaf(st.g, st.s[i], cur.r[i] * d[i]), a.d_min), a.d_max);
            }
        }
    }
    float e[E];  // dL/dd_{t+1}
#pragma unroll
    for (int i = 0; i < E; ++i) e[i] = a.dd ? a.dd[static_cast<size_t>(bh) * K + lane * E + i] : 0.f;
    for (int c = nch - 1; c >= 0; --c) {
        const int t0 = c * kChunk, t1 = min(T, t0 + kChunk);
#pragma unroll
        for (int i = 0; i < E; ++i) d[i] = ck[static_cast<size_t>(c) * K + lane * E + i];
        {
            In nx;
            load_in(t0, nx, false);
            for (int t = t0; t < t1; ++t) {
#pragma unroll
                for (int i = 0; i < E; ++i) sd[t - t0][lane * E + i] = d[i];
                const In cur = nx;
                if (t + 1 < t1) load_in(t + 1, nx, false);
                Step st;
                step_of(d, cur, st);
#pragma unroll
                for (int i = 0; i < E; ++i) d[i] = fminf(fmaxf(fmaf(st.g, st.s[i], cur.r[i] * d[i]), a.d_min), a.d_max);
            }
        }
        __syncwarp();
        In bnx;
        load_in(t1 - 1, bnx, true);
        for (int t = t1 - 1; t >= t0; --t) {
            const size_t r = row0 + static_cast<size_t>(t) * H;
            const In cur = bnx;
            if (t - 1 >= t0) load_in(t - 1, bnx, true);
            float dt[E];
#pragma unroll
            for (int i = 0; i < E; ++i) dt[i] = sd[t - t0][lane * E + i];
            const float(&kv)[E] = cur.kv;
            const float(&dktv)[E] = cur.dkt;
            Step st;
            step_of(dt, cur, st);
            float dd[E], ds[E], dg = 0.f, dr = 0.f;
#pragma unroll
            for (int i = 0; i < E; ++i) {
                const float x = fmaf(st.g, st.s[i], cur.r[i] * dt[i]);
                const float ex = (x >= a.d_min && x <= a.d_max) ? e[i] : 0.f;
                dd[i] = cur.r[i] * ex + dktv[i] * kv[i];
                dg = fmaf(ex, st.s[i], dg);
                ds[i] = st.g * ex;
                if (RMODE == 2) a.dr[r * K + lane * E + i] = ex * dt[i];
                else dr = fmaf(ex, dt[i], dr);
            }
            dg = warp_sum(dg);
            if (RMODE == 1) {
                dr = warp_sum(dr);
                if (lane == 0) a.dr[r] = dr;
            }
            const float nb = fmaxf(st.n, a.eps), cc = a.eta / nb;
            const float da = -cc * cur.bb * cur.bb * dg;
            const float db = cc * (1.f - 2.f * cur.bb * st.a_) * dg;
            const float dn = st.n > a.eps ? -(st.g / nb) * dg : 0.f;
            float dkl[E];
#pragma unroll
            for (int i = 0; i < E; ++i) {
                dd[i] = fmaf(da, st.s[i], dd[i]);
                ds[i] = ds[i] + da * dt[i] + dn;
                dkl[i] = 2.f * kv[i] * ds[i] + dktv[i] * dt[i];
                e[i] = dd[i];
            }
            // added without reading back (no stall on the load; nothing else writes these words now)
            float* dkp = a.dk + r * K + lane * E;
#pragma unroll
            for (int i = 0; i < E; ++i) atomicAdd(dkp + i, dkl[i]);
            if (a.beta_aware && lane == 0) atomicAdd(a.dbeta + r, db);
        }
        __syncwarp();
    }
    if (a.dd0) {
#pragma unroll
        for (int i = 0; i < E; ++i) a.dd0[static_cast<size_t>(bh) * K + lane * E + i] = e[i];
    }
}

// ---------------------------------------------------------------------------------------------
// Phase 1 from the forward scan's own record (16-bit keys, K = 128, one retention per head or
// none).  The blocked scan stores every token's step size g_t and every 64-token block's start
// state (an fp32 hi + lo pair); replaying d_{t+1} = clip(r_t d_t + g_t k_t^2) from them gives the
// forward's d_t exactly (the emission's arithmetic), with no reduction.  One warp per (batch,
// head) walks the blocks last first; each block's keys, dL/dk~, step sizes, gates and beta are
// copied to shared memory asynchronously one block ahead, so the per-token work reads shared
// memory only: the reverse step needs two sums over the key coordinates (a_t = <d_t, s_t> and
// <e, s_t>; with a retention gate also <e, d_t>), formed in one interleaved butterfly.
// ---------------------------------------------------------------------------------------------
template <typename TIn, bool HAS_R>
__global__ void __launch_bounds__(32) bwd_phase1_blk_kernel(OsdnBwdArgs a, const float* __restrict__ dkt,
                                                            const float* __restrict__ ws_g, const float* __restrict__ ws_d) {
    constexpr int K = 128, E = 4, J = kChunk;
    struct Buf {
        TIn k[J][K];
        float dkt[J][K];
        float g[J], r[J], bb[J];
    };
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Buf* buf = reinterpret_cast<Buf*>(smem_raw);  // [2]
    float(*sd)[K] = reinterpret_cast<float(*)[K]>(smem_raw + 2 * sizeof(Buf));  // d_t of the block
    float* sn = reinterpret_cast<float*>(smem_raw + 2 * sizeof(Buf) + J * K * 4);  // |k_t|^2
    const int lane = threadIdx.x;
    const int bh = blockIdx.x, b = bh / a.H, h = bh % a.H;
    const int T = a.T, H = a.H;
    const int nblk = (T + J - 1) / J;
    const TIn* kg = static_cast<const TIn*>(a.k);
    const size_t row0 = static_cast<size_t>(b) * T * H + h;

    // block m's inputs -> buf[m & 1] (cp.async; tokens past T are not fetched)
    auto stage = [&](int m) {
        Buf& B = buf[m & 1];
        const int t0 = m * J, jb = min(J, T - t0);
        for (int e = lane; e < jb * (K * 2 / 16); e += 32) {  // keys: 16 chunks of 16 B per token
            const int j = e >> 4, c = e & 15;
            cp_async16(&B.k[j][c * 8], kg + (row0 + static_cast<size_t>(t0 + j) * H) * K + c * 8);
        }
        for (int e = lane; e < jb * (K * 4 / 16); e += 32) {  // dL/dk~: 32 chunks per token
            const int j = e >> 5, c = e & 31;
            cp_async16(&B.dkt[j][c * 4], dkt + (row0 + static_cast<size_t>(t0 + j) * H) * K + c * 4);
        }
        cp_async_commit();
        for (int j = lane; j < J; j += 32) {
            const bool valid = j < jb;
            const size_t r = row0 + static_cast<size_t>(t0 + j) * H;
            B.g[j] = valid ? ws_g[static_cast<size_t>(bh) * T + t0 + j] : 0.f;
            B.r[j] = (HAS_R && valid) ? a.r[r] : 1.f;
            B.bb[j] = valid ? (a.beta_aware ? a.beta[r] : 1.f) : 0.f;
        }
    };

    float e[E];  // dL/dd_{t+1}
#pragma unroll
    for (int i = 0; i < E; ++i) e[i] = a.dd ? a.dd[static_cast<size_t>(bh) * K + lane * E + i] : 0.f;
    stage(nblk - 1);
    for (int m = nblk - 1; m >= 0; --m) {
        const Buf& B = buf[m & 1];
        const int t0 = m * J, jb = min(J, T - t0);
        if (m > 0) {
            stage(m - 1);  // the next block to walk, while this one is replayed and walked
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncwarp();
        // |k_t|^2, two tokens per lane (needs no d)
        for (int j = lane; j < jb; j += 32) {
            float n = 0.f;
#pragma unroll 8
            for (int i = 0; i < K; ++i) {
                const float kk = to_f32(B.k[j][i]);
                n = fmaf(kk, kk, n);
            }
            sn[j] = n;
        }
        // replay the block from its start state (the forward's emission arithmetic)
        const float* wd = ws_d + (static_cast<size_t>(bh) * nblk + m) * (2 * K);
        float d[E];
#pragma unroll
        for (int i = 0; i < E; ++i) d[i] = wd[lane * E + i] + wd[K + lane * E + i];
        for (int j = 0; j < jb; ++j) {
            float kv[E];
            VecIO<TIn, E>::load(&B.k[j][lane * E], kv);
            *reinterpret_cast<float4*>(&sd[j][lane * E]) = make_float4(d[0], d[1], d[2], d[3]);
#pragma unroll
            for (int i = 0; i < E; ++i) d[i] = replay_step(d[i], B.r[j], replay_inc(B.g[j], kv[i]), a.d_min, a.d_max);
        }
        __syncwarp();
        for (int j = jb - 1; j >= 0; --j) {
            const size_t r = row0 + static_cast<size_t>(t0 + j) * H;
            float kv[E], dt[E], dk[E];
            VecIO<TIn, E>::load(&B.k[j][lane * E], kv);
            VecIO<float, E>::load(&sd[j][lane * E], dt);
            VecIO<float, E>::load(&B.dkt[j][lane * E], dk);
            const float g = B.g[j], rr = B.r[j], bb = B.bb[j], n = sn[j];
            float s4[E], ex[E], al = 0.f, dg = 0.f, dr = 0.f;
#pragma unroll
            for (int i = 0; i < E; ++i) {
                s4[i] = kv[i] * kv[i];
                const float x = fmaf(rr, dt[i], replay_inc(g, kv[i]));
                ex[i] = (x >= a.d_min && x <= a.d_max) ? e[i] : 0.f;
                al = fmaf(dt[i], s4[i], al);
                dg = fmaf(ex[i], s4[i], dg);
                if (HAS_R) dr = fmaf(ex[i], dt[i], dr);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                al += __shfl_xor_sync(0xffffffffu, al, o);
                dg += __shfl_xor_sync(0xffffffffu, dg, o);
                if (HAS_R) dr += __shfl_xor_sync(0xffffffffu, dr, o);
            }
            if (HAS_R && lane == 0) a.dr[r] = dr;
            const float nb = fmaxf(n, a.eps), cc = a.eta / nb;
            const float da = -cc * bb * bb * dg;
            const float db = cc * (1.f - 2.f * bb * al) * dg;
            const float dn = n > a.eps ? -(g / nb) * dg : 0.f;
            float* dkp = a.dk + r * K + lane * E;
#pragma unroll
            for (int i = 0; i < E; ++i) {
                const float dd = fmaf(da, s4[i], fmaf(rr, ex[i], dk[i] * kv[i]));
                const float ds = g * ex[i] + da * dt[i] + dn;
                atomicAdd(dkp + i, 2.f * kv[i] * ds + dk[i] * dt[i]);
                e[i] = dd;
            }
            if (a.beta_aware && lane == 0) atomicAdd(a.dbeta + r, db);
        }
        __syncwarp();
    }
    if (a.dd0) {
#pragma unroll
        for (int i = 0; i < E; ++i) a.dd0[static_cast<size_t>(bh) * K + lane * E + i] = e[i];
    }
}

template <typename TIn>
constexpr size_t phase1_blk_smem() {
    return 2 * (sizeof(TIn) * kChunk * 128 + 4 * kChunk * 128 + 3 * 4 * kChunk) + 4 * kChunk * 128 + 4 * kChunk;
}

template <int K, typename TIn>
cudaError_t launch_bwd(const OsdnBwdArgs& a, void* ws, cudaStream_t s) {
    const int nch = (a.T + kChunk - 1) / kChunk;
    const size_t tok = static_cast<size_t>(a.B) * a.T * a.H;
    unsigned char* w = static_cast<unsigned char*>(ws);
    float* kt = reinterpret_cast<float*>(w);                              // [B,T,H,K] k~ (fp32)
    float* dkt = kt + tok * K;                                            // [B,T,H,K] dL/dk~
    float* ck2 = dkt + tok * K;                                           // S checkpoints
    float* ck1 = ck2 + static_cast<size_t>(a.B) * a.H * (a.V / kRows) * nch * kRows * K;  // d checkpoints
    // zero what the atomics accumulate into
    cudaError_t e = cudaMemsetAsync(dkt, 0, tok * K * sizeof(float), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(a.dq, 0, tok * K * sizeof(float), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(a.dk, 0, tok * K * sizeof(float), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(a.dbeta, 0, tok * sizeof(float), s);
    if (e != cudaSuccess) return e;
    // phase 1 forward: the write keys in fp32 (the library's scan); where the blocked scan applies,
    // its record of step sizes and block-start states drives the phase-1 reverse sweep
    OsdnScanArgs sa{a.k, a.dtype, a.beta, a.r, a.d0, kt, OSDN_F32, ck1, a.B, a.T, a.H, K, a.eta, a.d_min, a.d_max,
                    a.eps, a.beta_aware, a.r ? a.r_per_key : 0};
    // (the record drives bwd_phase1_blk_kernel, which takes one retention gate per head)
    const size_t scan_ws = (K == 128 && sizeof(TIn) == 2 && !sa.r_per_key) ? osdn_scan_block_workspace_bytes(sa) : 0;
    float* sws = ck1 + static_cast<size_t>(a.B) * a.H * (nch + 1) * K;
    // d_out of this scan is scratch (ck1 is overwritten below by the phase-1 kernel's checkpoints)
    e = osdn_launch_scan(sa, scan_ws ? sws : nullptr, scan_ws, s);
    if (e != cudaSuccess) return e;
    dim3 g2(static_cast<unsigned>(a.B * a.H), static_cast<unsigned>(a.V / kRows));
    {
        constexpr size_t smem2 = sizeof(P2Buf<K, TIn>);
        e = cudaFuncSetAttribute(bwd_phase2_st_kernel<K, TIn>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem2));
        if (e != cudaSuccess) return e;
        bwd_phase2_st_kernel<K, TIn><<<g2, kThreads2, smem2, s>>>(a, kt, ck2, dkt);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    dim3 g1(static_cast<unsigned>(a.B * a.H));
    if constexpr (K == 128 && sizeof(TIn) == 2) {
        if (scan_ws) {
            const float* ws_g = sws;
            const float* ws_d = ws_g + static_cast<size_t>(a.B) * a.H * a.T;
            constexpr size_t smem = phase1_blk_smem<TIn>();
            auto kern = a.r ? bwd_phase1_blk_kernel<TIn, true> : bwd_phase1_blk_kernel<TIn, false>;
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
            if (e != cudaSuccess) return e;
            kern<<<g1, 32, smem, s>>>(a, dkt, ws_g, ws_d);
            return cudaGetLastError();
        }
    }
    if (a.r && a.r_per_key) bwd_phase1_kernel<K, TIn, 2><<<g1, 32, 0, s>>>(a, dkt, ck1);
    else if (a.r) bwd_phase1_kernel<K, TIn, 1><<<g1, 32, 0, s>>>(a, dkt, ck1);
    else bwd_phase1_kernel<K, TIn, 0><<<g1, 32, 0, s>>>(a, dkt, ck1);
    return cudaGetLastError();
}

template <int K>
cudaError_t launch_k(const OsdnBwdArgs& a, void* ws, cudaStream_t s) {
    switch (a.dtype) {
        case OSDN_F32: return launch_bwd<K, float>(a, ws, s);
        case OSDN_BF16: return launch_bwd<K, __nv_bfloat16>(a, ws, s);
        case OSDN_F16: return launch_bwd<K, __half>(a, ws, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace
}  // namespace osdn

size_t osdn_bwd_workspace_bytes(int B, int T, int H, int K, int V) {
    if (B <= 0 || T <= 0 || H <= 0) return 0;
    const size_t nch = (static_cast<size_t>(T) + osdn::kChunk - 1) / osdn::kChunk;
    const size_t tok = static_cast<size_t>(B) * T * H;
    const size_t heads = static_cast<size_t>(B) * H;
    // k~ and dL/dk~ (fp32), S checkpoints, d checkpoints, then the blocked scan's record (K = 128)
    const size_t scan_rec = K == 128 ? heads * (static_cast<size_t>(T) + nch * 2 * K) : 0;
    return 4 * (2 * tok * K + heads * (V / osdn::kRows) * nch * osdn::kRows * K + heads * (nch + 1) * K + scan_rec);
}

cudaError_t osdn_launch_bwd(const OsdnBwdArgs& a, void* ws, cudaStream_t s) {
    if (a.V % osdn::kRows != 0) return cudaErrorInvalidValue;
    if (a.K == 128) return osdn::launch_k<128>(a, ws, s);
    if (a.K == 64) return osdn::launch_k<64>(a, ws, s);
    return cudaErrorInvalidValue;
}
