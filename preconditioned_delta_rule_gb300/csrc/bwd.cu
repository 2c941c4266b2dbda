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
// u_t in shared memory) and walked backward, S_{t-1} rebuilt from S_t.  Row-owned gradients (dv,
// the carried G) stay in the CTA; dq, dk, dk~ and dbeta sum over the rows of all CTAs of a head by
// fp32 atomics into zeroed buffers.  Phase 1 runs one warp per (batch, head): d at every 64-token
// block start is stored by a forward pass, then each block is replayed (d_t in shared memory) and
// walked backward.  Both are fp32 throughout; the d recurrence is not compensated here (its
// forward rounding is ~1e-7 relative per token).
#include "common.cuh"

namespace osdn {
namespace {

constexpr int kChunk = 64;
constexpr int kRows = 32;         // rows of S per phase-2 CTA
constexpr int kRowsPerWarp = 4;   // 8 warps x 4 rows
constexpr int kThreads2 = 256;

// ---------------------------------------------------------------------------------------------
// Phase 2
// ---------------------------------------------------------------------------------------------
template <int K, typename TIn>
__global__ void __launch_bounds__(kThreads2) bwd_phase2_kernel(OsdnBwdArgs a, const float* __restrict__ kt,
                                                               float* __restrict__ ckpt, float* __restrict__ dkt) {
    constexpr int E = K / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int bh = blockIdx.x, b = bh / a.H, h = bh % a.H;
    const int T = a.T, H = a.H, V = a.V;
    const int slice = blockIdx.y;
    const int r0 = slice * kRows + warp * kRowsPerWarp;  // this warp's first row of S
    const int nch = (T + kChunk - 1) / kChunk;
    const TIn* qg = static_cast<const TIn*>(a.q);
    const TIn* kg = static_cast<const TIn*>(a.k);
    const TIn* vg = static_cast<const TIn*>(a.v);
    const size_t row0 = static_cast<size_t>(b) * T * H + h;
    // checkpoints of this CTA's slice: [nch][kRows][K]
    float* ck = ckpt + (static_cast<size_t>(bh) * gridDim.y + slice) * static_cast<size_t>(nch) * kRows * K;
    __shared__ float su[kChunk][kRows];  // u_t of the chunk being walked
    __shared__ float red[8][K + 1];      // per-warp partial column sums
    __shared__ float redb[8];

    float S[kRowsPerWarp][E];
#pragma unroll
    for (int j = 0; j < kRowsPerWarp; ++j)
#pragma unroll
        for (int i = 0; i < E; ++i) {
            const size_t off = (static_cast<size_t>(bh) * V + r0 + j) * K + lane * E + i;
            S[j][i] = a.S0 ? a.S0[off] : 0.f;
        }

    auto load_vec = [&](const TIn* base, size_t r, float (&x)[E]) { VecIO<TIn, E>::load(base + r * K + lane * E, x); };
    // one forward step on the slice; returns u_t of this warp's rows in u[]
    auto fwd_step = [&](int t, float (&u)[kRowsPerWarp]) {
        const size_t r = row0 + static_cast<size_t>(t) * H;
        float kv[E], ktv[E];
        load_vec(kg, r, kv);
        VecIO<float, E>::load(kt + r * K + lane * E, ktv);
        const float bt = a.beta[r];
#pragma unroll
        for (int j = 0; j < kRowsPerWarp; ++j) {
            float sk = 0.f;
#pragma unroll
            for (int i = 0; i < E; ++i) sk = fmaf(S[j][i], kv[i], sk);
            sk = warp_sum(sk);
            u[j] = to_f32(vg[r * V + r0 + j]) - sk;
            const float bu = bt * u[j];
#pragma unroll
            for (int i = 0; i < E; ++i) S[j][i] = fmaf(bu, ktv[i], S[j][i]);
        }
    };
    // forward pass: checkpoints at chunk starts
    for (int c = 0; c < nch; ++c) {
#pragma unroll
        for (int j = 0; j < kRowsPerWarp; ++j)
#pragma unroll
            for (int i = 0; i < E; ++i) ck[(static_cast<size_t>(c) * kRows + warp * kRowsPerWarp + j) * K + lane * E + i] = S[j][i];
        const int t1 = min(T, (c + 1) * kChunk);
        for (int t = c * kChunk; t < t1; ++t) {
            float u[kRowsPerWarp];
            fwd_step(t, u);
        }
    }
    // G = dL/dS_T
    float G[kRowsPerWarp][E];
#pragma unroll
    for (int j = 0; j < kRowsPerWarp; ++j)
#pragma unroll
        for (int i = 0; i < E; ++i) {
            const size_t off = (static_cast<size_t>(bh) * V + r0 + j) * K + lane * E + i;
            G[j][i] = a.dS ? a.dS[off] : 0.f;
        }
    // column sum of this CTA's rows of x[j][i] (weighted per row by w[j]) -> atomically added to out
    auto col_add = [&](const float (&x)[kRowsPerWarp][E], const float (&w)[kRowsPerWarp], float* out) {
        float p[E];
#pragma unroll
        for (int i = 0; i < E; ++i) {
            p[i] = 0.f;
#pragma unroll
            for (int j = 0; j < kRowsPerWarp; ++j) p[i] = fmaf(x[j][i], w[j], p[i]);
            red[warp][lane * E + i] = p[i];
        }
        __syncthreads();
        for (int col = threadIdx.x; col < K; col += kThreads2) {
            float s = 0.f;
#pragma unroll
            for (int w8 = 0; w8 < 8; ++w8) s += red[w8][col];
            atomicAdd(out + col, s);
        }
        __syncthreads();
    };

    for (int c = nch - 1; c >= 0; --c) {
        // recompute the chunk from its checkpoint, keeping u_t
#pragma unroll
        for (int j = 0; j < kRowsPerWarp; ++j)
#pragma unroll
            for (int i = 0; i < E; ++i) S[j][i] = ck[(static_cast<size_t>(c) * kRows + warp * kRowsPerWarp + j) * K + lane * E + i];
        const int t0 = c * kChunk, t1 = min(T, t0 + kChunk);
        for (int t = t0; t < t1; ++t) {
            float u[kRowsPerWarp];
            fwd_step(t, u);
            if (lane < kRowsPerWarp) {
                // lane j of the warp records row j (all lanes hold the same u values)
                float uj = u[0];
#pragma unroll
                for (int j = 1; j < kRowsPerWarp; ++j) uj = lane == j ? u[j] : uj;
                su[t - t0][warp * kRowsPerWarp + lane] = uj;
            }
        }
        __syncwarp();
        __syncthreads();
        for (int t = t1 - 1; t >= t0; --t) {
            const size_t r = row0 + static_cast<size_t>(t) * H;
            float qv[E], kv[E], ktv[E], dov[kRowsPerWarp], u[kRowsPerWarp];
            load_vec(qg, r, qv);
            load_vec(kg, r, kv);
            VecIO<float, E>::load(kt + r * K + lane * E, ktv);
            const float bt = a.beta[r];
#pragma unroll
            for (int j = 0; j < kRowsPerWarp; ++j) {
                dov[j] = a.dout[r * V + r0 + j] * a.scale;
                u[j] = su[t - t0][warp * kRowsPerWarp + j];
            }
            // dq_t = scale S_t^T do_t  (S is S_t here)
            col_add(S, dov, a.dq + r * K);
            // G += scale do_t q_t^T
#pragma unroll
            for (int j = 0; j < kRowsPerWarp; ++j)
#pragma unroll
                for (int i = 0; i < E; ++i) G[j][i] = fmaf(dov[j], qv[i], G[j][i]);
            // gk = G k~, du = beta gk, dbeta += <u, gk>, dv = du
            float du[kRowsPerWarp], ub = 0.f;
#pragma unroll
            for (int j = 0; j < kRowsPerWarp; ++j) {
                float gk = 0.f;
#pragma unroll
                for (int i = 0; i < E; ++i) gk = fmaf(G[j][i], ktv[i], gk);
                gk = warp_sum(gk);
                du[j] = bt * gk;
                ub = fmaf(u[j], gk, ub);
                if (lane == 0) a.dv[r * V + r0 + j] = du[j];
            }
            if (lane == 0) redb[warp] = ub;
            // dk~_t = beta G^T u
            float bu[kRowsPerWarp];
#pragma unroll
            for (int j = 0; j < kRowsPerWarp; ++j) bu[j] = bt * u[j];
            col_add(G, bu, dkt + r * K);  // (its barriers also publish redb)
            if (threadIdx.x == 0) {
                float sb = 0.f;
#pragma unroll
                for (int w8 = 0; w8 < 8; ++w8) sb += redb[w8];
                atomicAdd(a.dbeta + r, sb);
            }
            // S_{t-1} = S_t - beta u k~^T
#pragma unroll
            for (int j = 0; j < kRowsPerWarp; ++j)
#pragma unroll
                for (int i = 0; i < E; ++i) S[j][i] = fmaf(-bu[j], ktv[i], S[j][i]);
            // dk_t += -S_{t-1}^T du
            float ndu[kRowsPerWarp];
#pragma unroll
            for (int j = 0; j < kRowsPerWarp; ++j) ndu[j] = -du[j];
            col_add(S, ndu, a.dk + r * K);
            // G <- G - du k^T
#pragma unroll
            for (int j = 0; j < kRowsPerWarp; ++j)
#pragma unroll
                for (int i = 0; i < E; ++i) G[j][i] = fmaf(-du[j], kv[i], G[j][i]);
        }
        __syncthreads();
    }
    if (a.dS0) {
#pragma unroll
        for (int j = 0; j < kRowsPerWarp; ++j)
#pragma unroll
            for (int i = 0; i < E; ++i) a.dS0[(static_cast<size_t>(bh) * V + r0 + j) * K + lane * E + i] = G[j][i];
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
    // phase 1 forward: the write keys in fp32 (the library's scan)
    OsdnScanArgs sa{a.k, a.dtype, a.beta, a.r, a.d0, kt, OSDN_F32, ck1, a.B, a.T, a.H, K, a.eta, a.d_min, a.d_max,
                    a.eps, a.beta_aware, a.r ? a.r_per_key : 0};
    // d_out of this scan is scratch (ck1 is overwritten below by the phase-1 kernel's checkpoints)
    e = osdn_launch_scan(sa, nullptr, 0, s);
    if (e != cudaSuccess) return e;
    dim3 g2(static_cast<unsigned>(a.B * a.H), static_cast<unsigned>(a.V / kRows));
    bwd_phase2_kernel<K, TIn><<<g2, kThreads2, 0, s>>>(a, kt, ck2, dkt);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    dim3 g1(static_cast<unsigned>(a.B * a.H));
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
    return 4 * (2 * tok * K + heads * (V / osdn::kRows) * nch * osdn::kRows * K + heads * (nch + 1) * K);
}

cudaError_t osdn_launch_bwd(const OsdnBwdArgs& a, void* ws, cudaStream_t s) {
    if (a.V % osdn::kRows != 0) return cudaErrorInvalidValue;
    if (a.K == 128) return osdn::launch_k<128>(a, ws, s);
    if (a.K == 64) return osdn::launch_k<64>(a, ws, s);
    return cudaErrorInvalidValue;
}
