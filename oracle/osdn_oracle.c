/*
 * osdn_oracle.c -- plain, slow, fp64 CPU reference of the OSDN forward path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call this file; only the test
 * suite, the package smoke check and the benchmark's CPU-baseline leg do.  It shares no code,
 * header, table or constant with the CUDA library.
 *
 * Source: "OSDN: Improving Delta Rule with Provable Online Preconditioning in Linear Attention"
 * (arXiv:2605.13473).
 *   - write-side substitution, Section 4.1 Eq. (2):      S_t = S_{t-1} + beta_t u_t (d_t . k_t)^T,
 *                                                        u_t = v_t - S_{t-1} k_t  (original key reads)
 *   - asymmetric transition, Section 4.3 Eq. (5)
 *   - phase-1 sweep, Section 4.2 Algorithm 1 / Eq. (4): emit k~_t = d_t . k_t, THEN
 *       d_{t+1} = clip(d_t + eta b (1 - b <d_t, k_t^2>) / max(|k_t|^2, eps) * k_t^2)
 *     with b = beta_t ("beta-aware", Listing 1 default) or b = 1 (the non-beta-aware 1.3B form,
 *     Appendix B); the memory write always keeps beta_t.
 *   - APF, Section 4.4 Eq. (7): d_{t+1} = clip(r_{t,h} d_t + same step), the step using the old d_t.
 *     Vector retention, Appendix A.5 (Prop. A.3): r_{t,h} I becomes diag(r_t), one gate per key
 *     coordinate (r_per_key = 1: r has the layout of k).
 *   - readout o_t = S_t q_t after the write (Section 4.1; the intra-chunk score of Listing 1 keeps
 *     the diagonal).  An optional scale multiplies q (Listing 1 uses K^-1/2; the equations use 1).
 *   - Gated DeltaNet with online scaling (OSGDN), Appendix B.1: an optional per-token, per-head
 *     state gate alpha_t in the post-gate residual form, Sbar = alpha_t S_{t-1},
 *     e_t = v_t - Sbar k_t, S_t = Sbar + beta_t e_t k~_t^T (phase 1 unchanged, Eq. (12)).
 *     alpha = NULL is the ungated rule (alpha = 1).
 *   - Kimi Delta Attention with online scaling (OSKDA), Appendix B.2: one state gate per key
 *     channel, Sbar = Diag(alpha_t) S_{t-1} in KDA's K x V convention; the state here is stored
 *     V x K (its transpose), so the gate scales column i of S by alpha_{t,i} (alpha_per_key = 1:
 *     alpha has the layout of k).  The write key k~ and the read key k keep their roles.
 *
 * Everything is a per-(batch, head) loop over tokens.  OpenMP runs independent heads in
 * parallel; within a head the arithmetic follows the definition above in order, in double.
 * Layouts (row-major, contiguous): q, k, k~ [B,T,H,K]; v, o [B,T,H,V]; beta, r, alpha [B,T,H]
 * (r [B,T,H,K] with r_per_key);
 * S [B,H,V,K]; d [B,H,K].  For a decode step T is absent: q, k [B,H,K], v, o [B,H,V], beta, r,
 * alpha [B,H].
 * Clamp: min(max(x, d_min), d_max) with IEEE fmin/fmax; +-inf bounds disable it.
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static size_t ix4(long b, long t, long h, long x, long T, long H, long X)
{
    return (size_t)(((b * T + t) * H + h) * X + x);
}

static double clip(double x, double lo, double hi) { return fmin(fmax(x, lo), hi); }

/* One phase-1 step on d (length K) for key k (length K): writes k~ = d . k (old d), then
 * updates d in place (Algorithm 1 lines "materialise write key" and "hypergradient step";
 * Eq. (7) when r is given: r[0] for every coordinate, or r[i] for coordinate i with r_per_key).
 * Returns a_t = beta <d_t, k_t^2> for diagnostics. */
static double phase1_step(double *d, const double *k, double *kt_out, int K, double beta,
                          const double *r, int r_per_key, double eta, double dmin, double dmax,
                          double eps, int beta_aware)
{
    double n = 0.0, align = 0.0;
    for (int i = 0; i < K; ++i) {
        double s = k[i] * k[i];
        n += s;
        align += d[i] * s;
        if (kt_out) kt_out[i] = d[i] * k[i];
    }
    double nbar = fmax(n, eps);
    double bp = beta_aware ? beta : 1.0;
    double step = eta * bp * (1.0 - bp * align) / nbar;
    for (int i = 0; i < K; ++i) {
        double s = k[i] * k[i];
        double ri = r ? r[r_per_key ? i : 0] : 1.0;
        d[i] = clip(ri * d[i] + step * s, dmin, dmax);
    }
    return beta * align;
}

/* One phase-2 step on S (V x K): S <- alpha S (the state gate, Appendix B.1; alpha = 1 without
 * it), or column i of S times alpha[i] with a gate per key channel (Appendix B.2), then
 * u = v - S k; S += beta u kt^T; o = scale * S q.  alpha may be NULL.  Returns |u|^2. */
static double phase2_step(double *S, const double *q, const double *k, const double *kt,
                          const double *v, double beta, const double *alpha, int alpha_per_key,
                          double *o, int K, int V, double scale, double *u /* scratch, length V */)
{
    double u2 = 0.0;
    if (alpha)
        for (int a = 0; a < V; ++a)
            for (int i = 0; i < K; ++i) S[(size_t)a * K + i] *= alpha[alpha_per_key ? i : 0];
    for (int a = 0; a < V; ++a) {
        double sk = 0.0;
        for (int i = 0; i < K; ++i) sk += S[(size_t)a * K + i] * k[i];
        u[a] = v[a] - sk;
        u2 += u[a] * u[a];
    }
    for (int a = 0; a < V; ++a)
        for (int i = 0; i < K; ++i) S[(size_t)a * K + i] += beta * u[a] * kt[i];
    if (o) {
        for (int a = 0; a < V; ++a) {
            double sq = 0.0;
            for (int i = 0; i < K; ++i) sq += S[(size_t)a * K + i] * q[i];
            o[a] = scale * sq;
        }
    }
    return u2;
}

static int set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
    return nthreads;
#else
    (void)nthreads;
    return 1;
#endif
}

/* Phase 1 alone (Algorithm 1 with the per-step clamp; Eq. (7) when r is given).
 * k_tilde [B,T,H,K] and d_out [B,H,K] are written; a_out [B,T,H] (optional) gets
 * a_t = beta_t <d_t, k_t^2>.  r and d0 may be NULL (r = 1, d0 = 1). */
int oracle_precond_scan(const double *k, const double *beta, const double *r, int r_per_key,
                        const double *d0, double *k_tilde, double *d_out, double *a_out, int B,
                        int T, int H, int K, double eta, double dmin, double dmax, double eps,
                        int beta_aware, int nthreads)
{
    if (B < 0 || T < 0 || H < 0 || K <= 0) return 1;
    int nt = set_threads(nthreads);
    (void)nt;
#pragma omp parallel for num_threads(nt) schedule(dynamic, 1)
    for (long bh = 0; bh < (long)B * H; ++bh) {
        long b = bh / H, h = bh % H;
        double *d = malloc(sizeof(double) * K);
        for (int i = 0; i < K; ++i) d[i] = d0 ? d0[(size_t)bh * K + i] : 1.0;
        for (long t = 0; t < T; ++t) {
            size_t kk = ix4(b, t, h, 0, T, H, K);
            size_t gg = ix4(b, t, h, 0, T, H, 1);
            double a = phase1_step(d, k + kk, k_tilde + kk, K, beta[gg],
                                   r ? r + (r_per_key ? kk : gg) : NULL, r_per_key, eta, dmin, dmax,
                                   eps, beta_aware);
            if (a_out) a_out[gg] = a;
        }
        memcpy(d_out + (size_t)bh * K, d, sizeof(double) * K);
        free(d);
    }
    return 0;
}

/* Phase 2 alone: the delta rule with the write key supplied (Eq. (2)/(5)), token by token, gated
 * by alpha when it is given (Appendix B.1).  o [B,T,H,V] and S_out [B,H,V,K] are written; S0 and
 * alpha may be NULL (zeros, no gate). */
int oracle_delta_phase2(const double *q, const double *k, const double *k_tilde, const double *v,
                        const double *beta, const double *alpha, int alpha_per_key, const double *S0, double *o,
                        double *S_out, int B,
                        int T, int H, int K, int V, double scale, int nthreads)
{
    if (B < 0 || T < 0 || H < 0 || K <= 0 || V <= 0) return 1;
    int nt = set_threads(nthreads);
    (void)nt;
#pragma omp parallel for num_threads(nt) schedule(dynamic, 1)
    for (long bh = 0; bh < (long)B * H; ++bh) {
        long b = bh / H, h = bh % H;
        size_t sz = (size_t)V * K;
        double *S = malloc(sizeof(double) * sz);
        double *u = malloc(sizeof(double) * V);
        if (S0) memcpy(S, S0 + (size_t)bh * sz, sizeof(double) * sz);
        else memset(S, 0, sizeof(double) * sz);
        for (long t = 0; t < T; ++t) {
            size_t kk = ix4(b, t, h, 0, T, H, K), vv = ix4(b, t, h, 0, T, H, V);
            size_t gg = ix4(b, t, h, 0, T, H, 1);
            phase2_step(S, q + kk, k + kk, k_tilde + kk, v + vv, beta[gg],
                        alpha ? alpha + (alpha_per_key ? kk : gg) : NULL, alpha_per_key, o + vv, K, V,
                        scale, u);
        }
        memcpy(S_out + (size_t)bh * sz, S, sizeof(double) * sz);
        free(u);
        free(S);
    }
    return 0;
}

/* The whole forward, both phases interleaved per token in the order of the definition:
 * emit k~_t with d_t, step d, read u_t with the ORIGINAL k_t, write with k~_t, read out o_t.
 * Optional diagnostics: a_out [B,T,H] = beta_t <d_t, k_t^2>, u2_out [B,T,H] = |u_t|^2. */
int oracle_osdn_forward(const double *q, const double *k, const double *v, const double *beta,
                        const double *r, int r_per_key, const double *alpha, int alpha_per_key,
                        const double *d0, const double *S0, double *o,
                        double *S_out, double *d_out, double *k_tilde, double *a_out,
                        double *u2_out, int B, int T, int H, int K, int V, double eta,
                        double dmin, double dmax, double eps, int beta_aware, double scale,
                        int nthreads)
{
    if (B < 0 || T < 0 || H < 0 || K <= 0 || V <= 0) return 1;
    int nt = set_threads(nthreads);
    (void)nt;
#pragma omp parallel for num_threads(nt) schedule(dynamic, 1)
    for (long bh = 0; bh < (long)B * H; ++bh) {
        long b = bh / H, h = bh % H;
        size_t sz = (size_t)V * K;
        double *S = malloc(sizeof(double) * sz);
        double *d = malloc(sizeof(double) * K);
        double *kt = malloc(sizeof(double) * K);
        double *u = malloc(sizeof(double) * V);
        if (S0) memcpy(S, S0 + (size_t)bh * sz, sizeof(double) * sz);
        else memset(S, 0, sizeof(double) * sz);
        for (int i = 0; i < K; ++i) d[i] = d0 ? d0[(size_t)bh * K + i] : 1.0;
        for (long t = 0; t < T; ++t) {
            size_t kk = ix4(b, t, h, 0, T, H, K), vv = ix4(b, t, h, 0, T, H, V);
            size_t gg = ix4(b, t, h, 0, T, H, 1);
            double a = phase1_step(d, k + kk, kt, K, beta[gg], r ? r + (r_per_key ? kk : gg) : NULL,
                                   r_per_key, eta, dmin, dmax, eps, beta_aware);
            if (k_tilde) memcpy(k_tilde + kk, kt, sizeof(double) * K);
            double u2 = phase2_step(S, q + kk, k + kk, kt, v + vv, beta[gg],
                                    alpha ? alpha + (alpha_per_key ? kk : gg) : NULL, alpha_per_key,
                                    o + vv, K, V, scale, u);
            if (a_out) a_out[gg] = a;
            if (u2_out) u2_out[gg] = u2;
        }
        memcpy(S_out + (size_t)bh * sz, S, sizeof(double) * sz);
        memcpy(d_out + (size_t)bh * K, d, sizeof(double) * K);
        free(u);
        free(kt);
        free(d);
        free(S);
    }
    return 0;
}

/* One recurrent decode step, in place on S [B,H,V,K] and d [B,H,K]: the forward above for a
 * single token.  q, k [B,H,K]; v, o [B,H,V]; beta, r, alpha [B,H] (r [B,H,K] with r_per_key; r
 * and alpha may be NULL). */
int oracle_decode_step(const double *q, const double *k, const double *v, const double *beta,
                       const double *r, int r_per_key, const double *alpha, int alpha_per_key, double *S,
                       double *d,
                       double *o, int B, int H, int K,
                       int V, double eta, double dmin, double dmax, double eps, int beta_aware,
                       double scale, int nthreads)
{
    if (B < 0 || H < 0 || K <= 0 || V <= 0) return 1;
    int nt = set_threads(nthreads);
    (void)nt;
#pragma omp parallel for num_threads(nt) schedule(dynamic, 1)
    for (long bh = 0; bh < (long)B * H; ++bh) {
        size_t sz = (size_t)V * K;
        double *kt = malloc(sizeof(double) * K);
        double *u = malloc(sizeof(double) * V);
        phase1_step(d + (size_t)bh * K, k + (size_t)bh * K, kt, K, beta[bh],
                    r ? r + (r_per_key ? (size_t)bh * K : (size_t)bh) : NULL, r_per_key, eta, dmin,
                    dmax, eps, beta_aware);
        phase2_step(S + (size_t)bh * sz, q + (size_t)bh * K, k + (size_t)bh * K, kt,
                    v + (size_t)bh * V, beta[bh],
                    alpha ? alpha + (alpha_per_key ? (size_t)bh * K : (size_t)bh) : NULL, alpha_per_key,
                    o + (size_t)bh * V, K, V, scale, u);
        free(u);
        free(kt);
    }
    return 0;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
