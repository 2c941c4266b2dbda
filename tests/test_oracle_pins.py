"""Pins for the fp64 oracle: each test checks the oracle against something other than itself --
an identity or closed form proved in "OSDN: Improving Delta Rule with Provable Online
Preconditioning in Linear Attention" (arXiv:2605.13473), a special case that reduces to a
textbook routine, a value printed on the pages (tests/golden/), or an independent formulation
(the chunkwise WY form of Appendix A.2).  A plausible slip in the oracle -- a dropped beta, a
swapped read/write key, a wrong sign, emission after the update, a transposed state -- fails at
least one of them.
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
INF = float("inf")


def rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def rand_problem(seed, B=1, T=32, H=2, K=8, V=6, unit_keys=True, apf=False):
    g = rng(seed)
    q = unit(g.standard_normal((B, T, H, K)))
    k = g.standard_normal((B, T, H, K))
    k = unit(k) if unit_keys else k
    v = g.standard_normal((B, T, H, V))
    beta = 1.0 / (1.0 + np.exp(-g.standard_normal((B, T, H))))
    r = 1.0 / (1.0 + np.exp(-(2.0 + g.standard_normal((B, T, H))))) if apf else None
    return q, k, v, beta, r


def step_forward(q, k, v, beta, r, d, S, **kw):
    """Run the oracle forward on a single token (T=1) carrying (d, S); returns (o, S, d, kt)."""
    out = oracle.osdn_forward(q[:, None], k[:, None], v[:, None], beta[:, None],
                              None if r is None else r[:, None], d, S, **kw)
    return out["o"][:, 0], out["S"], out["d"], out["k_tilde"][:, 0]


# ---------------------------------------------------------------------------------------------
# Special case that reduces to a textbook routine: eta = 0, d = 1 is DeltaNet (Section 3 /
# Algorithm 2 part (1)).
# ---------------------------------------------------------------------------------------------
def textbook_deltanet(q, k, v, beta):
    B, T, H, K = k.shape
    V = v.shape[-1]
    o = np.zeros((B, T, H, V))
    S_all = np.zeros((B, H, V, K))
    for b in range(B):
        for h in range(H):
            S = np.zeros((V, K))
            for t in range(T):
                u = v[b, t, h] - S @ k[b, t, h]
                S = S + beta[b, t, h] * np.outer(u, k[b, t, h])
                o[b, t, h] = S @ q[b, t, h]
            S_all[b, h] = S
    return o, S_all


def test_textbook_deltanet_at_eta0():
    q, k, v, beta, _ = rand_problem(1, B=2, T=40, H=3, K=8, V=5)
    out = oracle.osdn_forward(q, k, v, beta, eta=0.0)
    o_ref, S_ref = textbook_deltanet(q, k, v, beta)
    np.testing.assert_allclose(out["o"], o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(out["S"], S_ref, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(out["k_tilde"], k)
    np.testing.assert_array_equal(out["d"], np.ones_like(out["d"]))


# ---------------------------------------------------------------------------------------------
# Lemma 4.1 and its proof (Appendix A.3): S_t k_t - v_t = -u_t (1 - a_t), a_t = beta <d_t, k_t^2>,
# and the closed-form surrogate h_t = ((1 - a_t)^2 - 1) / (2 n_t).
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("beta_aware", [True, False])
def test_residual_identity_and_closed_form_surrogate(beta_aware):
    q, k, v, beta, _ = rand_problem(2, B=1, T=24, H=2, K=7, V=5, unit_keys=False)
    g = rng(22)
    d = g.uniform(0.5, 2.0, size=(1, 2, 7))
    S = g.standard_normal((1, 2, 5, 7)) * 0.3
    for t in range(24):
        S_prev, d_prev = S.copy(), d.copy()
        o, S, d, kt = step_forward(q[:, t], k[:, t], v[:, t], beta[:, t], None, d, S, eta=0.3,
                                   beta_aware=beta_aware)
        for h in range(2):
            kk, vv, bb = k[0, t, h], v[0, t, h], beta[0, t, h]
            u = vv - S_prev[0, h] @ kk
            a = bb * np.dot(d_prev[0, h], kk * kk)
            lhs = S[0, h] @ kk - vv
            np.testing.assert_allclose(lhs, -u * (1.0 - a), rtol=1e-11, atol=1e-12)
            n = np.dot(kk, kk)
            f_new, f_old = 0.5 * np.sum(lhs ** 2), 0.5 * np.sum(u ** 2)
            h_direct = (f_new - f_old) / (np.sum(u ** 2) * n)
            np.testing.assert_allclose(h_direct, ((1 - a) ** 2 - 1) / (2 * n), rtol=1e-10, atol=1e-13)
            # readout after the write: o_t = S_t q_t
            np.testing.assert_allclose(o[0, h], S[0, h] @ q[0, t, h], rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------------------------
# The phase-1 step is projected online gradient descent on the surrogate (Section 4.2, Eq. (4)),
# with retention on the old d for APF (Eq. (7)).  The gradient is taken here by central finite
# differences of h(d) = [f(S_t(d)) - f(S_{t-1})] / |grad f(S_{t-1})|^2, where S_t(d) comes from the
# oracle's own phase-2 step with write key d . k -- so the d update is tied to the memory write
# through the pages' definition, not through a retyped formula.
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("beta_aware,apf", [(True, False), (False, False), (True, True)])
def test_d_step_is_ogd_on_surrogate(beta_aware, apf):
    g = rng(3)
    K, V = 6, 4
    for trial in range(6):
        k = g.standard_normal(K) * (0.6 if trial % 2 else 1.0)
        v = g.standard_normal(V)
        S0 = g.standard_normal((V, K)) * 0.5
        beta = float(1 / (1 + np.exp(-g.standard_normal())))
        r = float(1 / (1 + np.exp(-(2 + g.standard_normal())))) if apf else 1.0
        d0 = g.uniform(0.6, 1.8, size=K)
        eta = 0.05
        b_fb = beta if beta_aware else 1.0  # the beta seen by the phase-1 feedback

        def h_of(dvec):
            kt = (dvec * k)[None, None, None, :]
            _, S1 = oracle.delta_phase2(k[None, None, None], k[None, None, None], kt,
                                        v[None, None, None], np.array([[[b_fb]]]), S0[None, None])
            res_new = S1[0, 0] @ k - v
            res_old = S0 @ k - v
            return (0.5 * res_new @ res_new - 0.5 * res_old @ res_old) / ((res_old @ res_old) * (k @ k))

        grad = np.zeros(K)
        step = 1e-4
        for i in range(K):
            e = np.zeros(K)
            e[i] = step
            grad[i] = (h_of(d0 + e) - h_of(d0 - e)) / (2 * step)
        _, d1 = oracle.precond_scan(k[None, None, None], np.array([[[beta]]]),
                                    np.array([[[r]]]) if apf else None, d0[None, None],
                                    eta=eta, d_min=-INF, d_max=INF, beta_aware=beta_aware)
        np.testing.assert_allclose(d1[0, 0], r * d0 - eta * grad, rtol=1e-8, atol=1e-10)
        # with the box switched on, the step is the projection of the same point
        _, d1c = oracle.precond_scan(k[None, None, None], np.array([[[beta]]]),
                                     np.array([[[r]]]) if apf else None, d0[None, None],
                                     eta=eta, d_min=0.9, d_max=1.2, beta_aware=beta_aware)
        np.testing.assert_allclose(d1c[0, 0], np.clip(r * d0 - eta * grad, 0.9, 1.2), rtol=1e-8,
                                   atol=1e-10)


def test_eps_floor_on_tiny_key():
    """|k|^2 = 1e-8 < eps = 1e-6: the normaliser is eps (Listing 1 clamps the squared norm).
    Hand-computed: step = 0.003*0.5*(1 - 0.5e-8)/1e-6 = 1499.9999925, d_0 += step * 1e-8."""
    k = np.array([1e-4, 0.0])[None, None, None]
    kt, d1 = oracle.precond_scan(k, np.array([[[0.5]]]), None, np.ones((1, 1, 2)), eta=0.003,
                                 eps=1e-6)
    assert d1[0, 0, 0] == pytest.approx(1.000014999999925, rel=0, abs=1e-15)
    assert d1[0, 0, 1] == 1.0
    np.testing.assert_array_equal(kt, k)  # emitted with d_1 = 1, before the update


# ---------------------------------------------------------------------------------------------
# Emission order (Algorithm 1: emit k~_t = d_t . k_t BEFORE the update) and projection onto D.
# ---------------------------------------------------------------------------------------------
def test_emission_uses_d_before_update():
    _, k, _, beta, r = rand_problem(4, B=1, T=6, H=1, K=5, V=2, apf=True)
    d0 = rng(44).uniform(0.5, 2.0, size=(1, 1, 5))
    kw = dict(eta=0.2, d_min=0.5, d_max=2.0)
    kt, _ = oracle.precond_scan(k, beta, r, d0, **kw)
    np.testing.assert_array_equal(kt[0, 0, 0], d0[0, 0] * k[0, 0, 0])
    for t in range(1, 6):
        _, d_t = oracle.precond_scan(k[:, :t], beta[:, :t], r[:, :t], d0, **kw)
        np.testing.assert_allclose(kt[0, t, 0], d_t[0, 0] * k[0, t, 0], rtol=1e-15, atol=0)


def test_box_invariant_and_binding():
    _, k, _, beta, _ = rand_problem(5, B=2, T=300, H=3, K=16, V=2, unit_keys=False)
    # long keys (beta <d, k^2> > 1) push d down, short keys push it up
    k = k * np.where(np.arange(2)[:, None, None, None] == 0, 1.0, 0.15)
    hit_lo = hit_hi = False
    for eta in (0.3, 3.0):
        kt, d = oracle.precond_scan(k, beta, None, None, eta=eta, d_min=0.5, d_max=2.0)
        dt = kt / k  # every intermediate d_t, read back through the emitted keys
        assert np.all(dt >= 0.5 - 1e-15) and np.all(dt <= 2.0 + 1e-15)
        assert np.all(d >= 0.5) and np.all(d <= 2.0)
        hit_lo |= bool(np.any(dt == 0.5))
        hit_hi |= bool(np.any(dt == 2.0))
    assert hit_lo and hit_hi  # the projection binds on both faces of the box


def test_fixed_point_leaves_d_unchanged():
    """If beta <d, k^2> = 1 the hypergradient vanishes (Appendix D.4: exact matching)."""
    k = unit(rng(6).standard_normal(8))
    beta = 0.8
    d0 = np.full(8, 1.0 / beta)  # <d, k^2> = 1/beta for a unit key
    _, d1 = oracle.precond_scan(k[None, None, None], np.array([[[beta]]]), None, d0[None, None],
                                eta=0.5, d_min=0.5, d_max=2.0)
    np.testing.assert_allclose(d1[0, 0], d0, rtol=0, atol=1e-15)


# ---------------------------------------------------------------------------------------------
# Corollary A.2: unit keys, d in [0.5, 2], beta in (0, 1)  =>  0 < a_t < 2 and q_t < 1, with the
# residual ratio f_t(S_t) / f_t(S_{t-1}) = (1 - a_t)^2 measured on the states.
# ---------------------------------------------------------------------------------------------
def test_stability_band_unit_keys():
    q, k, v, beta, r = rand_problem(7, B=1, T=64, H=2, K=8, V=5, apf=True)
    out = oracle.osdn_forward(q, k, v, beta, r, eta=0.3)
    a = beta * np.sum(out["k_tilde"] * k, axis=-1)  # beta <d_t . k_t, k_t> = beta <d_t, k_t^2>
    assert np.all(a > 0) and np.all(a < 2)
    d = None
    S = None
    for t in range(64):
        S_prev = np.zeros((1, 2, 5, 8)) if S is None else S
        _, S, d, _ = step_forward(q[:, t], k[:, t], v[:, t], beta[:, t], r[:, t], d, S, eta=0.3)
        for h in range(2):
            f_new = 0.5 * np.sum((S[0, h] @ k[0, t, h] - v[0, t, h]) ** 2)
            f_old = 0.5 * np.sum((S_prev[0, h] @ k[0, t, h] - v[0, t, h]) ** 2)
            np.testing.assert_allclose(f_new / f_old, (1 - a[0, t, h]) ** 2, rtol=1e-9)
            assert f_new < f_old


def test_worked_example():
    with open(os.path.join(GOLDEN, "worked_example.json")) as f:
        ex = json.load(f)
    k = np.array(ex["k"])[None, None, None]
    for case in ex["cases"]:
        d0 = np.array(case["d"])[None, None]
        v = np.ones((1, 1, 1, 1))
        out = oracle.osdn_forward(k, k, v, np.array([[[ex["beta"]]]]), d0=d0, eta=0.0)
        S1 = out["S"][0, 0]
        ratio = (0.5 * np.sum((S1 @ k[0, 0, 0] - 1.0) ** 2)) / 0.5
        assert ratio == pytest.approx(case["q"], abs=1e-15)
        assert out["a"][0, 0, 0] == pytest.approx(case["a"], abs=1e-15)


def test_counterexample_alternating():
    with open(os.path.join(GOLDEN, "counterexample.json")) as f:
        ex = json.load(f)
    T = ex["T"]
    v = np.array(ex["v"], dtype=float).reshape(1, T, 1, 1)
    one = np.ones((1, T, 1, 1))
    for eta in (0.003, 0.7):
        out = oracle.osdn_forward(one, one, v, np.full((1, T, 1), ex["beta"]),
                                  d0=np.full((1, 1, 1), ex["d0"]), eta=eta, d_min=0.5, d_max=2.0)
        np.testing.assert_array_equal(out["o"].reshape(T), np.array(ex["S_after_each_token"], float))
        assert out["d"][0, 0, 0] == ex["d_final"]


# ---------------------------------------------------------------------------------------------
# Corollary D.8: block-disjoint orthogonal class keys with fixed targets:
# prod_c F_c(S_T) / F_c(S_0) = prod_t q_t,  q_t = (1 - a_t)^2.
# ---------------------------------------------------------------------------------------------
def test_repeated_key_contraction_identity():
    g = rng(8)
    n_cls, blk = 4, 3
    K, V, T = n_cls * blk, 5, 40
    keys = np.zeros((n_cls, K))
    for c in range(n_cls):
        keys[c, c * blk:(c + 1) * blk] = unit(g.standard_normal(blk))
    targets = g.standard_normal((n_cls, V))
    cls = np.concatenate([np.arange(n_cls), g.integers(0, n_cls, T - n_cls)])
    k = keys[cls].reshape(1, T, 1, K)
    v = targets[cls].reshape(1, T, 1, V)
    beta = (1 / (1 + np.exp(-g.standard_normal(T)))).reshape(1, T, 1)
    S0 = g.standard_normal((1, 1, V, K))
    out = oracle.osdn_forward(k, k, v, beta, S0=S0, eta=0.4)
    a = beta[0, :, 0] * np.sum(out["k_tilde"][0, :, 0] * k[0, :, 0], axis=-1)
    log_q = np.sum(np.log((1 - a) ** 2))
    F = lambda S, c: 0.5 * np.sum((S @ keys[c] - targets[c]) ** 2)
    log_F = sum(np.log(F(out["S"][0, 0], c) / F(S0[0, 0], c)) for c in range(n_cls))
    assert log_F == pytest.approx(log_q, rel=1e-9, abs=1e-9)


# ---------------------------------------------------------------------------------------------
# Independent formulation: the chunkwise WY/UT form (Appendix A.2, Eqs. (8)-(11); Section 4.3
# Eq. (6)) written here in numpy from the equations, against the token recurrence.
# ---------------------------------------------------------------------------------------------
def chunk_form(q, k, kt, v, beta, S0, C):
    B, T, H, K = k.shape
    V = v.shape[-1]
    o = np.zeros((B, T, H, V))
    S_out = np.zeros((B, H, V, K))
    for b in range(B):
        for h in range(H):
            S = S0[b, h].copy()
            for c0 in range(0, T, C):
                sl = slice(c0, c0 + C)
                Kc, Ktc, Vc, Qc, bc = k[b, sl, h], kt[b, sl, h], v[b, sl, h], q[b, sl, h], beta[b, sl, h]
                n = Kc.shape[0]
                A = np.tril(bc[:, None] * (Kc @ Ktc.T), -1)
                Tm = np.linalg.inv(np.eye(n) + A)                     # Eq. (8)
                W = Tm @ (bc[:, None] * Kc)                            # Eq. (9)
                U = Tm @ (bc[:, None] * Vc)
                X = U - W @ S.T
                o[b, sl, h] = Qc @ S.T + np.tril(Qc @ Ktc.T, 0) @ X     # score keeps the diagonal
                S = S + X.T @ Ktc                                      # Eq. (11)
            S_out[b, h] = S
    return o, S_out


@pytest.mark.parametrize("C", [16, 64])
def test_chunk_form_equals_sequential(C):
    q, k, v, beta, r = rand_problem(9, B=1, T=256, H=2, K=16, V=12, apf=True)
    S0 = rng(99).standard_normal((1, 2, 12, 16)) * 0.1
    kt, _ = oracle.precond_scan(k, beta, r, None, eta=0.3)
    o_seq, S_seq = oracle.delta_phase2(q, k, kt, v, beta, S0)
    o_chk, S_chk = chunk_form(q, k, kt, v, beta, S0, C)
    np.testing.assert_allclose(o_seq, o_chk, rtol=0, atol=1e-11)
    np.testing.assert_allclose(S_seq, S_chk, rtol=0, atol=1e-11)


def test_wy_product_identity():
    """Eq. (10): prod_i (I - beta_i k_i k~_i^T) = I - W^T K~ (product ordered left to right)."""
    g = rng(10)
    C, K = 12, 7
    Kc = g.standard_normal((C, K)) * 0.4
    Ktc = Kc * g.uniform(0.5, 2.0, size=K)
    bc = 1 / (1 + np.exp(-g.standard_normal(C)))
    P = np.eye(K)
    for i in range(C):
        P = P @ (np.eye(K) - bc[i] * np.outer(Kc[i], Ktc[i]))
    W = np.linalg.inv(np.eye(C) + np.tril(bc[:, None] * (Kc @ Ktc.T), -1)) @ (bc[:, None] * Kc)
    np.testing.assert_allclose(P, np.eye(K) - W.T @ Ktc, rtol=0, atol=1e-13)


# ---------------------------------------------------------------------------------------------
# Structural consequences of the recurrence.
# ---------------------------------------------------------------------------------------------
def test_decoupling_two_phases_equal_interleaved():
    """Lemma 4.1 (i): the d trajectory needs only keys and gates, so phase 1 then phase 2 equals
    the per-token interleaving."""
    q, k, v, beta, r = rand_problem(11, B=2, T=50, H=2, K=8, V=6, apf=True)
    full = oracle.osdn_forward(q, k, v, beta, r, eta=0.2, scale=0.7)
    kt, d = oracle.precond_scan(k, beta, r, None, eta=0.2)
    o, S = oracle.delta_phase2(q, k, kt, v, beta, None, scale=0.7)
    np.testing.assert_array_equal(kt, full["k_tilde"])
    np.testing.assert_array_equal(d, full["d"])
    np.testing.assert_allclose(o, full["o"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(S, full["S"], rtol=0, atol=1e-13)


def test_continuation_split_equals_whole():
    q, k, v, beta, r = rand_problem(12, B=1, T=70, H=2, K=8, V=6, apf=True)
    kw = dict(eta=0.2)
    whole = oracle.osdn_forward(q, k, v, beta, r, **kw)
    first = oracle.osdn_forward(q[:, :33], k[:, :33], v[:, :33], beta[:, :33], r[:, :33], **kw)
    second = oracle.osdn_forward(q[:, 33:], k[:, 33:], v[:, 33:], beta[:, 33:], r[:, 33:],
                                 d0=first["d"], S0=first["S"], **kw)
    np.testing.assert_allclose(np.concatenate([first["o"], second["o"]], 1), whole["o"], atol=1e-13)
    np.testing.assert_allclose(second["S"], whole["S"], atol=1e-13)
    np.testing.assert_allclose(second["d"], whole["d"], atol=1e-15)


def test_decode_steps_equal_forward():
    q, k, v, beta, r = rand_problem(13, B=2, T=20, H=3, K=8, V=6, apf=True)
    g = rng(130)
    S0 = g.standard_normal((2, 3, 6, 8)) * 0.1
    d0 = g.uniform(0.5, 2.0, size=(2, 3, 8))
    kw = dict(eta=0.2, scale=0.5)
    whole = oracle.osdn_forward(q, k, v, beta, r, d0, S0, **kw)
    S, d = S0, d0
    for t in range(20):
        o, S, d = oracle.decode_step(q[:, t], k[:, t], v[:, t], beta[:, t], S, d, r[:, t], **kw)
        np.testing.assert_allclose(o, whole["o"][:, t], atol=1e-13)
    np.testing.assert_allclose(S, whole["S"], atol=1e-13)
    np.testing.assert_allclose(d, whole["d"], atol=1e-15)


def test_retention_one_is_eq4():
    """Eq. (7) with r = 1 recovers Eq. (4)."""
    q, k, v, beta, _ = rand_problem(14, B=1, T=40, H=2, K=8, V=6)
    a = oracle.osdn_forward(q, k, v, beta, None, eta=0.2)
    b = oracle.osdn_forward(q, k, v, beta, np.ones_like(beta), eta=0.2)
    for key in ("o", "S", "d", "k_tilde"):
        np.testing.assert_array_equal(a[key], b[key])


def test_scale_multiplies_readout():
    q, k, v, beta, _ = rand_problem(15, B=1, T=16, H=1, K=8, V=4)
    a = oracle.osdn_forward(q, k, v, beta, scale=1.0)
    b = oracle.osdn_forward(q, k, v, beta, scale=0.125)
    np.testing.assert_allclose(b["o"], 0.125 * a["o"], rtol=1e-15, atol=0)
    np.testing.assert_array_equal(a["S"], b["S"])


# ---------------------------------------------------------------------------------------------
# Vector retention (Appendix A.5, Prop. A.3): r_{t,h} I becomes diag(r_t), one gate per key
# coordinate, with the rest of the step unchanged.
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("beta_aware", [True, False])
def test_vector_retention_step_is_the_affine_matrix_form(beta_aware):
    """Prop. A.3 written as a matrix: d' = (diag(r) - eta b^2 / n s s^T) d + eta b / n s."""
    g = rng(21)
    K = 7
    for trial in range(5):
        k = g.standard_normal(K)
        beta = float(1 / (1 + np.exp(-g.standard_normal())))
        r = 1 / (1 + np.exp(-(1.5 + g.standard_normal(K))))
        d0 = g.uniform(0.6, 1.8, size=K)
        eta = 0.3
        b = beta if beta_aware else 1.0
        s = k * k
        n = max(s.sum(), 1e-6)
        want = (np.diag(r) - eta * b * b / n * np.outer(s, s)) @ d0 + eta * b / n * s
        kt, d1 = oracle.precond_scan(k[None, None, None], np.array([[[beta]]]), r[None, None, None],
                                     d0[None, None], eta=eta, d_min=-INF, d_max=INF, beta_aware=beta_aware)
        np.testing.assert_allclose(d1[0, 0], want, rtol=1e-13, atol=1e-15)
        np.testing.assert_array_equal(kt[0, 0, 0], d0 * k)  # emitted with the old d
        _, d1c = oracle.precond_scan(k[None, None, None], np.array([[[beta]]]), r[None, None, None],
                                     d0[None, None], eta=eta, d_min=0.9, d_max=1.2, beta_aware=beta_aware)
        np.testing.assert_allclose(d1c[0, 0], np.clip(want, 0.9, 1.2), rtol=1e-13, atol=1e-15)


def test_vector_retention_with_equal_gates_is_the_scalar_gate():
    q, k, v, beta, r = rand_problem(22, B=2, T=24, H=2, K=8, V=5, apf=True)
    a = oracle.osdn_forward(q, k, v, beta, r, eta=0.2)
    b = oracle.osdn_forward(q, k, v, beta, np.repeat(r[..., None], k.shape[-1], axis=-1), eta=0.2)
    for key in ("o", "S", "d", "k_tilde"):
        np.testing.assert_array_equal(a[key], b[key])


def test_vector_retention_eta0_is_a_product_of_gates():
    """eta = 0: d_t = d_0 . prod_{s<t} r_s per coordinate (inside the box), k~_t = d_t . k_t."""
    g = rng(23)
    B, T, H, K = 1, 12, 2, 5
    k = g.standard_normal((B, T, H, K))
    beta = np.full((B, T, H), 0.5)
    r = g.uniform(0.8, 1.0, size=(B, T, H, K))
    d0 = g.uniform(0.8, 1.5, size=(B, H, K))
    kt, d = oracle.precond_scan(k, beta, r, d0, eta=0.0, d_min=0.0, d_max=INF)
    prod = np.concatenate([np.ones((B, 1, H, K)), np.cumprod(r, axis=1)], axis=1)  # prod_{s<t}
    np.testing.assert_allclose(kt, d0[:, None] * prod[:, :T] * k, rtol=1e-13)
    np.testing.assert_allclose(d, d0 * prod[:, T], rtol=1e-13)


# ---------------------------------------------------------------------------------------------
# The OSGDN state gate (Appendix B.1): S_t = alpha_t S_{t-1} (I - beta_t k_t k~_t^T)
# + beta_t v_t k~_t^T, post-gate residual; phase 1 unchanged.
# ---------------------------------------------------------------------------------------------
def gates(seed, shape, lo=0.6):
    return rng(seed).uniform(lo, 1.0, size=shape)


def textbook_gated_deltanet(q, k, v, beta, alpha):
    """Gated DeltaNet in its transition-matrix form S_t = S_{t-1} (alpha_t (I - beta_t k_t k_t^T))
    + beta_t v_t k_t^T, o_t = S_t q_t (written independently of the oracle's residual form)."""
    B, T, H, K = k.shape
    V = v.shape[-1]
    o = np.zeros((B, T, H, V))
    S_all = np.zeros((B, H, V, K))
    for b in range(B):
        for h in range(H):
            S = np.zeros((V, K))
            for t in range(T):
                kk = k[b, t, h]
                S = S @ (alpha[b, t, h] * (np.eye(K) - beta[b, t, h] * np.outer(kk, kk))) \
                    + beta[b, t, h] * np.outer(v[b, t, h], kk)
                o[b, t, h] = S @ q[b, t, h]
            S_all[b, h] = S
    return o, S_all


def gated_chunk_form(q, k, kt, v, beta, alpha, S0, C):
    """Eqs. (13)-(15) with the readout of each chunk: with gamma_i the gate product from the chunk
    start through token i, A_ij = beta_i (gamma_i / gamma_j) <k_i, k~_j> (j < i),
    M = (I + A)^-1 diag(beta), W = M (gamma . K), U = M V, X = U - W S^T,
    O = diag(gamma) Q S^T + (tril(Q K~^T, 0) . gamma_i / gamma_j) X,
    S <- gamma_C S + X^T (rho . K~), rho_j = gamma_C / gamma_j."""
    B, T, H, K = k.shape
    V = v.shape[-1]
    o = np.zeros((B, T, H, V))
    S_out = np.zeros((B, H, V, K))
    for b in range(B):
        for h in range(H):
            S = S0[b, h].copy()
            for c0 in range(0, T, C):
                sl = slice(c0, c0 + C)
                Kc, Ktc, Vc, Qc, bc = k[b, sl, h], kt[b, sl, h], v[b, sl, h], q[b, sl, h], beta[b, sl, h]
                gam = np.cumprod(alpha[b, sl, h])
                ratio = gam[:, None] / gam[None, :]
                n = Kc.shape[0]
                A = np.tril(bc[:, None] * ratio * (Kc @ Ktc.T), -1)
                M = np.linalg.inv(np.eye(n) + A) @ np.diag(bc)        # Eq. (13)
                W = M @ (gam[:, None] * Kc)                           # Eq. (14)
                U = M @ Vc
                X = U - W @ S.T
                o[b, sl, h] = gam[:, None] * (Qc @ S.T) + (np.tril(Qc @ Ktc.T, 0) * ratio) @ X
                S = gam[-1] * S + X.T @ ((gam[-1] / gam)[:, None] * Ktc)  # Eq. (15)
            S_out[b, h] = S
    return o, S_out


def test_gate_one_is_the_ungated_rule():
    q, k, v, beta, r = rand_problem(31, B=2, T=40, H=2, K=8, V=6, apf=True)
    a = oracle.osdn_forward(q, k, v, beta, r, eta=0.2)
    b = oracle.osdn_forward(q, k, v, beta, r, alpha=np.ones_like(beta), eta=0.2)
    for key in ("o", "S", "d", "k_tilde"):
        np.testing.assert_array_equal(a[key], b[key])


def test_gated_eta0_is_textbook_gated_deltanet():
    q, k, v, beta, _ = rand_problem(32, B=2, T=48, H=3, K=8, V=6)
    alpha = gates(33, beta.shape)
    out = oracle.osdn_forward(q, k, v, beta, alpha=alpha, eta=0.0)
    o_ref, S_ref = textbook_gated_deltanet(q, k, v, beta, alpha)
    np.testing.assert_allclose(out["o"], o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(out["S"], S_ref, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(out["k_tilde"], k)


@pytest.mark.parametrize("C", [16, 64])
def test_gated_chunk_form_equals_sequential(C):
    q, k, v, beta, r = rand_problem(34, B=1, T=256, H=2, K=16, V=12, apf=True)
    alpha = gates(35, beta.shape, lo=0.3)
    S0 = rng(36).standard_normal((1, 2, 12, 16)) * 0.1
    kt, _ = oracle.precond_scan(k, beta, r, None, eta=0.3)
    o_seq, S_seq = oracle.delta_phase2(q, k, kt, v, beta, S0, alpha=alpha)
    o_chk, S_chk = gated_chunk_form(q, k, kt, v, beta, alpha, S0, C)
    np.testing.assert_allclose(o_seq, o_chk, rtol=0, atol=1e-11)
    np.testing.assert_allclose(S_seq, S_chk, rtol=0, atol=1e-11)


def test_zero_gate_forgets_the_state():
    """alpha_t = 0: the post-gate reference is empty, so S_t = beta_t v_t k~_t^T and everything
    after t is the rule started from S = 0 at t."""
    q, k, v, beta, _ = rand_problem(37, B=1, T=30, H=2, K=8, V=6)
    alpha = gates(38, beta.shape)
    alpha[:, 12] = 0.0
    S0 = rng(39).standard_normal((1, 2, 6, 8))
    kt, _ = oracle.precond_scan(k, beta, None, None, eta=0.2)
    o, S = oracle.delta_phase2(q, k, kt, v, beta, S0, alpha=alpha)
    o2, S2 = oracle.delta_phase2(q[:, 12:], k[:, 12:], kt[:, 12:], v[:, 12:], beta[:, 12:], None,
                                 alpha=alpha[:, 12:])
    np.testing.assert_array_equal(o[:, 12:], o2)
    np.testing.assert_array_equal(S, S2)


def test_gated_decode_steps_equal_forward():
    q, k, v, beta, r = rand_problem(40, B=2, T=6, H=2, K=8, V=5, apf=True)
    alpha = gates(41, beta.shape)
    g = rng(42)
    S = g.standard_normal((2, 2, 5, 8)) * 0.1
    d = g.uniform(0.6, 1.8, size=(2, 2, 8))
    full = oracle.osdn_forward(q, k, v, beta, r, d, S, alpha=alpha, eta=0.2)
    for t in range(6):
        o, S, d = oracle.decode_step(q[:, t], k[:, t], v[:, t], beta[:, t], S, d, r[:, t],
                                     alpha=alpha[:, t], eta=0.2)
        np.testing.assert_allclose(o, full["o"][:, t], rtol=0, atol=1e-13)
    np.testing.assert_allclose(S, full["S"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(d, full["d"], rtol=0, atol=1e-15)


# ---------------------------------------------------------------------------------------------
# The backward reference (oracle/backward.py): its forward is the C oracle's, and its gradients
# are central finite differences of the C oracle's forward (independent of autograd).
# ---------------------------------------------------------------------------------------------
from oracle import backward as obw  # noqa: E402


def bw_problem(seed, T=12, K=4, V=3, H=2, apf=False, gated=False, per_key=False):
    q, k, v, beta, r = rand_problem(seed, B=1, T=T, H=H, K=K, V=V, apf=apf)
    g = rng(seed + 100)
    if apf and per_key:
        r = g.uniform(0.6, 1.0, size=k.shape)
    alpha = g.uniform(0.6, 1.0, size=(k.shape if gated == "key" else beta.shape)) if gated else None
    d0 = g.uniform(0.7, 1.6, size=(1, H, K))
    S0 = g.standard_normal((1, H, V, K)) * 0.3
    return dict(q=q, k=k, v=v, beta=beta, r=r, d0=d0, S0=S0, alpha=alpha)


@pytest.mark.parametrize("apf,gated,per_key,beta_aware", [
    (False, False, False, True), (True, False, False, True), (True, False, True, False), (False, True, False, True),
    (False, "key", False, True)])
def test_backward_reference_forward_is_the_oracle(apf, gated, per_key, beta_aware):
    p = bw_problem(81, T=20, K=8, V=5, apf=apf, gated=gated, per_key=per_key)
    kw = dict(eta=0.3, d_min=0.5, d_max=2.0, eps=1e-6, beta_aware=beta_aware, scale=0.7)
    ref = oracle.osdn_forward(p["q"], p["k"], p["v"], p["beta"], p["r"], p["d0"], p["S0"], alpha=p["alpha"], **kw)
    t = {n: obw._t(x) for n, x in p.items()}
    o, S, d, kt = obw.forward(t["q"], t["k"], t["v"], t["beta"], t["r"], t["d0"], t["S0"], t["alpha"], **kw)
    np.testing.assert_allclose(o.numpy(), ref["o"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(S.numpy(), ref["S"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(d.numpy(), ref["d"], rtol=1e-14)
    np.testing.assert_allclose(kt.numpy(), ref["k_tilde"], rtol=1e-14)


@pytest.mark.parametrize("apf,gated,per_key,beta_aware", [
    (False, False, False, True), (True, False, False, False), (True, False, True, True), (False, True, False, True),
    (False, "key", False, True)])
def test_backward_reference_equals_finite_differences(apf, gated, per_key, beta_aware):
    """<grad_X L, delta> against (L(X + h delta) - L(X - h delta)) / 2h with the C oracle's forward,
    for every input X and a random direction delta; the upstream gradients weight o, S_T, d_T, k~."""
    p = bw_problem(82, T=14, K=5, V=3, apf=apf, gated=gated, per_key=per_key)
    kw = dict(eta=0.3, d_min=0.5, d_max=2.0, eps=1e-6, beta_aware=beta_aware, scale=0.9)
    g = rng(83)
    up = dict(do=g.standard_normal(p["v"].shape), dS=g.standard_normal(p["S0"].shape),
              dd=g.standard_normal(p["d0"].shape), dkt=g.standard_normal(p["k"].shape))

    def loss(pp):
        f = oracle.osdn_forward(pp["q"], pp["k"], pp["v"], pp["beta"], pp["r"], pp["d0"], pp["S0"], alpha=pp["alpha"],
                                **kw)
        return (np.sum(f["o"] * up["do"]) + np.sum(f["S"] * up["dS"]) + np.sum(f["d"] * up["dd"])
                + np.sum(f["k_tilde"] * up["dkt"]))

    grads = obw.layer_backward(p["q"], p["k"], p["v"], p["beta"], p["r"], p["d0"], p["S0"], p["alpha"], **up, **kw)
    h = 1e-6
    for name in ("q", "k", "v", "beta", "r", "d0", "S0", "alpha"):
        if p[name] is None:
            continue
        delta = g.standard_normal(p[name].shape)
        plus = dict(p, **{name: p[name] + h * delta})
        minus = dict(p, **{name: p[name] - h * delta})
        fd = (loss(plus) - loss(minus)) / (2 * h)
        an = float(np.sum(grads["d" + name] * delta))
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)


def test_backward_reference_clipped_coordinates_pass_no_gradient():
    """A coordinate that stays clipped at every step: d_T does not depend on d0 there."""
    p = bw_problem(84, T=10, K=4, V=3)
    p["d0"][..., 0] = 0.1   # below d_min = 0.5, with eta = 0 the first step clips it to 0.5 for good
    grads = obw.layer_backward(p["q"], p["k"], p["v"], p["beta"], None, p["d0"], p["S0"],
                               dd=np.ones_like(p["d0"]), eta=0.0, d_min=0.5, d_max=2.0)
    assert np.all(grads["dd0"][..., 0] == 0.0)
    np.testing.assert_allclose(grads["dd0"][..., 1:], 1.0, rtol=0, atol=0)  # eta = 0: d_T = d0 inside the box


# ---------------------------------------------------------------------------------------------
# One state gate per key channel (OSKDA, Appendix B.2): KDA's K x V state S_t =
# (I - beta_t k~_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k~_t v_t^T, o_t = S_t^T q_t; this library
# stores the V x K transpose.
# ---------------------------------------------------------------------------------------------
def textbook_kda(q, k, kt, v, beta, alpha):
    """KDA with the write key on the left, in its own K x V convention (written independently)."""
    B, T, H, K = k.shape
    V = v.shape[-1]
    o = np.zeros((B, T, H, V))
    S_all = np.zeros((B, H, K, V))
    for b in range(B):
        for h in range(H):
            S = np.zeros((K, V))
            for t in range(T):
                a = (np.eye(K) - beta[b, t, h] * np.outer(kt[b, t, h], k[b, t, h])) @ np.diag(alpha[b, t, h])
                S = a @ S + beta[b, t, h] * np.outer(kt[b, t, h], v[b, t, h])
                o[b, t, h] = S.T @ q[b, t, h]
            S_all[b, h] = S
    return o, S_all


def test_channel_gates_follow_textbook_kda():
    q, k, v, beta, _ = rand_problem(91, B=2, T=30, H=2, K=6, V=4)
    alpha = gates(92, k.shape, lo=0.5)
    kt, _ = oracle.precond_scan(k, beta, None, None, eta=0.3)
    o, S = oracle.delta_phase2(q, k, kt, v, beta, None, alpha=alpha)
    o_ref, S_ref = textbook_kda(q, k, kt, v, beta, alpha)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(np.swapaxes(S, -1, -2), S_ref, rtol=0, atol=1e-12)


def test_equal_channel_gates_are_the_head_gate():
    q, k, v, beta, r = rand_problem(93, B=1, T=25, H=2, K=6, V=4, apf=True)
    alpha = gates(94, beta.shape)
    a = oracle.osdn_forward(q, k, v, beta, r, alpha=alpha, eta=0.2)
    b = oracle.osdn_forward(q, k, v, beta, r, alpha=np.repeat(alpha[..., None], k.shape[-1], axis=-1), eta=0.2)
    for key in ("o", "S", "d", "k_tilde"):
        np.testing.assert_array_equal(a[key], b[key])


def test_channel_gated_decode_steps_equal_forward():
    q, k, v, beta, r = rand_problem(95, B=2, T=5, H=2, K=8, V=5, apf=True)
    alpha = gates(96, k.shape)
    g = rng(97)
    S = g.standard_normal((2, 2, 5, 8)) * 0.1
    d = g.uniform(0.6, 1.8, size=(2, 2, 8))
    full = oracle.osdn_forward(q, k, v, beta, r, d, S, alpha=alpha, eta=0.2)
    for t in range(5):
        o, S, d = oracle.decode_step(q[:, t], k[:, t], v[:, t], beta[:, t], S, d, r[:, t], alpha=alpha[:, t], eta=0.2)
        np.testing.assert_allclose(o, full["o"][:, t], rtol=0, atol=1e-13)
    np.testing.assert_allclose(S, full["S"], rtol=0, atol=1e-13)
