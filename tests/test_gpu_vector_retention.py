"""GPU parity of the vector retention (one APF gate per key coordinate, diag(r_t) in place of
r_{t,h} I: "OSDN: Improving Delta Rule with Provable Online Preconditioning in Linear Attention",
Appendix A.5, Prop. A.3) against the fp64 oracle: the phase-1 scan, the layer call and the decode
step.  Bars as for the per-head gate: k~ and d within 1e-5 relative; o and S max-abs 2e-2 (bf16)
or 1e-4 (fp32).  16-bit keys with K = 128 take the blocked scan (every block by Jacobi sweeps on
the clipped recurrence, one gate per coordinate); fp32 keys and K = 64 take the token-by-token
kernel, where a vector of equal gates must give exactly what the per-head gate gives."""
import numpy as np
import pytest
import torch

import oracle
from preconditioned_delta_rule_gb300 import binding, osdn_decode_step, osdn_layer_fwd, osdn_precond_scan
from preconditioned_delta_rule_gb300 import workloads as W
from tests._parity import assert_maxabs, assert_rel, np64, to_dev

pytestmark = pytest.mark.gpu


def vector_gates(shape, seed, mean=2.0):
    """Gates in (0, 1): sigmoid(mean + N(0, 1)) per key coordinate, like the per-head APF gates."""
    g = torch.Generator().manual_seed(seed)
    return torch.sigmoid(mean + torch.randn(*shape, generator=g))


@pytest.mark.parametrize("name,B,H,T,kt_dtype", [
    ("layer_1p3b_apf", 2, 4, 512, torch.float32),   # bf16 keys, K = 128
    ("layer_1p3b_apf", 1, 3, 200, torch.bfloat16),  # ragged T, bf16 write keys
    ("tiny_f32", 2, 2, 256, torch.float32),          # fp32 keys, K = 64
])
def test_scan_vector_retention(name, B, H, T, kt_dtype):
    w = W.WORKLOADS[name]
    inp = W.make_prefill(w, B=B, H=H, T=T, seed=41)
    K = inp["k"].shape[-1]
    # gates near 1 and a wide box keep d inside it (with sigmoid(2 + N) gates d collapses onto
    # d_min within a few tokens and every coordinate ends equal)
    r = vector_gates((B, T, H, K), 7, mean=4.0)
    box = dict(d_min=0.1, d_max=4.0)
    dev = to_dev(inp)
    kt, d = osdn_precond_scan(dev["k"], dev["beta"], r.cuda(), None, kt_dtype=kt_dtype, eta=0.3,
                              eps=w.eps, **box)
    torch.cuda.synchronize()
    kt_ref, d_ref = oracle.precond_scan(inp["k"], inp["beta"], r, None, eta=0.3, eps=w.eps, **box)
    ulp = 2.0 ** -8 if kt_dtype == torch.bfloat16 else 0.0
    assert_rel(kt, kt_ref, 1e-5 + ulp, what="k_tilde")
    assert_rel(d, d_ref, 1e-5, what="d")
    # the gates act per coordinate: the trajectory leaves the per-head family (coordinates with
    # the same key history but different gates end at different d)
    assert np.ptp(np64(d)) > 0


def test_equal_vector_gates_match_the_head_gate():
    w = W.WORKLOADS["layer_1p3b_apf"]
    inp = W.make_prefill(w, B=1, H=4, T=256, seed=42)
    dev = to_dev(inp)
    r_vec = dev["r"][..., None].expand(*dev["r"].shape, 128).contiguous()
    kw = dict(kt_dtype=torch.float32, eta=0.3, d_min=w.d_min, d_max=w.d_max, eps=w.eps)
    # fp32 keys: the token-by-token kernel for both gate layouts, the same arithmetic
    kf = dev["k"].float()
    kt1, d1 = osdn_precond_scan(kf, dev["beta"], r_vec, None, **kw)
    kt2, d2 = osdn_precond_scan(kf, dev["beta"], dev["r"], None, **kw)
    # 16-bit keys: the blocked scan, clipped sweeps for the vector against the Gram solve for the
    # head gate (the same recurrence, reassociated)
    kt3, d3 = osdn_precond_scan(dev["k"], dev["beta"], r_vec, None, **kw)
    kt4, d4 = osdn_precond_scan(dev["k"], dev["beta"], dev["r"], None, **kw)
    torch.cuda.synchronize()
    assert torch.equal(kt1, kt2) and torch.equal(d1, d2)
    assert_rel(kt3, np64(kt4), 1e-5, what="k_tilde, vector vs head gate")
    assert_rel(d3, np64(d4), 1e-5, what="d, vector vs head gate")
    kt_ref, d_ref = oracle.precond_scan(inp["k"], inp["beta"], inp["r"], None, eta=0.3, d_min=w.d_min,
                                        d_max=w.d_max, eps=w.eps)
    assert_rel(kt3, kt_ref, 1e-5, what="k_tilde")
    assert_rel(d3, d_ref, 1e-5, what="d")


def test_scan_vector_retention_full_size():
    """The bench's vector-retention workload (1.3B-shaped, B4 H16 T4096, bf16 keys, gates
    sigmoid(4 + N(0, 1)) per coordinate) with a start state, on the blocked scan."""
    w = W.WORKLOADS["layer_1p3b_apf"]
    inp = W.make_prefill(w)
    B, T, H, K = inp["k"].shape
    r = torch.sigmoid(4.0 + torch.randn(B, T, H, K, generator=torch.Generator().manual_seed(4)))
    d0 = torch.rand(B, H, K, generator=torch.Generator().manual_seed(5)) * 1.5 + 0.5
    dev = to_dev(inp)
    kw = dict(eta=w.eta, d_min=w.d_min, d_max=w.d_max, eps=w.eps)
    kt, d = osdn_precond_scan(dev["k"], dev["beta"], r.cuda(), d0.cuda(), kt_dtype=torch.float32, **kw)
    torch.cuda.synchronize()
    kt_ref, d_ref = oracle.precond_scan(inp["k"], inp["beta"], r, d0, **kw)
    assert_rel(kt, kt_ref, 1e-5, what="k_tilde")
    assert_rel(d, d_ref, 1e-5, what="d")


@pytest.mark.parametrize("kt_dtype", [torch.bfloat16, torch.float32])
def test_vector_retention_parallel_emission_matches_in_kernel_emission(kt_dtype):
    """With a workspace the write keys come from the parallel emission kernel (each thread reads
    its coordinate's gates); without one the scan writes them: the same replay, bit-identical."""
    w = W.WORKLOADS["layer_1p3b_apf"]
    B, H, T = 2, 4, 1000  # ragged last block
    inp = W.make_prefill(w, B=B, H=H, T=T, seed=44)
    r = vector_gates((B, T, H, 128), 9, mean=4.0).cuda()
    dev = to_dev(inp)
    kw = dict(kt_dtype=kt_dtype, eta=w.eta, d_min=w.d_min, d_max=w.d_max, eps=w.eps)
    kt0, d0 = osdn_precond_scan(dev["k"], dev["beta"], r, None, workspace=False, **kw)
    need = binding.osdn_precond_scan_workspace_bytes(B, T, H, 128, dev["k"].dtype)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")
    kt1, d1 = osdn_precond_scan(dev["k"], dev["beta"], r, None, workspace=ws, **kw)
    torch.cuda.synchronize()
    assert torch.equal(kt0, kt1) and torch.equal(d0, d1)
    kt_ref, d_ref = oracle.precond_scan(inp["k"], inp["beta"], r.cpu(), None, eta=w.eta, d_min=w.d_min,
                                        d_max=w.d_max, eps=w.eps)
    ulp = 2.0 ** -8 if kt_dtype == torch.bfloat16 else 0.0
    assert_rel(kt0, kt_ref, 1e-5 + ulp, what="k_tilde")
    assert_rel(d0, d_ref, 1e-5, what="d")


def test_vector_gates_above_one_and_clipping():
    """Gates in [0.95, 1.05] (the sweeps' contraction bound no longer holds: they run until no step
    size moves) and a narrow box: about 4 % of the coordinates end on each face."""
    w = W.WORKLOADS["layer_1p3b_apf"]
    B, H, T = 1, 4, 640
    inp = W.make_prefill(w, B=B, H=H, T=T, seed=45)
    g = torch.Generator().manual_seed(10)
    r = 0.95 + 0.1 * torch.rand(B, T, H, 128, generator=g)
    box = dict(d_min=0.8, d_max=1.25)
    dev = to_dev(inp)
    kt, d = osdn_precond_scan(dev["k"], dev["beta"], r.cuda(), None, kt_dtype=torch.float32, eta=0.3,
                              eps=w.eps, **box)
    torch.cuda.synchronize()
    kt_ref, d_ref = oracle.precond_scan(inp["k"], inp["beta"], r, None, eta=0.3, eps=w.eps, **box)
    assert_rel(kt, kt_ref, 1e-5, what="k_tilde")
    assert_rel(d, d_ref, 1e-5, what="d")
    dd = np64(d)
    lo, hi = float(np.float32(0.8)), float(np.float32(1.25))  # the box as the fp32 state holds it
    assert np.any(dd == lo) and np.any(dd == hi) and np.any((dd > lo) & (dd < hi))


def test_layer_vector_retention_against_oracle():
    w = W.WORKLOADS["layer_1p3b_apf"]
    B, H, T = 2, 4, 384
    inp = W.make_prefill(w, B=B, H=H, T=T, seed=43)
    r = vector_gates((B, T, H, 128), 8)
    dev = to_dev(inp)
    o, S, d, kt = osdn_layer_fwd(dev["q"], dev["k"], dev["v"], dev["beta"], r.cuda(), eta=0.3,
                                 d_min=w.d_min, d_max=w.d_max, eps=w.eps)
    torch.cuda.synchronize()
    ref = oracle.osdn_forward(inp["q"], inp["k"], inp["v"], inp["beta"], r, eta=0.3, d_min=w.d_min,
                              d_max=w.d_max, eps=w.eps)
    assert_rel(kt, ref["k_tilde"], 1e-5 + 2.0 ** -8, what="k_tilde (bf16)")
    assert_rel(d, ref["d"], 1e-5, what="d")
    assert_maxabs(o, ref["o"], 2e-2, what="o")
    assert_maxabs(S, ref["S"], 2e-2, what="S")


@pytest.mark.parametrize("dtype,K,V", [(torch.bfloat16, 128, 128), (torch.float32, 64, 128)])
def test_decode_vector_retention(dtype, K, V):
    g = torch.Generator().manual_seed(K + V + 1)
    B, H, steps = 3, 5, 6
    q = torch.nn.functional.normalize(torch.randn(steps, B, H, K, generator=g), dim=-1).to(dtype)
    k = torch.nn.functional.normalize(torch.randn(steps, B, H, K, generator=g), dim=-1).to(dtype)
    v = torch.randn(steps, B, H, V, generator=g).to(dtype)
    beta = torch.sigmoid(torch.randn(steps, B, H, generator=g))
    r = vector_gates((steps, B, H, K), K)
    S = torch.randn(B, H, V, K, generator=g) * 0.05
    d = torch.rand(B, H, K, generator=g) * 1.5 + 0.5
    S_ref, d_ref = np64(S), np64(d)
    Sd, dd = S.cuda(), d.cuda()
    tol = 1e-4 if dtype == torch.float32 else 2e-2
    for t in range(steps):
        o = osdn_decode_step(q[t].cuda(), k[t].cuda(), v[t].cuda(), beta[t].cuda(), Sd, dd,
                             r[t].cuda(), eta=0.3)
        torch.cuda.synchronize()
        o_ref, S_ref, d_ref = oracle.decode_step(q[t], k[t], v[t], beta[t], S_ref, d_ref, r[t],
                                                 eta=0.3)
        assert_maxabs(o, o_ref, tol, what=f"o step {t}")
    assert_maxabs(Sd, S_ref, tol, what="S")
    assert_rel(dd, d_ref, 1e-5, what="d")


def test_scan_vector_retention_fp16_keys_not_beta_aware():
    """fp16 keys on the blocked scan's vector-gate mode, with the step not fed by beta."""
    w = W.WORKLOADS["layer_1p3b_apf"]
    B, H, T = 2, 3, 448
    inp = W.make_prefill(w, B=B, H=H, T=T, seed=47)
    k16 = inp["k"].to(torch.float16)
    r = vector_gates((B, T, H, 128), 11, mean=4.0)
    box = dict(d_min=0.1, d_max=4.0)
    kt, d = osdn_precond_scan(k16.cuda(), inp["beta"].cuda(), r.cuda(), None, kt_dtype=torch.float32,
                              eta=0.3, eps=w.eps, beta_aware=False, **box)
    torch.cuda.synchronize()
    kt_ref, d_ref = oracle.precond_scan(k16, inp["beta"], r, None, eta=0.3, eps=w.eps, beta_aware=False, **box)
    assert_rel(kt, kt_ref, 1e-5, what="k_tilde")
    assert_rel(d, d_ref, 1e-5, what="d")
