"""GPU parity of the gated variant (OSGDN: "OSDN: Improving Delta Rule with Provable Online
Preconditioning in Linear Attention", Appendix B.1, Eqs. (13)-(15)): phase 2 with a per-token,
per-head state gate alpha in the post-gate residual form, against the fp64 oracle; phase 1 is
unchanged.  Bars as for the ungated rule: o and S max-abs 2e-2 (bf16) or 1e-4 (fp32), d 1e-5
relative.  A gate of ones must give exactly the ungated result on the same kernel."""
import numpy as np
import pytest
import torch

import oracle
from preconditioned_delta_rule_gb300 import osdn_chunk_fwd, osdn_decode_step, osdn_layer_fwd, osdn_precond_scan
from preconditioned_delta_rule_gb300 import workloads as W
from tests._parity import assert_maxabs, assert_rel, np64, to_dev

pytestmark = pytest.mark.gpu


def state_gates(shape, seed, lo=0.5):
    """Gates in [lo, 1): the decay range of Gated DeltaNet's per-token scalar gate."""
    g = torch.Generator().manual_seed(seed)
    return lo + (1.0 - lo) * torch.rand(*shape, generator=g)


@pytest.mark.parametrize("name,B,H,T", [
    ("layer_340m", 2, 4, 512),        # bf16, K = V = 128: 8 chunks
    ("layer_1p3b_apf", 1, 3, 384),    # bf16 with APF retention in phase 1
    ("tiny_f32", 1, 2, 256),          # fp32, K = V = 64
])
def test_gated_chunk_against_oracle(name, B, H, T):
    w = W.WORKLOADS[name]
    inp = W.make_prefill(w, B=B, H=H, T=T, seed=51)
    K, V = inp["k"].shape[-1], inp["v"].shape[-1]
    alpha = state_gates((B, T, H), 52)
    S0 = torch.randn(B, H, V, K, generator=torch.Generator().manual_seed(53)) * 0.1
    # the write keys come from the oracle's phase 1, rounded to the input dtype, for both sides
    kt_ref, _ = oracle.precond_scan(inp["k"], inp["beta"], inp["r"], None, eta=w.eta, d_min=w.d_min,
                                    d_max=w.d_max, eps=w.eps)
    kt = torch.from_numpy(kt_ref).to(inp["k"].dtype)
    dev = to_dev(inp)
    o, S = osdn_chunk_fwd(dev["q"], dev["k"], kt.cuda(), dev["v"], dev["beta"], S0.cuda(), alpha=alpha.cuda())
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.delta_phase2(inp["q"], inp["k"], kt, inp["v"], inp["beta"], S0, alpha=alpha)
    tol = 1e-4 if inp["k"].dtype == torch.float32 else 2e-2
    assert_maxabs(o, o_ref, tol, what="o")
    assert_maxabs(S, S_ref, tol, what="S")


@pytest.mark.parametrize("name,B,H,T", [("layer_340m", 2, 4, 640), ("longctx_unit", 1, 4, 1024)])
def test_gated_layer_against_oracle(name, B, H, T):
    w = W.WORKLOADS[name]
    inp = W.make_prefill(w, B=B, H=H, T=T, seed=54)
    alpha = state_gates((B, T, H), 55, lo=0.8)
    dev = to_dev(inp)
    o, S, d, kt = osdn_layer_fwd(dev["q"], dev["k"], dev["v"], dev["beta"], dev["r"], alpha=alpha.cuda(),
                                 eta=0.3, d_min=w.d_min, d_max=w.d_max, eps=w.eps)
    torch.cuda.synchronize()
    ref = oracle.osdn_forward(inp["q"], inp["k"], inp["v"], inp["beta"], inp["r"], alpha=alpha, eta=0.3,
                              d_min=w.d_min, d_max=w.d_max, eps=w.eps)
    assert_rel(d, ref["d"], 1e-5, what="d")
    assert_maxabs(o, ref["o"], 2e-2, what="o")
    assert_maxabs(S, ref["S"], 2e-2, what="S")


def test_gate_of_ones_is_the_ungated_rule():
    """fp32 inputs run one kernel for both: the gate multiplies by exactly 1."""
    w = W.WORKLOADS["tiny_f32"]
    inp = W.make_prefill(w, B=2, H=2, T=192, seed=56)
    dev = to_dev(inp)
    kt, _ = osdn_precond_scan(dev["k"], dev["beta"], None, None, eta=0.2)
    o1, S1 = osdn_chunk_fwd(dev["q"], dev["k"], kt, dev["v"], dev["beta"])
    o2, S2 = osdn_chunk_fwd(dev["q"], dev["k"], kt, dev["v"], dev["beta"], alpha=torch.ones_like(dev["beta"]))
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(S1, S2)


def test_zero_gate_forgets_the_state():
    """alpha_t = 0 at a chunk boundary: the output after it is the rule started from S = 0."""
    w = W.WORKLOADS["layer_340m"]
    B, H, T, t0 = 1, 2, 256, 128
    inp = W.make_prefill(w, B=B, H=H, T=T, seed=57)
    alpha = state_gates((B, T, H), 58, lo=0.7)
    alpha[:, t0] = 0.0
    dev = to_dev(inp)
    kt, _ = osdn_precond_scan(dev["k"], dev["beta"], None, None, kt_dtype=dev["k"].dtype, eta=w.eta)
    S0 = torch.randn(B, H, 128, 128, generator=torch.Generator().manual_seed(59)).cuda()
    o, S = osdn_chunk_fwd(dev["q"], dev["k"], kt, dev["v"], dev["beta"], S0, alpha=alpha.cuda())
    sl = lambda x: x[:, t0:].contiguous()
    o2, S2 = osdn_chunk_fwd(sl(dev["q"]), sl(dev["k"]), sl(kt), sl(dev["v"]), sl(dev["beta"]),
                            alpha=sl(alpha).cuda())
    torch.cuda.synchronize()
    assert_maxabs(o[:, t0:], np64(o2), 2e-2, what="o after the zero gate")
    assert_maxabs(S, np64(S2), 2e-2, what="S")


@pytest.mark.parametrize("dtype,K,V", [(torch.bfloat16, 128, 128), (torch.float32, 64, 128)])
def test_gated_decode_against_oracle(dtype, K, V):
    g = torch.Generator().manual_seed(K + V + 2)
    B, H, steps = 3, 5, 6
    q = torch.nn.functional.normalize(torch.randn(steps, B, H, K, generator=g), dim=-1).to(dtype)
    k = torch.nn.functional.normalize(torch.randn(steps, B, H, K, generator=g), dim=-1).to(dtype)
    v = torch.randn(steps, B, H, V, generator=g).to(dtype)
    beta = torch.sigmoid(torch.randn(steps, B, H, generator=g))
    alpha = state_gates((steps, B, H), K + V)
    S = torch.randn(B, H, V, K, generator=g) * 0.05
    d = torch.rand(B, H, K, generator=g) * 1.5 + 0.5
    S_ref, d_ref = np64(S), np64(d)
    Sd, dd = S.cuda(), d.cuda()
    tol = 1e-4 if dtype == torch.float32 else 2e-2
    for t in range(steps):
        o = osdn_decode_step(q[t].cuda(), k[t].cuda(), v[t].cuda(), beta[t].cuda(), Sd, dd,
                             alpha=alpha[t].cuda(), eta=0.3)
        torch.cuda.synchronize()
        o_ref, S_ref, d_ref = oracle.decode_step(q[t], k[t], v[t], beta[t], S_ref, d_ref, alpha=alpha[t],
                                                 eta=0.3)
        assert_maxabs(o, o_ref, tol, what=f"o step {t}")
    assert_maxabs(Sd, S_ref, tol, what="S")
    assert_rel(dd, d_ref, 1e-5, what="d")


def test_gated_decode_continues_the_gated_prefill():
    """Prefill T tokens with the chunk form, then one decode step: equals the prefill of T + 1."""
    w = W.WORKLOADS["layer_340m"]
    B, H, T = 2, 3, 256
    inp = W.make_prefill(w, B=B, H=H, T=T + 64, seed=60)
    alpha = state_gates((B, T + 64, H), 61, lo=0.8)
    dev = to_dev(inp)
    a = alpha.cuda()
    o, S, d, _ = osdn_layer_fwd(dev["q"][:, :T].contiguous(), dev["k"][:, :T].contiguous(),
                                dev["v"][:, :T].contiguous(), dev["beta"][:, :T].contiguous(),
                                alpha=a[:, :T].contiguous(), eta=0.3)
    o1 = osdn_decode_step(dev["q"][:, T].contiguous(), dev["k"][:, T].contiguous(), dev["v"][:, T].contiguous(),
                          dev["beta"][:, T].contiguous(), S, d, alpha=a[:, T].contiguous(), eta=0.3)
    torch.cuda.synchronize()
    ref = oracle.osdn_forward(inp["q"][:, :T + 1], inp["k"][:, :T + 1], inp["v"][:, :T + 1],
                              inp["beta"][:, :T + 1], alpha=alpha[:, :T + 1], eta=0.3)
    assert_maxabs(o1, ref["o"][:, T], 2e-2, what="decoded o")
    assert_maxabs(S, ref["S"], 2e-2, what="S after decode")
    assert np.isfinite(np64(o)).all()


@pytest.mark.parametrize("name,B,H,T", [("layer_340m", 2, 4, 512), ("layer_1p3b_apf", 1, 6, 640)])
def test_gated_layer_equals_two_calls(name, B, H, T):
    """The fused layer call (phase 1 and the gated chunk prep in one launch, then the gated chain)
    replays the same arithmetic as osdn_precond_scan then osdn_chunk_fwd: identical results."""
    w = W.WORKLOADS[name]
    inp = W.make_prefill(w, B=B, H=H, T=T, seed=62)
    alpha = state_gates((B, T, H), 63, lo=0.6).cuda()
    d = to_dev(inp)
    S0 = (torch.randn(B, H, 128, 128, generator=torch.Generator().manual_seed(64)) * 0.05).cuda()
    o, S, dd, kt = osdn_layer_fwd(d["q"], d["k"], d["v"], d["beta"], d["r"], None, S0, alpha=alpha, eta=0.05,
                                  d_min=w.d_min, d_max=w.d_max, eps=w.eps)
    kt2, dd2 = osdn_precond_scan(d["k"], d["beta"], d["r"], None, kt_dtype=d["k"].dtype, eta=0.05, d_min=w.d_min,
                                 d_max=w.d_max, eps=w.eps)
    o2, S2 = osdn_chunk_fwd(d["q"], d["k"], kt2, d["v"], d["beta"], S0, alpha=alpha)
    torch.cuda.synchronize()
    assert torch.equal(kt, kt2) and torch.equal(dd, dd2)
    assert torch.equal(o, o2), "o differs"
    assert torch.equal(S, S2), "S differs"
