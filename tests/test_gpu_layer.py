"""GPU tests of osdn_layer_fwd: the fused path (phase 1 and the chunk prep in one cooperative
launch, prep workers forming the write keys from the published step sizes) must give exactly
what osdn_precond_scan followed by osdn_chunk_fwd give, since both replay the same arithmetic;
the fallback paths (no workspace, fp32 inputs, other head sizes) must too.  Parity with the
oracle at full sizes is in test_gpu_pipeline.py."""
import pytest
import torch

import oracle
from preconditioned_delta_rule_gb300 import (osdn_chunk_fwd, osdn_layer_fwd, osdn_layer_fwd_workspace_bytes,
                                             osdn_precond_scan)
from preconditioned_delta_rule_gb300 import workloads as W
from tests._parity import assert_maxabs, assert_rel, to_dev

pytestmark = pytest.mark.gpu


def two_calls(d, w, S0=None, d0=None, scale=1.0, eta=None):
    eta = w.eta if eta is None else eta
    kt, dd = osdn_precond_scan(d["k"], d["beta"], d["r"], d0, kt_dtype=d["k"].dtype, eta=eta, d_min=w.d_min,
                               d_max=w.d_max, eps=w.eps, beta_aware=w.beta_aware)
    o, S = osdn_chunk_fwd(d["q"], d["k"], kt, d["v"], d["beta"], S0, scale=scale)
    return o, S, dd, kt


@pytest.mark.parametrize("name,B,H,T,dtype", [
    ("layer_340m", 2, 4, 512, torch.bfloat16),
    ("layer_1p3b_apf", 2, 4, 640, torch.bfloat16),   # retention gates
    ("layer_340m", 1, 3, 256, torch.float16),
    ("longctx_unit", 1, 16, 1024, torch.bfloat16),  # 16 scan CTAs, many prep CTAs
])
def test_layer_equals_two_calls(name, B, H, T, dtype):
    w = W.WORKLOADS[name]
    inp = W.make_prefill(w, B=B, H=H, T=T, seed=31)
    d = to_dev(inp)
    if dtype != d["k"].dtype:
        for key in ("q", "k", "v"):
            d[key] = d[key].to(dtype)
    g = torch.Generator().manual_seed(3)
    S0 = (torch.randn(B, H, 128, 128, generator=g) * 0.05).cuda()
    d0 = (torch.rand(B, H, 128, generator=g) * 1.5 + 0.5).cuda()
    assert osdn_layer_fwd_workspace_bytes(B, T, H, 128, 128, 64, dtype) > 0
    for rep in range(2):  # the second call reuses the (now dirty) cached workspace
        o, S, dd, kt = osdn_layer_fwd(d["q"], d["k"], d["v"], d["beta"], d["r"], d0, S0, eta=0.05, d_min=w.d_min,
                                      d_max=w.d_max, eps=w.eps, scale=0.5, beta_aware=w.beta_aware)
        o2, S2, dd2, kt2 = two_calls(d, w, S0, d0, scale=0.5, eta=0.05)
        torch.cuda.synchronize()
        assert torch.equal(kt, kt2), f"k_tilde differs (call {rep})"
        assert torch.equal(dd, dd2), f"d differs (call {rep})"
        assert torch.equal(o, o2), f"o differs (call {rep})"
        assert torch.equal(S, S2), f"S differs (call {rep})"


def test_layer_without_workspace_and_against_oracle():
    w = W.WORKLOADS["layer_1p3b_apf"]
    inp = W.make_prefill(w, B=1, H=2, T=384, seed=5)
    d = to_dev(inp)
    o1, S1, d1, kt1 = osdn_layer_fwd(d["q"], d["k"], d["v"], d["beta"], d["r"], eta=w.eta, d_min=w.d_min,
                                     d_max=w.d_max, eps=w.eps)
    o2, S2, d2, kt2 = osdn_layer_fwd(d["q"], d["k"], d["v"], d["beta"], d["r"], eta=w.eta, d_min=w.d_min,
                                     d_max=w.d_max, eps=w.eps, workspace=False)
    torch.cuda.synchronize()
    assert torch.equal(kt1, kt2) and torch.equal(d1, d2)
    # without a workspace phase 2 runs the fused single kernel: same products, other summation order
    assert_maxabs(S1, S2, 5e-3, what="S")
    ref = oracle.osdn_forward(inp["q"], inp["k"], inp["v"], inp["beta"], inp["r"], eta=w.eta, d_min=w.d_min,
                              d_max=w.d_max, eps=w.eps)
    assert_maxabs(o1, ref["o"], 2e-2, what="o")
    assert_maxabs(S1, ref["S"], 2e-2, what="S")
    assert_rel(d1, ref["d"], 1e-5, what="d")


@pytest.mark.parametrize("name,T", [("tiny_f32", 192), ("tiny_f32", 0)])
def test_layer_fallback_fp32_and_empty(name, T):
    """fp32 inputs with K = V = 64 take the two separate calls; T = 0 copies the initial state."""
    w = W.WORKLOADS[name]
    inp = W.make_prefill(w, B=2, H=2, T=max(T, 64), seed=8)
    inp = {k: (v[:, :T] if isinstance(v, torch.Tensor) and v.dim() >= 3 else v) for k, v in inp.items()}
    d = to_dev(inp)
    g = torch.Generator().manual_seed(4)
    S0 = (torch.randn(2, 2, 64, 64, generator=g) * 0.1).cuda()
    d0 = (torch.rand(2, 2, 64, generator=g) + 0.5).cuda()
    o, S, dd, kt = osdn_layer_fwd(d["q"], d["k"], d["v"], d["beta"], d["r"], d0, S0, eta=0.1)
    torch.cuda.synchronize()
    if T == 0:
        assert torch.equal(S, S0) and torch.equal(dd, d0)
        return
    o2, S2, dd2, kt2 = two_calls(d, w, S0, d0, eta=0.1)
    torch.cuda.synchronize()
    assert torch.equal(kt, kt2) and torch.equal(dd, dd2) and torch.equal(o, o2) and torch.equal(S, S2)


def test_chunk_calls_on_two_streams_get_separate_scratch():
    """Two chunk forwards queued on two streams may run at the same time: each stream gets its own
    cached workspace, so both give what they give one after the other."""
    w = W.WORKLOADS["layer_340m"]
    prob = []
    for seed in (71, 72):
        d = to_dev(W.make_prefill(w, B=2, H=4, T=512, seed=seed))
        kt, _ = osdn_precond_scan(d["k"], d["beta"], None, None, kt_dtype=d["k"].dtype, eta=w.eta)
        prob.append((d, kt))
    ref = [osdn_chunk_fwd(d["q"], d["k"], kt, d["v"], d["beta"]) for d, kt in prob]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    out = []
    for (d, kt), s in zip(prob, streams):
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            out.append(osdn_chunk_fwd(d["q"], d["k"], kt, d["v"], d["beta"], stream=s))
    torch.cuda.synchronize()
    for (o, S), (o2, S2) in zip(ref, out):
        assert torch.equal(o, o2) and torch.equal(S, S2)
