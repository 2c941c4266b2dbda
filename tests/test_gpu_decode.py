"""GPU parity of osdn_decode_step against the fp64 oracle, and the decode-vs-chunk consistency
protocol of the pages' Appendix L (a token-by-token decode must agree with the chunk forward).
Bar: o and S max-abs 2e-2 (bf16 inputs), d within 1e-5 relative."""
import numpy as np
import pytest
import torch

import oracle
from preconditioned_delta_rule_gb300 import (osdn_chunk_fwd, osdn_decode_step,
                                             osdn_precond_scan)
from preconditioned_delta_rule_gb300 import workloads as W
from tests._parity import assert_maxabs, assert_rel, np64, to_dev

pytestmark = pytest.mark.gpu


def test_decode_full_size_all_heads_few_steps():
    w = W.DECODE
    steps = 4
    inp = W.make_decode_steps(w, steps, device="cuda")
    S, d = W.make_decode_state(w, device="cuda")
    S_ref, d_ref = np64(S), np64(d)
    for t in range(steps):
        o = osdn_decode_step(inp["q"][t], inp["k"][t], inp["v"][t], inp["beta"][t], S, d,
                             eta=w.eta, d_min=w.d_min, d_max=w.d_max, eps=w.eps)
        torch.cuda.synchronize()
        o_ref, S_ref, d_ref = oracle.decode_step(inp["q"][t], inp["k"][t], inp["v"][t],
                                                 inp["beta"][t], S_ref, d_ref, eta=w.eta,
                                                 d_min=w.d_min, d_max=w.d_max, eps=w.eps)
        assert_maxabs(o, o_ref, 2e-2, what=f"o step {t}")
    assert_maxabs(S, S_ref, 2e-2, what="S")
    assert_rel(d, d_ref, 1e-5, what="d")


def test_decode_full_length_sampled_heads():
    """All 1024 steps of the decode workload; the oracle follows 24 sampled (b, h) pairs."""
    w = W.DECODE
    steps = w.steps
    inp = W.make_decode_steps(w, steps, device="cuda")
    S, d = W.make_decode_state(w, device="cuda")
    g = np.random.Generator(np.random.PCG64(77))
    bs = g.choice(w.B, 24, replace=False)
    hs = g.integers(0, w.H, 24)
    sel = lambda x: x[bs, hs].unsqueeze(0)  # [1, 24, ...]
    S_ref, d_ref = np64(sel(S)), np64(sel(d))
    worst = 0.0
    for t in range(steps):
        o = osdn_decode_step(inp["q"][t], inp["k"][t], inp["v"][t], inp["beta"][t], S, d,
                             eta=w.eta, d_min=w.d_min, d_max=w.d_max, eps=w.eps)
        o_ref, S_ref, d_ref = oracle.decode_step(sel(inp["q"][t]), sel(inp["k"][t]),
                                                 sel(inp["v"][t]), sel(inp["beta"][t]), S_ref,
                                                 d_ref, eta=w.eta, d_min=w.d_min, d_max=w.d_max,
                                                 eps=w.eps)
        worst = max(worst, assert_maxabs(sel(o), o_ref, 2e-2, what=f"o step {t}"))
    torch.cuda.synchronize()
    assert_maxabs(sel(S), S_ref, 2e-2, what="S")
    assert_rel(sel(d), d_ref, 1e-5, what="d")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("K,V", [(128, 128), (64, 64), (64, 128)])
def test_decode_apf_scale_dtypes(dtype, K, V):
    g = torch.Generator().manual_seed(K + V)
    B, H = 3, 5
    q = torch.nn.functional.normalize(torch.randn(6, B, H, K, generator=g), dim=-1).to(dtype)
    k = torch.nn.functional.normalize(torch.randn(6, B, H, K, generator=g), dim=-1).to(dtype)
    v = torch.randn(6, B, H, V, generator=g).to(dtype)
    beta = torch.sigmoid(torch.randn(6, B, H, generator=g))
    r = torch.sigmoid(2 + torch.randn(6, B, H, generator=g))
    S = torch.randn(B, H, V, K, generator=g) * 0.05
    d = torch.rand(B, H, K, generator=g) * 1.5 + 0.5
    S_ref, d_ref = np64(S), np64(d)
    Sd, dd = S.cuda(), d.cuda()
    tol = 1e-4 if dtype == torch.float32 else 2e-2
    for t in range(6):
        o = osdn_decode_step(q[t].cuda(), k[t].cuda(), v[t].cuda(), beta[t].cuda(), Sd, dd,
                             r[t].cuda(), eta=0.3, scale=K ** -0.5)
        torch.cuda.synchronize()
        o_ref, S_ref, d_ref = oracle.decode_step(q[t], k[t], v[t], beta[t], S_ref, d_ref, r[t],
                                                 eta=0.3, scale=K ** -0.5)
        assert_maxabs(o, o_ref, tol, what="o")
    assert_maxabs(Sd, S_ref, tol, what="S")
    assert_rel(dd, d_ref, 1e-5, what="d")


def _prefill(inp, w, T):
    dev = to_dev(inp)
    sl = lambda x: x[:, :T].contiguous()
    kt, d = osdn_precond_scan(sl(dev["k"]), sl(dev["beta"]), None, None, eta=w.eta)
    o, S = osdn_chunk_fwd(sl(dev["q"]), sl(dev["k"]), kt, sl(dev["v"]), sl(dev["beta"]))
    return o, S, d


def test_decode_64_tokens_equals_chunk_forward():
    """The pages' consistency protocol (T = 64): a token-by-token decode from zero state and
    d = 1 against the chunk forward on the same 64 tokens."""
    w = W.WORKLOADS["layer_340m"]
    inp = W.make_prefill(w, B=2, H=4, T=64, seed=31)
    o_c, S_c, d_c = _prefill(inp, w, 64)
    dev = to_dev(inp)
    S = torch.zeros(2, 4, 128, 128, device="cuda")
    d = torch.ones(2, 4, 128, device="cuda")
    outs = []
    for t in range(64):
        outs.append(osdn_decode_step(dev["q"][:, t].contiguous(), dev["k"][:, t].contiguous(),
                                     dev["v"][:, t].contiguous(), dev["beta"][:, t].contiguous(),
                                     S, d, eta=w.eta))
    torch.cuda.synchronize()
    o_d = torch.stack(outs, 1)
    assert_maxabs(o_d, o_c, 2e-2, what="decode vs chunk o")
    assert_maxabs(S, S_c, 2e-2, what="decode vs chunk S")
    assert_rel(d, d_c, 1e-5, what="decode vs scan d")


def test_prefill_128_then_decode_equals_oracle_129():
    """Prefill 128 tokens (scan + chunk), then one decode token, against the oracle on 129."""
    w = W.WORKLOADS["layer_340m"]
    inp = W.make_prefill(w, B=2, H=4, T=129, seed=32)
    o_c, S, d = _prefill(inp, w, 128)
    dev = to_dev(inp)
    o_last = osdn_decode_step(dev["q"][:, 128].contiguous(), dev["k"][:, 128].contiguous(),
                              dev["v"][:, 128].contiguous(), dev["beta"][:, 128].contiguous(),
                              S, d, eta=w.eta)
    torch.cuda.synchronize()
    ref = oracle.osdn_forward(inp["q"], inp["k"], inp["v"], inp["beta"], eta=w.eta)
    assert_maxabs(o_c, ref["o"][:, :128], 2e-2, what="prefill o")
    assert_maxabs(o_last, ref["o"][:, 128], 2e-2, what="decode o")
    assert_maxabs(S, ref["S"], 2e-2, what="S")
    assert_rel(d, ref["d"], 1e-5, what="d")
