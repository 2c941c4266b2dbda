"""GPU parity of the layer backward (osdn_layer_bwd) against the fp64 oracle backward (reverse-mode
differentiation of the token loop of "OSDN: Improving Delta Rule with Provable Online
Preconditioning in Linear Attention", pinned by finite differences): every gradient (q, k, v,
beta, r, d0, S0) for a loss weighting o, S_T and d_T.  The GPU sweeps are fp32 over T tokens; each
gradient is compared as max-abs error against its own largest magnitude (bar stated below)."""
import numpy as np
import pytest
import torch

from oracle import backward as obw
from preconditioned_delta_rule_gb300 import osdn_layer_bwd
from preconditioned_delta_rule_gb300 import workloads as W
from tests._parity import np64

pytestmark = pytest.mark.gpu

# max |gpu - ref| <= REL * max |ref| for every gradient: fp32 sweeps over a few hundred tokens
# measured 2e-7 .. 7e-7 on GB300; the bar leaves a factor of ~30
REL = 2e-5


def check(name, got, ref):
    g, r = np64(got), np64(ref)
    assert g.shape == r.shape, name
    assert np.all(np.isfinite(g)), name
    scale = max(float(np.abs(r).max()), 1e-12)
    err = float(np.abs(g - r).max())
    assert err <= REL * scale, f"{name}: max-abs error {err:.3e} > {REL} x {scale:.3e}"
    return err / scale


def problem(name, B, H, T, seed, r_mode=0):
    w = W.WORKLOADS[name]
    inp = W.make_prefill(w, B=B, H=H, T=T, seed=seed)
    K, V = inp["k"].shape[-1], inp["v"].shape[-1]
    g = torch.Generator().manual_seed(seed + 7)
    r = None
    if r_mode == 1:
        r = torch.sigmoid(3.0 + torch.randn(B, T, H, generator=g))
    elif r_mode == 2:
        r = torch.sigmoid(3.0 + torch.randn(B, T, H, K, generator=g))
    d0 = torch.rand(B, H, K, generator=g) * 1.2 + 0.6
    S0 = torch.randn(B, H, V, K, generator=g) * 0.1
    do = torch.randn(B, T, H, V, generator=g)
    dS = torch.randn(B, H, V, K, generator=g) * 0.1
    dd = torch.randn(B, H, K, generator=g)
    return w, inp, r, d0, S0, do, dS, dd


@pytest.mark.parametrize("name,B,H,T,r_mode,beta_aware", [
    ("layer_340m", 1, 2, 200, 0, True),     # bf16, K = V = 128, a ragged last chunk
    ("layer_340m", 2, 1, 128, 1, False),    # per-head retention, non-beta-aware phase 1
    ("tiny_f32", 1, 2, 150, 2, True),       # fp32, K = V = 64, one retention per coordinate
])
def test_layer_bwd_against_oracle(name, B, H, T, r_mode, beta_aware):
    w, inp, r, d0, S0, do, dS, dd = problem(name, B, H, T, 91, r_mode)
    kw = dict(eta=0.3, d_min=w.d_min, d_max=w.d_max, eps=w.eps, beta_aware=beta_aware, scale=0.8)
    c = lambda x: None if x is None else x.cuda()
    got = osdn_layer_bwd(c(inp["q"]), c(inp["k"]), c(inp["v"]), c(inp["beta"]), c(do), c(r), c(d0), c(S0),
                         dS=c(dS), dd=c(dd), **kw)
    torch.cuda.synchronize()
    ref = obw.layer_backward(inp["q"], inp["k"], inp["v"], inp["beta"], r, d0, S0, do=do, dS=dS, dd=dd, **kw)
    errs = {n: check(n, got[n], ref[n]) for n in ("dq", "dk", "dv", "dbeta", "dd0", "dS0")}
    if r is not None:
        errs["dr"] = check("dr", got["dr"], ref["dr"])
    print(name, errs)


def test_layer_bwd_without_tokens_passes_the_state_gradients():
    B, H, K, V = 1, 2, 128, 128
    e = lambda *s: torch.zeros(*s, device="cuda")
    q = torch.zeros(B, 0, H, K, dtype=torch.bfloat16, device="cuda")
    dS = torch.randn(B, H, V, K, device="cuda")
    dd = torch.randn(B, H, K, device="cuda")
    got = osdn_layer_bwd(q, q, q, e(B, 0, H), e(B, 0, H, V), dS=dS, dd=dd)
    torch.cuda.synchronize()
    assert torch.equal(got["dS0"], dS) and torch.equal(got["dd0"], dd)
