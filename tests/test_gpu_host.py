"""GPU parity of the layer forward on host buffers (osdn_layer_fwd_host): the sequence runs as
consecutive pieces, each copied in while the previous one computes, with (d, S) carried on the
device.  "OSDN: Improving Delta Rule with Provable Online Preconditioning in Linear Attention",
Algorithm 1 and Eqs. (2), (4), (7) carry only (d, S) across tokens, so every split must give the
fp64 oracle's result for the whole sequence.  Bars as for osdn_layer_fwd: d 1e-5 relative, o and S
max-abs 2e-2 (bf16) or 1e-4 (fp32).  One piece is exactly one osdn_layer_fwd call."""
import pytest
import torch

import oracle
from preconditioned_delta_rule_gb300 import osdn_layer_fwd, osdn_layer_fwd_host
from preconditioned_delta_rule_gb300 import workloads as W
from tests._parity import assert_maxabs, assert_rel

pytestmark = pytest.mark.gpu


def problem(name, B, H, T, seed, apf=False, gated=False, start=True):
    w = W.WORKLOADS[name]
    inp = W.make_prefill(w, B=B, H=H, T=T, seed=seed)
    K, V = inp["k"].shape[-1], inp["v"].shape[-1]
    g = torch.Generator().manual_seed(seed + 1)
    if not apf:
        inp["r"] = None
    inp["alpha"] = 0.7 + 0.3 * torch.rand(B, T, H, generator=g) if gated else None
    inp["d0"] = torch.rand(B, H, K, generator=g) * 1.5 + 0.5 if start else None
    inp["S0"] = torch.randn(B, H, V, K, generator=g) * 0.05 if start else None
    return w, inp


def pinned(inp):
    return {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def run_host(w, inp, segments, eta, pin=True):
    x = pinned(inp) if pin else inp
    return osdn_layer_fwd_host(x["q"], x["k"], x["v"], x["beta"], x["r"], x["d0"], x["S0"], alpha=x["alpha"],
                               segments=segments, eta=eta, d_min=w.d_min, d_max=w.d_max, eps=w.eps)


@pytest.mark.parametrize("name,B,H,T,segments,apf,gated", [
    ("layer_340m", 2, 4, 512, 4, False, False),       # bf16 tensor-core layer path, four pieces
    ("layer_340m", 2, 4, 512, 1, False, False),       # one piece: copy in, compute, copy out in turn
    ("layer_1p3b_apf", 1, 3, 384, 3, True, False),    # APF retention in phase 1, B = 1 (plain copies)
    ("layer_340m", 2, 3, 256, 2, False, True),        # gated phase 2
    ("tiny_f32", 2, 2, 256, 4, False, False),         # fp32, K = V = 64 (CUDA-core kernels)
])
def test_host_layer_against_oracle(name, B, H, T, segments, apf, gated):
    w, inp = problem(name, B, H, T, seed=81 + T + segments, apf=apf, gated=gated)
    eta = 0.3
    o, S, d = run_host(w, inp, segments, eta)
    assert not o.is_cuda and not S.is_cuda and not d.is_cuda
    ref = oracle.osdn_forward(inp["q"], inp["k"], inp["v"], inp["beta"], inp["r"], inp["d0"], inp["S0"],
                              alpha=inp["alpha"], eta=eta, d_min=w.d_min, d_max=w.d_max, eps=w.eps)
    tol = 1e-4 if inp["k"].dtype == torch.float32 else 2e-2
    assert_rel(d, ref["d"], 1e-5, what="d")
    assert_maxabs(o, ref["o"], tol, what="o")
    assert_maxabs(S, ref["S"], tol, what="S")


def test_one_piece_equals_the_device_call():
    """segments = 1 runs one osdn_layer_fwd on the copied inputs: bit-identical outputs."""
    w, inp = problem("layer_340m", 2, 4, 384, seed=90)
    o, S, d = run_host(w, inp, 1, 0.05)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    o2, S2, d2, _ = osdn_layer_fwd(dev["q"], dev["k"], dev["v"], dev["beta"], None, dev["d0"], dev["S0"], eta=0.05,
                                   d_min=w.d_min, d_max=w.d_max, eps=w.eps)
    torch.cuda.synchronize()
    assert torch.equal(o, o2.cpu()) and torch.equal(S, S2.cpu()) and torch.equal(d, d2.cpu())


def test_pageable_buffers_and_default_start_state():
    """Pageable host memory gives the pinned result; NULL d0 / S0 mean ones / zeros."""
    w, inp = problem("layer_340m", 1, 4, 256, seed=91, start=False)
    a = run_host(w, inp, 2, 0.05, pin=True)
    b = run_host(w, inp, 2, 0.05, pin=False)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    ref = oracle.osdn_forward(inp["q"], inp["k"], inp["v"], inp["beta"], eta=0.05, d_min=w.d_min, d_max=w.d_max,
                              eps=w.eps)
    assert_rel(a[2], ref["d"], 1e-5, what="d")
    assert_maxabs(a[0], ref["o"], 2e-2, what="o")


def test_no_tokens_returns_the_start_state():
    w, inp = problem("layer_340m", 2, 2, 64, seed=92)
    sl = lambda x: x[:, :0].contiguous()
    o, S, d = osdn_layer_fwd_host(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["beta"]), None, inp["d0"],
                                  inp["S0"], segments=1)
    assert o.shape[1] == 0
    assert torch.equal(S, inp["S0"]) and torch.equal(d, inp["d0"])


@pytest.mark.parametrize("name,segments", [("layer_340m", 4), ("layer_1p3b_apf", 4)])
def test_host_layer_full_size(name, segments):
    """The host-buffer call as the bench times it (full workload, seeded inputs, pinned buffers)
    against the oracle's forward."""
    w = W.WORKLOADS[name]
    inp = W.make_prefill(w)
    x = pinned(inp)
    o, S, d = osdn_layer_fwd_host(x["q"], x["k"], x["v"], x["beta"], x["r"], segments=segments, eta=w.eta,
                                  d_min=w.d_min, d_max=w.d_max, eps=w.eps)
    ref = oracle.osdn_forward(inp["q"], inp["k"], inp["v"], inp["beta"], inp["r"], eta=w.eta, d_min=w.d_min,
                              d_max=w.d_max, eps=w.eps)
    assert_rel(d, ref["d"], 1e-5, what=f"{name} d")
    assert_maxabs(o, ref["o"], 2e-2, what=f"{name} o")
    assert_maxabs(S, ref["S"], 2e-2, what=f"{name} S")
