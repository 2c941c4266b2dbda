"""GPU tests of osdn_chunk_fwd_static_ws, the chunk forward for callers that cannot allocate
device memory when they call (an engine that plans all GPU memory once at start-up, or code that
cannot take an allocator call -- its latency, synchronisation or possible failure -- mid-step).

The entry point is called through the C ABI.  It runs the same kernels as osdn_chunk_fwd given a
workspace of the chunk images' size (the two-kernel path without the segment split), only on a
fixed scratch array, so its results must be bit-identical to that path on two calls in a row (the
array is shared by every call and keeps the previous call's contents);
one call is also checked against the oracle at the chunk tests' tolerance.  The capacity edge
(exactly 1008 chunk-heads accepted, 1009 refused) and a gated call are covered too.  This file is
collected last on purpose.
"""
import ctypes

import pytest
import torch

import oracle
from preconditioned_delta_rule_gb300 import binding, osdn_chunk_fwd, osdn_precond_scan
from preconditioned_delta_rule_gb300 import workloads as W
from tests._parity import assert_maxabs

pytestmark = pytest.mark.gpu

TOL = 2e-2          # max-abs on o and S for bf16 inputs, as in test_gpu_chunk.py
OSDN_ERR_ARG = 1
OSDN_ERR_CAPACITY = 8


def call_static(q, k, kt, v, beta, S0, o, S_out, scale=1.0, alpha=None, alpha_per_key=0):
    B, T, H, K = k.shape
    V = v.shape[-1]
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return binding.lib().osdn_chunk_fwd_static_ws(
        p(q), p(k), p(kt), p(v), binding._code(k.dtype), p(beta), p(alpha), int(alpha_per_key), p(S0), p(o),
        p(S_out), B, T, H, K, V, 64, float(scale), stream)


def _inputs(B, H, T, seed):
    w = W.WORKLOADS["layer_1p3b_apf"]
    inp = W.make_prefill(w, B=B, H=H, T=T, seed=seed)
    g = {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in inp.items()}
    kt, _ = osdn_precond_scan(g["k"], g["beta"], g["r"], None, eta=w.eta)
    return inp, g, kt


def _workspace_path(g, kt, S0, **kw):
    """osdn_chunk_fwd on a workspace of exactly the chunk images' size (B H (T / 64) x 33280 bytes):
    the two-kernel path the static scratch runs."""
    B, T, H, _ = g["k"].shape
    ws = torch.empty(B * H * (T // 64) * 33280, dtype=torch.uint8, device="cuda")
    return osdn_chunk_fwd(g["q"], g["k"], kt, g["v"], g["beta"], S0, workspace=ws, **kw)


def _run_static(g, kt, S0, scale=1.0, alpha=None, alpha_per_key=0, like=None):
    o = torch.full_like(like[0], float("nan"))
    S = torch.full_like(like[1], float("nan"))
    st = call_static(g["q"], g["k"], kt, g["v"], g["beta"], S0, o, S, scale=scale, alpha=alpha,
                     alpha_per_key=alpha_per_key)
    assert st == 0, binding.osdn_status_string(st)
    torch.cuda.synchronize()
    binding.osdn_check()
    return o, S


def test_static_scratch_matches_workspace_path_twice():
    inp, g, kt = _inputs(2, 4, 512, seed=17)
    S0 = torch.randn(2, 4, 128, 128, generator=torch.Generator().manual_seed(5)).cuda() * 0.1
    o_ref, S_ref = _workspace_path(g, kt, S0, scale=0.5)
    for call in range(2):
        o, S = _run_static(g, kt, S0, scale=0.5, like=(o_ref, S_ref))
        assert torch.equal(o, o_ref), f"o differs from the workspace path (call {call})"
        assert torch.equal(S, S_ref), f"S differs from the workspace path (call {call})"
        if call == 0:  # and the result itself against the oracle's token recurrence
            ko, ks = oracle.delta_phase2(inp["q"], inp["k"], kt.cpu(), inp["v"], inp["beta"], S0.cpu(), scale=0.5)
            assert_maxabs(o, ko, TOL, what="o vs oracle")
            assert_maxabs(S, ks, TOL, what="S vs oracle")


def test_static_scratch_gated_matches_workspace_path():
    """The gated chain reads the decay words the prep wrote into the scratch."""
    inp, g, kt = _inputs(1, 4, 256, seed=23)
    gen = torch.Generator().manual_seed(29)
    alpha = torch.sigmoid(4.0 + torch.randn(1, 256, 4, generator=gen)).cuda()
    o_ref, S_ref = _workspace_path(g, kt, None, alpha=alpha)
    for call in range(2):
        o, S = _run_static(g, kt, None, alpha=alpha, like=(o_ref, S_ref))
        assert torch.equal(o, o_ref), f"gated o differs (call {call})"
        assert torch.equal(S, S_ref), f"gated S differs (call {call})"


def test_static_scratch_exact_capacity():
    """B=1, H=16, T=4032: 16 x 63 = 1008 chunk-heads, the whole array; the last slots must hold
    correct results too."""
    inp, g, kt = _inputs(1, 16, 4032, seed=31)
    o_ref, S_ref = _workspace_path(g, kt, None)
    o, S = _run_static(g, kt, None, like=(o_ref, S_ref))
    assert torch.equal(o, o_ref) and torch.equal(S, S_ref)


def _zeros(B, T, H):
    e = lambda *s: torch.zeros(*s, dtype=torch.bfloat16, device="cuda")
    return e(B, T, H, 128), e(B, T, H, 128), e(B, T, H, 128), e(B, T, H, 128), torch.zeros(B, T, H, device="cuda")


def test_static_scratch_rejects_requests_over_capacity():
    """1009 chunk-heads need 1009 x 33280 B > 32 MiB: refused before any launch; argument errors
    are still reported as such on a shape that is over capacity."""
    B, T, H = 1, 64 * 1009, 1
    q, k, kt, v, beta = _zeros(B, T, H)
    o = torch.zeros_like(v)
    S = torch.zeros(B, H, 128, 128, device="cuda")
    assert call_static(q, k, kt, v, beta, None, o, S) == OSDN_ERR_CAPACITY
    assert call_static(q, k, kt, v, beta, None, o, S, scale=float("nan")) == OSDN_ERR_ARG
    assert "OSDN_ERR_CAPACITY" in binding.osdn_status_string(OSDN_ERR_CAPACITY)


def test_static_scratch_channel_gate_needs_no_scratch():
    """One gate per key channel runs the CUDA-core kernel here, which needs no scratch: never refused
    for capacity, and identical to osdn_chunk_fwd without a workspace (the same kernel; with the
    channel-gated workspace osdn_chunk_fwd takes the tensor-core path instead)."""
    B, T, H = 1, 64 * 1009, 1
    gen = torch.Generator().manual_seed(37)
    mk = lambda *s: (torch.randn(*s, generator=gen) * 0.1).to(torch.bfloat16).cuda()
    q, k, kt, v = mk(B, T, H, 128), mk(B, T, H, 128), mk(B, T, H, 128), mk(B, T, H, 128)
    beta = torch.sigmoid(torch.randn(B, T, H, generator=gen)).cuda()
    alpha = torch.sigmoid(4.0 + torch.randn(B, T, H, 128, generator=gen)).cuda()
    g = dict(q=q, k=k, v=v, beta=beta)
    o_ref, S_ref = osdn_chunk_fwd(q, k, kt, v, beta, None, alpha=alpha, workspace=False)  # one gate per channel
    o, S = _run_static(g, kt, None, alpha=alpha, alpha_per_key=1, like=(o_ref, S_ref))
    assert torch.equal(o, o_ref) and torch.equal(S, S_ref)
