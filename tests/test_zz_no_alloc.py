"""GPU test of osdn_chunk_fwd_static_ws, the chunk forward for callers that cannot allocate
device memory when they call (an engine that plans all GPU memory once at start-up, or code that
cannot take an allocator call -- its latency, synchronisation or possible failure -- mid-step).

It is called through the C ABI and compared with osdn_chunk_fwd given a normal workspace, on two
calls in a row (the fixed scratch array is shared by every call and keeps the previous call's
contents), within the chunk tests' tolerance.  This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

from preconditioned_delta_rule_gb300 import binding, osdn_chunk_fwd, osdn_precond_scan
from preconditioned_delta_rule_gb300 import workloads as W
from tests._parity import assert_maxabs

pytestmark = pytest.mark.gpu

TOL = 2e-2          # max-abs on o and S for bf16 inputs, as in test_gpu_chunk.py
OSDN_ERR_CAPACITY = 8


def call_static(q, k, kt, v, beta, S0, o, S_out, scale=1.0):
    B, T, H, K = k.shape
    V = v.shape[-1]
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return binding.lib().osdn_chunk_fwd_static_ws(
        p(q), p(k), p(kt), p(v), binding._code(k.dtype), p(beta), None, 0, p(S0), p(o), p(S_out),
        B, T, H, K, V, 64, float(scale), stream)


def test_static_scratch_matches_workspace_path_twice():
    w = W.WORKLOADS["layer_1p3b_apf"]
    inp = W.make_prefill(w, B=2, H=4, T=512, seed=17)
    g = {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in inp.items()}
    kt, _ = osdn_precond_scan(g["k"], g["beta"], g["r"], None, eta=w.eta)
    S0 = torch.randn(2, 4, 128, 128, generator=torch.Generator().manual_seed(5)).cuda() * 0.1
    o_ref, S_ref = osdn_chunk_fwd(g["q"], g["k"], kt, g["v"], g["beta"], S0, scale=0.5)
    for call in range(2):
        o = torch.full_like(o_ref, float("nan"))
        S = torch.full_like(S_ref, float("nan"))
        st = call_static(g["q"], g["k"], kt, g["v"], g["beta"], S0, o, S, scale=0.5)
        assert st == 0, binding.osdn_status_string(st)
        torch.cuda.synchronize()
        binding.osdn_check()
        assert_maxabs(o, o_ref, TOL, what=f"o (call {call})")
        assert_maxabs(S, S_ref, TOL, what=f"S (call {call})")


def test_static_scratch_rejects_requests_over_capacity():
    """1037 chunk-heads need 1037 x 33280 B > 32 MiB: refused before any launch."""
    B, T, H = 1, 64 * 61, 17
    e = lambda *s: torch.zeros(*s, dtype=torch.bfloat16, device="cuda")
    q, k, kt, v = e(B, T, H, 128), e(B, T, H, 128), e(B, T, H, 128), e(B, T, H, 128)
    beta = torch.zeros(B, T, H, device="cuda")
    o = e(B, T, H, 128)
    S = torch.zeros(B, H, 128, 128, device="cuda")
    assert call_static(q, k, kt, v, beta, None, o, S) == OSDN_ERR_CAPACITY
    assert "OSDN_ERR_CAPACITY" in binding.osdn_status_string(OSDN_ERR_CAPACITY)
