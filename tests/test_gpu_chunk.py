"""GPU parity of osdn_chunk_fwd (phase 2: Eqs. (2), (5), (8)-(11)) against the fp64 oracle's
token recurrence fed the SAME write keys.  Bar (from the method's stated tolerances): max-abs
2e-2 on o and final S for bf16/f16 inputs, 1e-4 for fp32 inputs."""
import numpy as np
import pytest
import torch

import oracle
from preconditioned_delta_rule_gb300 import osdn_chunk_fwd, osdn_chunk_fwd_workspace_bytes
from preconditioned_delta_rule_gb300 import workloads as W
from tests._parity import assert_maxabs, np64, to_dev

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2, torch.float16: 2e-2}


def write_keys(inp, w, dtype):
    """k~ from the oracle's phase 1, rounded to the storage dtype (identical on both sides)."""
    kt, _ = oracle.precond_scan(inp["k"], inp["beta"], inp["r"], None, eta=w.eta, d_min=w.d_min,
                                d_max=w.d_max, eps=w.eps, beta_aware=w.beta_aware)
    return torch.from_numpy(kt).to(torch.float32).to(dtype)


def check(inp, w, kt, S0=None, scale=1.0, dtype=None, alias=False, workspace=None):
    dtype = dtype or inp["k"].dtype
    cast = lambda t: t.to(dtype)
    q, k, v = cast(inp["q"]), cast(inp["k"]), cast(inp["v"])
    dev = dict(q=q.cuda(), k=k.cuda(), kt=kt.to(dtype).cuda(), v=v.cuda(), beta=inp["beta"].cuda())
    S0d = None if S0 is None else S0.clone().cuda()
    o, S = osdn_chunk_fwd(dev["q"], dev["k"], dev["kt"], dev["v"], dev["beta"], S0d,
                          S_out=S0d if alias else None, scale=scale, workspace=workspace)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.delta_phase2(q, k, kt.to(dtype), v, inp["beta"], S0, scale=scale)
    tol = TOL[dtype]
    eo = assert_maxabs(o, o_ref, tol, what="o")
    es = assert_maxabs(S, S_ref, tol, what="S")
    return eo, es


def test_chunk_tiny_f32():
    w = W.WORKLOADS["tiny_f32"]
    inp = W.make_prefill(w)
    check(inp, w, write_keys(inp, w, torch.float32))


@pytest.mark.parametrize("workspace", [None, False], ids=["two_kernel", "fused"])
@pytest.mark.parametrize("name", ["layer_340m", "layer_1p3b_apf", "longctx_unit"])
def test_chunk_workloads_full_size(name, workspace):
    w = W.WORKLOADS[name]
    inp = W.make_prefill(w)
    eo, es = check(inp, w, write_keys(inp, w, torch.bfloat16), workspace=workspace)
    print(f"{name} ({'fused' if workspace is False else 'two-kernel'}): "
          f"max|o err| {eo:.3e} max|S err| {es:.3e}")


def test_chunk_paths_agree_and_workspace_reuse():
    """The fused kernel and the two-kernel path compute the same products with different operand
    arrangements (the two-kernel chain forms T'V as hi(T')V + lo(T')V from an exact bf16 split and
    Q K~^T from the loaded bf16 tiles), so they agree to fp32 summation order, which can move an
    fp16-rounded operand by one unit; a reused (dirty) workspace and an explicitly passed one give
    identical results."""
    w = W.WORKLOADS["layer_1p3b_apf"]
    inp = W.make_prefill(w, B=2, H=3, T=512, seed=13)
    kt = write_keys(inp, w, torch.bfloat16).cuda()
    d = to_dev(inp)
    S0 = torch.randn(2, 3, 128, 128, generator=torch.Generator().manual_seed(7)).cuda() * 0.1
    o1, S1 = osdn_chunk_fwd(d["q"], d["k"], kt, d["v"], d["beta"], S0, workspace=False)
    need = osdn_chunk_fwd_workspace_bytes(2, 512, 3, 128, 128)
    assert need == 2 * 3 * 8 * 33280
    ws = torch.full((need + 4096,), 0xAB, dtype=torch.uint8, device="cuda")
    o2, S2 = osdn_chunk_fwd(d["q"], d["k"], kt, d["v"], d["beta"], S0, workspace=ws)
    o3, S3 = osdn_chunk_fwd(d["q"], d["k"], kt, d["v"], d["beta"], S0, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o2, o3) and torch.equal(S2, S3)
    # o is bf16: a one-unit flip of its last place (2^-7 relative) is allowed on top
    g, r = np64(o2), np64(o1)
    assert np.all(np.abs(g - r) <= 5e-3 + 2.0 ** -7 * np.abs(r)), float(np.max(np.abs(g - r)))
    assert_maxabs(S2, S1, 5e-3, what="S two-kernel vs fused")


@pytest.mark.parametrize("T", [64, 128, 448])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
def test_chunk_lengths_dtypes_state(T, dtype):
    w = W.WORKLOADS["layer_340m"]
    inp = W.make_prefill(w, B=2, H=3, T=T, seed=21)
    g = torch.Generator().manual_seed(3)
    S0 = torch.randn(2, 3, 128, 128, generator=g) * 0.1
    check(inp, w, write_keys(inp, w, dtype), S0=S0, scale=128 ** -0.5, dtype=dtype)


def test_chunk_state_alias_and_single_head():
    w = W.WORKLOADS["layer_340m"]
    inp = W.make_prefill(w, B=1, H=1, T=256, seed=4)
    S0 = torch.randn(1, 1, 128, 128, generator=torch.Generator().manual_seed(4)) * 0.1
    check(inp, w, write_keys(inp, w, torch.bfloat16), S0=S0, alias=True)


@pytest.mark.parametrize("K,V", [(64, 64), (64, 128), (128, 64)])
def test_chunk_other_head_dims(K, V):
    w = W.PrefillWorkload("hd", B=1, H=2, T=192, K=K, V=V, dtype="bf16", seed=8)
    inp = W.make_prefill(w)
    check(inp, w, write_keys(inp, w, torch.bfloat16))


def test_chunk_t_zero_copies_state():
    S0 = torch.randn(2, 2, 128, 128).cuda()
    e = torch.empty(2, 0, 2, 128, dtype=torch.bfloat16, device="cuda")
    beta = torch.empty(2, 0, 2, device="cuda")
    o, S = osdn_chunk_fwd(e, e, e, e, beta, S0)
    torch.cuda.synchronize()
    assert o.shape == (2, 0, 2, 128)
    assert torch.equal(S, S0)
    o, S = osdn_chunk_fwd(e, e, e, e, beta, None)
    torch.cuda.synchronize()
    assert torch.count_nonzero(S) == 0


def test_chunk_eta_zero_is_deltanet():
    """eta = 0, d = 1: the write key is the key itself and phase 2 is plain DeltaNet."""
    w = W.WORKLOADS["layer_340m"]
    inp = W.make_prefill(w, B=2, H=2, T=512, seed=6)
    check(inp, w, inp["k"].clone())
