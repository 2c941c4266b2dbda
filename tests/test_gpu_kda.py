"""GPU parity of one state gate per key channel (OSKDA: "OSDN: Improving Delta Rule with Provable
Online Preconditioning in Linear Attention", Appendix B.2; KDA's K x V state Diag(alpha_t)
S_{t-1}, stored here as its V x K transpose) against the fp64 oracle: the chunk call, the layer
call, packed variable-length sequences and the decode step.  Bars as for the ungated rule: o and S
max-abs 2e-2 (bf16) or 1e-4 (fp32), d 1e-5 relative."""
import numpy as np
import pytest
import torch

import oracle
from preconditioned_delta_rule_gb300 import (binding, osdn_chunk_fwd, osdn_decode_step, osdn_layer_fwd,
                                             osdn_layer_fwd_varlen, osdn_precond_scan)
from preconditioned_delta_rule_gb300 import workloads as W
from tests._parity import assert_maxabs, assert_rel, np64, to_dev

pytestmark = pytest.mark.gpu


def channel_gates(shape, seed, lo=0.6):
    g = torch.Generator().manual_seed(seed)
    return lo + (1.0 - lo) * torch.rand(*shape, generator=g)


@pytest.mark.parametrize("name,B,H,T", [("layer_340m", 1, 3, 256), ("tiny_f32", 2, 2, 128)])
def test_channel_gated_chunk_against_oracle(name, B, H, T):
    w = W.WORKLOADS[name]
    inp = W.make_prefill(w, B=B, H=H, T=T, seed=61)
    K, V = inp["k"].shape[-1], inp["v"].shape[-1]
    alpha = channel_gates((B, T, H, K), 62)
    S0 = torch.randn(B, H, V, K, generator=torch.Generator().manual_seed(63)) * 0.1
    kt_ref, _ = oracle.precond_scan(inp["k"], inp["beta"], None, None, eta=0.2)
    kt = torch.from_numpy(kt_ref).to(inp["k"].dtype)
    dev = to_dev(inp)
    o, S = osdn_chunk_fwd(dev["q"], dev["k"], kt.cuda(), dev["v"], dev["beta"], S0.cuda(), alpha=alpha.cuda())
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.delta_phase2(inp["q"], inp["k"], kt, inp["v"], inp["beta"], S0, alpha=alpha)
    tol = 1e-4 if w.dtype == "f32" else 2e-2
    assert_maxabs(o, o_ref, tol, what="o")
    assert_maxabs(S, S_ref, tol, what="S")


def test_channel_gated_layer_against_oracle():
    w = W.WORKLOADS["layer_1p3b_apf"]
    B, H, T = 1, 3, 192
    inp = W.make_prefill(w, B=B, H=H, T=T, seed=64)
    alpha = channel_gates((B, T, H, 128), 65, lo=0.8)
    dev = to_dev(inp)
    o, S, d, kt = osdn_layer_fwd(dev["q"], dev["k"], dev["v"], dev["beta"], dev["r"], alpha=alpha.cuda(), eta=0.3,
                                 d_min=w.d_min, d_max=w.d_max, eps=w.eps)
    torch.cuda.synchronize()
    ref = oracle.osdn_forward(inp["q"], inp["k"], inp["v"], inp["beta"], inp["r"], alpha=alpha, eta=0.3,
                              d_min=w.d_min, d_max=w.d_max, eps=w.eps)
    assert_rel(d, ref["d"], 1e-5, what="d")
    assert_maxabs(o, ref["o"], 2e-2, what="o")
    assert_maxabs(S, ref["S"], 2e-2, what="S")


def test_equal_channel_gates_are_the_head_gate():
    """fp32, K = 64: both layouts run the CUDA-core kernel; equal channels multiply by the same value."""
    w = W.WORKLOADS["tiny_f32"]
    inp = W.make_prefill(w, B=1, H=2, T=192, seed=66)
    dev = to_dev(inp)
    a = channel_gates((1, 192, 2), 67).cuda()
    kt, _ = osdn_precond_scan(dev["k"], dev["beta"], None, None, eta=0.2)
    o1, S1 = osdn_chunk_fwd(dev["q"], dev["k"], kt, dev["v"], dev["beta"], alpha=a)
    o2, S2 = osdn_chunk_fwd(dev["q"], dev["k"], kt, dev["v"], dev["beta"], alpha=a[..., None].expand(1, 192, 2, 64).contiguous())
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(S1, S2)


def test_channel_gated_varlen_against_oracle():
    w = W.WORKLOADS["layer_340m"]
    lengths = [70, 0, 130]
    total, H = sum(lengths), 2
    inp = W.make_prefill(w, B=1, H=H, T=total, seed=68)
    inp = {k: (v[0].contiguous() if isinstance(v, torch.Tensor) and v.dim() >= 3 else v) for k, v in inp.items()}
    alpha = channel_gates((total, H, 128), 69)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
    o, S, d, kt = osdn_layer_fwd_varlen(inp["q"].cuda(), inp["k"].cuda(), inp["v"].cuda(), inp["beta"].cuda(), cu.cuda(),
                                        alpha=alpha.cuda(), eta=0.2)
    torch.cuda.synchronize()
    binding.osdn_check()
    for n in range(len(lengths)):
        s, e = int(cu[n]), int(cu[n + 1])
        sl = lambda x: x[None, s:e]
        ref = oracle.osdn_forward(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["beta"]), alpha=sl(alpha), eta=0.2)
        assert_maxabs(S[n:n + 1], ref["S"], 2e-2, what=f"S of sequence {n}")
        if e > s:
            assert_maxabs(o[None, s:e], ref["o"], 2e-2, what=f"o of sequence {n}")


@pytest.mark.parametrize("dtype,K,V", [(torch.bfloat16, 128, 128), (torch.float32, 64, 128)])
def test_channel_gated_decode_against_oracle(dtype, K, V):
    g = torch.Generator().manual_seed(K + V + 3)
    B, H, steps = 3, 4, 5
    q = torch.nn.functional.normalize(torch.randn(steps, B, H, K, generator=g), dim=-1).to(dtype)
    k = torch.nn.functional.normalize(torch.randn(steps, B, H, K, generator=g), dim=-1).to(dtype)
    v = torch.randn(steps, B, H, V, generator=g).to(dtype)
    beta = torch.sigmoid(torch.randn(steps, B, H, generator=g))
    alpha = channel_gates((steps, B, H, K), K + V)
    S = torch.randn(B, H, V, K, generator=g) * 0.05
    d = torch.rand(B, H, K, generator=g) * 1.5 + 0.5
    S_ref, d_ref = np64(S), np64(d)
    Sd, dd = S.cuda(), d.cuda()
    tol = 1e-4 if dtype == torch.float32 else 2e-2
    for t in range(steps):
        o = osdn_decode_step(q[t].cuda(), k[t].cuda(), v[t].cuda(), beta[t].cuda(), Sd, dd, alpha=alpha[t].cuda(), eta=0.3)
        torch.cuda.synchronize()
        o_ref, S_ref, d_ref = oracle.decode_step(q[t], k[t], v[t], beta[t], S_ref, d_ref, alpha=alpha[t], eta=0.3)
        assert_maxabs(o, o_ref, tol, what=f"o step {t}")
    assert_maxabs(Sd, S_ref, tol, what="S")
    assert_rel(dd, d_ref, 1e-5, what="d")


# ---- the tensor-core path for one gate per key channel (a workspace of the channel-gated size) ----

def bench_like_gates(shape, seed):
    """sigmoid(4 + N(0, 1)) per token, head and channel: the bench's channel-gated leg."""
    g = torch.Generator().manual_seed(seed)
    return torch.sigmoid(4.0 + torch.randn(*shape, generator=g))


@pytest.mark.parametrize("gates", ["bench", "harsh"])
def test_channel_gated_tensor_core_full_size(gates):
    """The 340M-shaped layer (B8 H8 T2048) on the tensor-core path against the fp64 oracle: the
    bench's gates, and gates uniform in [0.6, 1] whose decay over a chunk reaches ~1e-7 (K~ / Gamma
    far beyond fp16's range, carried by the split-bf16 products)."""
    w = W.WORKLOADS["layer_340m"]
    inp = W.make_prefill(w, seed=71)
    B, T, H, K = inp["k"].shape
    V = inp["v"].shape[-1]
    alpha = bench_like_gates((B, T, H, K), 72) if gates == "bench" else channel_gates((B, T, H, K), 72)
    S0 = torch.randn(B, H, V, K, generator=torch.Generator().manual_seed(73)) * 0.1
    kt_ref, _ = oracle.precond_scan(inp["k"], inp["beta"], None, None, eta=w.eta)
    kt = torch.from_numpy(kt_ref).to(inp["k"].dtype)
    need = binding.osdn_chunk_fwd_workspace_bytes(B, T, H, K, V, 64, inp["k"].dtype, gated=2)
    assert need == B * H * (T // 64) * 66048
    dev = to_dev(inp)
    o, S = osdn_chunk_fwd(dev["q"], dev["k"], kt.cuda(), dev["v"], dev["beta"], S0.cuda(), alpha=alpha.cuda())
    torch.cuda.synchronize()
    binding.osdn_check()
    o_ref, S_ref = oracle.delta_phase2(inp["q"], inp["k"], kt, inp["v"], inp["beta"], S0, alpha=alpha)
    eo = assert_maxabs(o, o_ref, 2e-2, what="o")
    es = assert_maxabs(S, S_ref, 2e-2, what="S")
    print(f"{gates} gates: max|o err| {eo:.3e} max|S err| {es:.3e}")


def test_channel_gated_tensor_core_matches_cuda_core_path():
    """A workspace of the ungated size runs the fp32 CUDA-core kernel; the tensor-core path agrees
    with it within the 16-bit bar, and a dirty reused workspace gives identical results."""
    w = W.WORKLOADS["layer_1p3b_apf"]
    B, H, T = 2, 3, 512
    inp = W.make_prefill(w, B=B, H=H, T=T, seed=74)
    alpha = channel_gates((B, T, H, 128), 75, lo=0.8).cuda()
    dev = to_dev(inp)
    kt, _ = osdn_precond_scan(dev["k"], dev["beta"], dev["r"], None, eta=w.eta)
    small = torch.empty(binding.osdn_chunk_fwd_workspace_bytes(B, T, H, 128, 128), dtype=torch.uint8, device="cuda")
    o1, S1 = osdn_chunk_fwd(dev["q"], dev["k"], kt, dev["v"], dev["beta"], alpha=alpha, workspace=small)
    big = torch.full((binding.osdn_chunk_fwd_workspace_bytes(B, T, H, 128, 128, gated=2),), 0x7F, dtype=torch.uint8,
                     device="cuda")
    o2, S2 = osdn_chunk_fwd(dev["q"], dev["k"], kt, dev["v"], dev["beta"], alpha=alpha, workspace=big)
    o3, S3 = osdn_chunk_fwd(dev["q"], dev["k"], kt, dev["v"], dev["beta"], alpha=alpha, workspace=big)
    torch.cuda.synchronize()
    assert torch.equal(o2, o3) and torch.equal(S2, S3)
    assert_maxabs(o2, o1, 2e-2, what="o tensor-core vs CUDA-core")
    assert_maxabs(S2, S1, 2e-2, what="S tensor-core vs CUDA-core")
