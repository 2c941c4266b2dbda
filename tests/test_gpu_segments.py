"""GPU parity of the segment-parallel state pass (few heads, long sequences) against the fp64
oracle.  With few heads the chunk forward cuts each head's chunks into segments: the first runs
from S0, each later one from a zero state beside transition slices that carry the product of the
chunk transitions (I - K~^T W) (the paper's Appendix A.2, Eq. (10), applied segment by segment);
the segment start states are chained afterwards and the later segments' outputs corrected.  The
result must equal the plain recurrence within the same bars as the unsegmented path (max-abs 2e-2
on o and S for 16-bit inputs)."""
import numpy as np
import pytest
import torch

import oracle
from preconditioned_delta_rule_gb300 import chunk_osdn, osdn_chunk_fwd, osdn_chunk_fwd_workspace_bytes
from preconditioned_delta_rule_gb300 import workloads as W
from tests._parity import assert_maxabs, to_dev

pytestmark = pytest.mark.gpu


def write_keys(inp, w, dtype):
    kt, _ = oracle.precond_scan(inp["k"], inp["beta"], inp["r"], None, eta=w.eta, d_min=w.d_min,
                                d_max=w.d_max, eps=w.eps, beta_aware=w.beta_aware)
    return torch.from_numpy(kt).to(torch.float32).to(dtype)


@pytest.mark.parametrize("B,H,T", [(1, 2, 2048), (1, 1, 4096), (1, 2, 3200), (2, 1, 2112)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_segmented_chunk_against_oracle(B, H, T, dtype):
    """Two to four segments (equal and ragged), a random start state and the 1/sqrt(K) scale."""
    w = W.WORKLOADS["longctx_unit"]
    inp = W.make_prefill(w, B=B, H=H, T=T, seed=61)
    need = osdn_chunk_fwd_workspace_bytes(B, T, H, 128, 128)
    plain = B * H * (T // 64) * 33280
    assert need > plain, "these shapes take the segmented pass"
    kt = write_keys(inp, w, dtype)
    S0 = torch.randn(B, H, 128, 128, generator=torch.Generator().manual_seed(62)) * 0.1
    cast = lambda t: t.to(dtype)
    q, k, v = cast(inp["q"]), cast(inp["k"]), cast(inp["v"])
    o, S = osdn_chunk_fwd(q.cuda(), k.cuda(), kt.cuda(), v.cuda(), inp["beta"].cuda(), S0.cuda(),
                          scale=128 ** -0.5)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.delta_phase2(q, k, kt, v, inp["beta"], S0, scale=128 ** -0.5)
    eo = assert_maxabs(o, o_ref, 2e-2, what="o")
    es = assert_maxabs(S, S_ref, 2e-2, what="S")
    print(f"B{B} H{H} T{T} {dtype}: max|o err| {eo:.3e} max|S err| {es:.3e}")


def test_segmented_matches_unsegmented_and_aliases():
    """A workspace of exactly the image size runs the unsegmented chain: both agree to the fp16
    operand rounding; the segmented pass may write S_out over S0."""
    w = W.WORKLOADS["longctx_unit"]
    B, H, T = 1, 2, 2048
    inp = W.make_prefill(w, B=B, H=H, T=T, seed=63)
    kt = write_keys(inp, w, torch.bfloat16).cuda()
    d = to_dev(inp)
    S0 = torch.randn(B, H, 128, 128, generator=torch.Generator().manual_seed(64)).cuda() * 0.1
    plain = torch.empty(B * H * (T // 64) * 33280, dtype=torch.uint8, device="cuda")
    o1, S1 = osdn_chunk_fwd(d["q"], d["k"], kt, d["v"], d["beta"], S0, workspace=plain)
    S_in = S0.clone()
    o2, S2 = osdn_chunk_fwd(d["q"], d["k"], kt, d["v"], d["beta"], S_in, S_out=S_in)
    torch.cuda.synchronize()
    assert S2.data_ptr() == S_in.data_ptr()
    # o is bf16 and the later segments' outputs are rounded twice (before and after their
    # correction): one unit of its last place (2^-7 relative) is allowed on top
    g, r = o2.double().cpu().numpy(), o1.double().cpu().numpy()
    assert np.all(np.abs(g - r) <= 5e-3 + 2.0 ** -7 * np.abs(r)), float(np.max(np.abs(g - r)))
    assert_maxabs(S2, S1, 5e-3, what="S segmented vs unsegmented")


def test_segmented_layer_against_oracle():
    """Both phases (the fused layer call) on a few-head sequence: the chain runs segmented."""
    w = W.WORKLOADS["longctx_unit"]
    inp = W.make_prefill(w, B=1, H=2, T=2048, seed=65)
    d = to_dev(inp)
    o, S, dd = chunk_osdn(d["q"], d["k"], d["v"], d["beta"], d["r"], eta=w.eta, d_min=w.d_min,
                          d_max=w.d_max, eps=w.eps)
    torch.cuda.synchronize()
    ref = oracle.osdn_forward(inp["q"], inp["k"], inp["v"], inp["beta"], inp["r"], eta=w.eta,
                              d_min=w.d_min, d_max=w.d_max, eps=w.eps)
    assert_maxabs(o, ref["o"], 2e-2, what="o")
    assert_maxabs(S, ref["S"], 2e-2, what="S")
    rel = np.abs(dd.double().cpu().numpy() - ref["d"]) / np.abs(ref["d"])
    assert float(rel.max()) <= 1e-5
