"""End-to-end GPU parity of the layer forward (chunk_osdn -> osdn_layer_fwd: the fused phase-1 /
chunk-prep launch and the chain kernel for bf16 inputs, the two separate calls for fp32) against
the oracle's interleaved fp64 forward on the workloads' full sizes."""
import pytest
import torch

import oracle
from preconditioned_delta_rule_gb300 import chunk_osdn
from preconditioned_delta_rule_gb300 import workloads as W
from tests._parity import assert_maxabs, assert_rel, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny_f32", "layer_340m", "layer_1p3b_apf", "longctx_unit"])
def test_layer_forward_full_size(name):
    w = W.WORKLOADS[name]
    inp = W.make_prefill(w)
    dev = to_dev(inp)
    o, S, d = chunk_osdn(dev["q"], dev["k"], dev["v"], dev["beta"], dev["r"], eta=w.eta,
                         d_min=w.d_min, d_max=w.d_max, eps=w.eps)
    torch.cuda.synchronize()
    ref = oracle.osdn_forward(inp["q"], inp["k"], inp["v"], inp["beta"], inp["r"], eta=w.eta,
                              d_min=w.d_min, d_max=w.d_max, eps=w.eps)
    tol = 1e-4 if w.dtype == "f32" else 2e-2
    eo = assert_maxabs(o, ref["o"], tol, what=f"{name} o")
    es = assert_maxabs(S, ref["S"], tol, what=f"{name} S")
    assert_rel(d, ref["d"], 1e-5, what=f"{name} d")
    print(f"{name}: max|o err| {eo:.3e} max|S err| {es:.3e}")
