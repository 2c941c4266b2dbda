"""Failure detection without a GPU fault: a device-side bounded wait that runs out is reported.

The fused layer call's chunk-prep workers poll (bounded) for values that its phase-1 CTAs publish.
osdn_set_poll_limit(1) makes each of those waits give up after one poll, long before phase 1 has
published anything: the workers drain what they issued and exit, the call completes without a
CUDA error, and osdn_check must report OSDN_ERR_TIMEOUT.  With the default limit restored, the
next call on the same context must report OSDN_OK and match the oracle.  No wait is left
unbounded and nothing faults: the aborted call only leaves its outputs invalid.
"""
import pytest
import torch

import oracle
from preconditioned_delta_rule_gb300 import binding, chunk_osdn
from preconditioned_delta_rule_gb300 import workloads as W
from tests._parity import assert_maxabs, assert_rel, to_dev

pytestmark = pytest.mark.gpu

OSDN_ERR_TIMEOUT = 7


def _layer(g, w):
    return binding.osdn_layer_fwd(g["q"], g["k"], g["v"], g["beta"], g["r"], None, None, eta=w.eta,
                                  d_min=w.d_min, d_max=w.d_max, eps=w.eps, beta_aware=w.beta_aware)


def test_prep_poll_runs_out_and_is_reported():
    w = W.WORKLOADS["layer_340m"]
    inp = W.make_prefill(w, B=2, H=8, T=1024, seed=41)
    g = to_dev(inp)
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    B, T, H, K = g["k"].shape
    assert binding.osdn_layer_fwd_workspace_bytes(B, T, H, K, K, 64, g["k"].dtype) > 0 and B * H < n_sm, \
        "this shape must take the fused layer path"
    binding.osdn_check()  # nothing pending from earlier tests
    try:
        binding.osdn_set_poll_limit(1)
        _layer(g, w)
        torch.cuda.synchronize()  # the kernels ended normally: no CUDA error here
        with pytest.raises(binding.OsdnError) as exc:
            binding.osdn_check()
        assert exc.value.status == OSDN_ERR_TIMEOUT, str(exc.value)
    finally:
        binding.osdn_set_poll_limit(0)
    # the context is still usable and the flag was cleared: a normal call is exact again
    o, S, d, _ = _layer(g, w)
    binding.osdn_check()
    ref = oracle.osdn_forward(inp["q"], inp["k"], inp["v"], inp["beta"], inp["r"], eta=w.eta, d_min=w.d_min,
                              d_max=w.d_max, eps=w.eps, beta_aware=w.beta_aware)
    assert_maxabs(o, ref["o"], 2e-2, what="o after the timeout")
    assert_maxabs(S, ref["S"], 2e-2, what="S after the timeout")
    assert_rel(d, ref["d"], 1e-5, what="d after the timeout")
