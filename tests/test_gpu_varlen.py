"""GPU parity of the packed variable-length layer forward (cu_seqlens): every sequence of a packed
batch must get what the fp64 oracle gives for that sequence alone ("OSDN: Improving Delta Rule
with Provable Online Preconditioning in Linear Attention", Algorithm 1 and Eqs. (2), (4), (7);
Appendix B.1 with a state gate), with its own initial and final states.  Bars as for the batched
call: k~ and d 1e-5 relative (plus the bf16 rounding of k~), o and S max-abs 2e-2 (bf16) or 1e-4
(fp32)."""
import numpy as np
import pytest
import torch

import oracle
from preconditioned_delta_rule_gb300 import binding, osdn_layer_fwd, osdn_layer_fwd_varlen
from preconditioned_delta_rule_gb300 import workloads as W
from tests._parity import assert_maxabs, assert_rel, np64

pytestmark = pytest.mark.gpu


def packed_problem(name, lengths, H, seed, apf=False, gated=False):
    w = W.WORKLOADS[name]
    total = int(sum(lengths))
    inp = W.make_prefill(w, B=1, H=H, T=max(total, 1), seed=seed)
    inp = {k: (v[0, :total].contiguous() if isinstance(v, torch.Tensor) and v.dim() >= 3 else v) for k, v in inp.items()}
    K, V = inp["k"].shape[-1], inp["v"].shape[-1]
    N = len(lengths)
    g = torch.Generator().manual_seed(seed + 1)
    inp["r"] = torch.sigmoid(2.0 + torch.randn(total, H, generator=g)) if apf else None
    inp["alpha"] = 0.7 + 0.3 * torch.rand(total, H, generator=g) if gated else None
    inp["d0"] = torch.rand(N, H, K, generator=g) * 1.5 + 0.5
    inp["S0"] = torch.randn(N, H, V, K, generator=g) * 0.05
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
    return w, inp, cu


def run_varlen(inp, cu, **kw):
    d = lambda x: None if x is None else x.cuda()
    out = osdn_layer_fwd_varlen(d(inp["q"]), d(inp["k"]), d(inp["v"]), d(inp["beta"]), cu.cuda(), r=d(inp["r"]),
                                alpha=d(inp["alpha"]), d0=d(inp["d0"]), S0=d(inp["S0"]), **kw)
    torch.cuda.synchronize()
    binding.osdn_check()
    return out


def check_against_oracle(w, inp, cu, out, tol, kt_ulp, eta):
    o, S, d, kt = out
    for n in range(len(cu) - 1):
        s, e = int(cu[n]), int(cu[n + 1])
        sl = lambda x: None if x is None else x[None, s:e]
        ref = oracle.osdn_forward(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["beta"]), sl(inp["r"]),
                                  inp["d0"][n:n + 1], inp["S0"][n:n + 1], alpha=sl(inp["alpha"]), eta=eta,
                                  d_min=w.d_min, d_max=w.d_max, eps=w.eps)
        assert_rel(d[n:n + 1], ref["d"], 1e-5, what=f"d of sequence {n}")
        assert_maxabs(S[n:n + 1], ref["S"], tol, what=f"S of sequence {n}")
        if e > s:
            assert_rel(kt[None, s:e], ref["k_tilde"], 1e-5 + kt_ulp, what=f"k_tilde of sequence {n}")
            assert_maxabs(o[None, s:e], ref["o"], tol, what=f"o of sequence {n}")


@pytest.mark.parametrize("lengths,apf,gated", [
    ([200, 64, 1, 0, 65, 128, 63, 300], False, False),  # ragged, empty, one-token and chunk-edge sequences
    ([130, 257, 64], True, False),                       # APF retention in phase 1
    ([190, 70, 256], False, True),                       # the gated variant
])
def test_varlen_bf16_against_oracle(lengths, apf, gated):
    w, inp, cu = packed_problem("layer_340m", lengths, 4, 71, apf=apf, gated=gated)
    out = run_varlen(inp, cu, eta=0.3, d_min=w.d_min, d_max=w.d_max, eps=w.eps)
    check_against_oracle(w, inp, cu, out, 2e-2, 2.0 ** -8, 0.3)


def test_varlen_fp32_against_oracle():
    w, inp, cu = packed_problem("tiny_f32", [100, 37, 0, 64], 2, 72)
    out = run_varlen(inp, cu, eta=0.2, d_min=w.d_min, d_max=w.d_max, eps=w.eps)
    check_against_oracle(w, inp, cu, out, 1e-4, 0.0, 0.2)


def test_varlen_equal_lengths_equal_the_batched_call():
    """All sequences of one multiple-of-64 length: the padded batch is the batched layer call."""
    w, inp, cu = packed_problem("layer_340m", [256, 256, 256], 4, 73)
    o, S, d, kt = run_varlen(inp, cu, eta=0.05)
    b = lambda x: x.reshape(3, 256, *x.shape[1:]).cuda()
    o2, S2, d2, kt2 = osdn_layer_fwd(b(inp["q"]), b(inp["k"]), b(inp["v"]), b(inp["beta"]), None,
                                     inp["d0"].cuda(), inp["S0"].cuda(), eta=0.05)
    torch.cuda.synchronize()
    assert torch.equal(kt.reshape(3, 256, 4, 128), kt2) and torch.equal(d, d2)
    assert torch.equal(o.reshape(3, 256, 4, 128), o2) and torch.equal(S, S2)


def test_varlen_rejects_a_sequence_longer_than_max_len():
    """The device checks every range: a sequence longer than max_len is skipped and reported."""
    w, inp, cu = packed_problem("layer_340m", [64, 100, 32], 2, 74)
    d = lambda x: x.cuda()
    osdn_layer_fwd_varlen(d(inp["q"]), d(inp["k"]), d(inp["v"]), d(inp["beta"]), cu.cuda(), max_len=64,
                          d0=d(inp["d0"]), S0=d(inp["S0"]), eta=0.05)
    with pytest.raises(binding.OsdnError, match="SHAPE"):
        binding.osdn_check()
    binding.osdn_check()  # the flag is cleared
