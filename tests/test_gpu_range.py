"""Numeric range of the 16-bit tensor-core chunk path (fp16 operands, fp32 accumulation and state).

- Large but representable magnitudes (v ~ N(0, 1000^2), S0 ~ N(0, 10^2)) stay within the chunk tests'
  2e-2 bar, applied to the output's own scale (max-abs error <= 2e-2 x max|ref|: the rule is linear
  in (v, S0), so the unit-scale bar scales with them; bf16 rounding of o alone is ~4e-3 of it).
- Values that leave fp16's range (v ~ N(0, (1e5)^2): |v| > 65504) make osdn_check report
  OSDN_ERR_RANGE instead of passing silently, and the documented remedy -- the same call with fp32
  inputs (the fp32 CUDA-core path) -- matches the oracle.
- Keys whose elements sit below fp16's normal range (|k| ~ 1e-7 .. 1e-4) still meet the unit-scale
  bar (2e-2 max-abs).
"""
import pytest
import torch

import oracle
from preconditioned_delta_rule_gb300 import binding, osdn_chunk_fwd
from preconditioned_delta_rule_gb300 import workloads as W
from tests._parity import assert_maxabs, np64

pytestmark = pytest.mark.gpu

OSDN_ERR_RANGE = 9


def _case(v_scale=1.0, s0_scale=0.0, k_scale=None, T=1024, B=1, H=4, seed=51):
    w = W.WORKLOADS["layer_340m"]
    inp = W.make_prefill(w, B=B, H=H, T=T, seed=seed)
    k = inp["k"]
    if k_scale is not None:  # every other token's key scaled down (bf16 keeps the small values)
        sc = torch.ones(1, T, 1, 1)
        sc[:, 1::2] = k_scale
        k = (k.float() * sc).to(torch.bfloat16)
    v = (inp["v"].float() * v_scale).to(torch.bfloat16)
    kt, _ = oracle.precond_scan(k, inp["beta"], None, None, eta=w.eta, d_min=w.d_min, d_max=w.d_max, eps=w.eps)
    kt = torch.from_numpy(kt).float().to(torch.bfloat16)
    gen = torch.Generator().manual_seed(seed + 1)
    S0 = torch.randn(B, H, 128, 128, generator=gen) * s0_scale if s0_scale else None
    return inp["q"], k, kt, v, inp["beta"], S0


def _run(q, k, kt, v, beta, S0, dtype=torch.bfloat16):
    c = lambda t: t.to(dtype).cuda()
    o, S = osdn_chunk_fwd(c(q), c(k), c(kt), c(v), beta.cuda(), None if S0 is None else S0.cuda())
    torch.cuda.synchronize()
    return o, S


def test_large_magnitudes_within_scaled_bar():
    q, k, kt, v, beta, S0 = _case(v_scale=1000.0, s0_scale=10.0)
    o, S = _run(q, k, kt, v, beta, S0)
    binding.osdn_check()  # no range error
    o_ref, S_ref = oracle.delta_phase2(q, k, kt, v, beta, S0)
    assert_maxabs(o, o_ref, 2e-2 * float(abs(o_ref).max()), what="o (scaled bar)")
    assert_maxabs(S, S_ref, 2e-2 * float(abs(S_ref).max()), what="S (scaled bar)")


def test_out_of_range_values_are_reported_and_fp32_path_is_exact():
    q, k, kt, v, beta, S0 = _case(v_scale=1e5)
    assert float(v.float().abs().max()) > 65504.0
    _run(q, k, kt, v, beta, S0)
    with pytest.raises(binding.OsdnError) as exc:
        binding.osdn_check()
    assert exc.value.status == OSDN_ERR_RANGE, str(exc.value)
    binding.osdn_check()  # the flag was cleared
    # the documented remedy: the same call on fp32 inputs (CUDA-core kernel, fp32 throughout)
    o, S = _run(q, k, kt, v, beta, S0, dtype=torch.float32)
    binding.osdn_check()
    o_ref, S_ref = oracle.delta_phase2(q.float(), k.float(), kt.float(), v.float(), beta, S0)
    assert_maxabs(o, o_ref, 1e-4 * float(abs(o_ref).max()), what="o (fp32 path)")
    assert_maxabs(S, S_ref, 1e-4 * float(abs(S_ref).max()), what="S (fp32 path)")


@pytest.mark.parametrize("k_scale", [1e-3, 1e-6])
def test_keys_below_fp16_normal_range(k_scale):
    q, k, kt, v, beta, S0 = _case(k_scale=k_scale)
    small = float(abs(np64(k[:, 1::2])).max())
    assert small < (6.1e-5 if k_scale <= 1e-4 else 1e-3)  # all subnormal in fp16, or straddling
    o, S = _run(q, k, kt, v, beta, S0)
    binding.osdn_check()
    o_ref, S_ref = oracle.delta_phase2(q, k, kt, v, beta, S0)
    assert_maxabs(o, o_ref, 2e-2, what="o")
    assert_maxabs(S, S_ref, 2e-2, what="S")
