"""GPU parity of osdn_precond_scan (phase 1: Algorithm 1 / Eq. (4), APF Eq. (7)) against the
fp64 oracle.  Bar: k~ (fp32 output) and d within 1e-5 relative, elementwise; a bf16 k~ output
within one bf16 rounding (2^-8 relative) of the exact value."""
import numpy as np
import pytest
import torch

import oracle
from preconditioned_delta_rule_gb300 import binding, osdn_precond_scan
from preconditioned_delta_rule_gb300 import workloads as W
from tests._parity import assert_rel, np64, to_dev

pytestmark = pytest.mark.gpu


def run_both(inp, w, kt_dtype=torch.float32, d0=None, eta=None, d_min=None, d_max=None,
             beta_aware=None):
    eta = w.eta if eta is None else eta
    d_min = w.d_min if d_min is None else d_min
    d_max = w.d_max if d_max is None else d_max
    beta_aware = w.beta_aware if beta_aware is None else beta_aware
    dev = to_dev(inp)
    d0_dev = None if d0 is None else d0.cuda()
    kt, d = osdn_precond_scan(dev["k"], dev["beta"], dev["r"], d0_dev, kt_dtype=kt_dtype, eta=eta,
                              d_min=d_min, d_max=d_max, eps=w.eps, beta_aware=beta_aware)
    torch.cuda.synchronize()
    kt_ref, d_ref = oracle.precond_scan(inp["k"], inp["beta"], inp["r"], d0, eta=eta, d_min=d_min,
                                        d_max=d_max, eps=w.eps, beta_aware=beta_aware)
    return kt, d, kt_ref, d_ref


@pytest.mark.parametrize("name", ["tiny_f32", "layer_340m", "layer_1p3b_apf", "longctx_raw"])
def test_scan_workloads_full_size(name):
    w = W.WORKLOADS[name]
    inp = W.make_prefill(w)
    kt, d, kt_ref, d_ref = run_both(inp, w)
    assert_rel(kt, kt_ref, 1e-5, what=f"{name} k_tilde")
    assert_rel(d, d_ref, 1e-5, what=f"{name} d")


@pytest.mark.parametrize("beta_aware", [True, False])
def test_scan_interior_and_both_faces(beta_aware):
    """eta = 0.3 moves d through the interior of the box and onto both faces."""
    w = W.WORKLOADS["layer_340m"]
    inp = W.make_prefill(w, B=2, H=4, T=1024, seed=11)
    head_scale = torch.tensor([0.2, 0.5, 1.5, 3.0]).view(1, 1, 4, 1)  # short keys push d up, long down
    inp["k"] = (inp["k"].float() * head_scale).to(inp["k"].dtype)
    g = torch.Generator().manual_seed(5)
    d0 = torch.rand(2, 4, 128, generator=g) * 1.5 + 0.5
    kt, d, kt_ref, d_ref = run_both(inp, w, d0=d0, eta=0.3, beta_aware=beta_aware)
    assert_rel(kt, kt_ref, 1e-5, what="k_tilde")
    assert_rel(d, d_ref, 1e-5, what="d")
    traj = np64(kt_ref) / np64(inp["k"])  # every d_t, read back through the write keys
    traj = traj[np.isfinite(traj)]
    assert (traj == 0.5).any() and (traj == 2.0).any() and ((traj > 0.5) & (traj < 2.0)).any()


@pytest.mark.parametrize("kt_dtype", [torch.bfloat16, torch.float16])
def test_scan_half_precision_write_keys(kt_dtype):
    w = W.WORKLOADS["layer_1p3b_apf"]
    inp = W.make_prefill(w, B=1, H=4, T=512)
    kt, d, kt_ref, d_ref = run_both(inp, w, kt_dtype=kt_dtype)
    assert kt.dtype == kt_dtype
    ulp = 2.0 ** -8 if kt_dtype == torch.bfloat16 else 2.0 ** -11
    assert_rel(kt, kt_ref, ulp + 1e-5, floor=1e-7 if kt_dtype == torch.float16 else 1e-30,
               what="k_tilde half")
    assert_rel(d, d_ref, 1e-5, what="d")


def test_scan_no_box_and_eta_zero():
    w = W.WORKLOADS["layer_340m"]
    inp = W.make_prefill(w, B=1, H=2, T=256)
    kt, d, kt_ref, d_ref = run_both(inp, w, eta=0.0)
    assert torch.equal(kt.cpu(), inp["k"].float())  # d = 1 throughout: k~ = k exactly
    assert torch.all(d == 1.0)
    kt, d, kt_ref, d_ref = run_both(inp, w, eta=0.05, d_min=-np.inf, d_max=np.inf)
    assert_rel(kt, kt_ref, 1e-5, what="k_tilde no box")
    assert_rel(d, d_ref, 1e-5, what="d no box")


@pytest.mark.parametrize("T", [0, 1, 31, 33, 200])
def test_scan_ragged_lengths(T):
    w = W.WORKLOADS["tiny_f32"]
    inp = W.make_prefill(w, B=2, H=3, T=max(T, 1), seed=9)
    inp = {k: (v[:, :T] if isinstance(v, torch.Tensor) and v.dim() >= 3 else v) for k, v in inp.items()}
    d0 = torch.rand(2, 3, 64, generator=torch.Generator().manual_seed(1)) + 0.5
    kt, d, kt_ref, d_ref = run_both(inp, w, d0=d0, eta=0.2)
    if T:
        assert_rel(kt, kt_ref, 1e-5, what="k_tilde")
    assert_rel(d, d_ref, 1e-5, what="d")


def test_scan_d_out_aliases_d0():
    w = W.WORKLOADS["layer_340m"]
    inp = W.make_prefill(w, B=1, H=2, T=128)
    d0 = torch.rand(1, 2, 128, generator=torch.Generator().manual_seed(2)) + 0.5
    d_dev = d0.clone().cuda()
    dev = to_dev(inp)
    osdn_precond_scan(dev["k"], dev["beta"], None, d_dev, d_out=d_dev, kt_dtype=torch.float32,
                      eta=0.1)
    torch.cuda.synchronize()
    _, d_ref = oracle.precond_scan(inp["k"], inp["beta"], None, d0, eta=0.1)
    assert_rel(d_dev, d_ref, 1e-5, what="aliased d")


@pytest.mark.parametrize("name,T,eta,kt_dtype", [
    ("layer_1p3b_apf", 1000, None, torch.bfloat16),    # APF retention, ragged last block
    ("layer_340m", 512, 0.3, torch.float32),           # interior and both faces of the box
    ("layer_340m", 64, None, torch.float16),
])
def test_scan_parallel_emission_matches_in_kernel_emission(name, T, eta, kt_dtype):
    """With a workspace the write keys come from the parallel emission kernel; without one the
    scan kernel writes them.  Both replay the same recurrence from the same states: bit-identical."""
    w = W.WORKLOADS[name]
    inp = W.make_prefill(w, B=2, H=4, T=T, seed=23)
    dev = to_dev(inp)
    kw = dict(kt_dtype=kt_dtype, eta=w.eta if eta is None else eta, d_min=w.d_min, d_max=w.d_max,
              eps=w.eps, beta_aware=w.beta_aware)
    kt0, d0 = osdn_precond_scan(dev["k"], dev["beta"], dev["r"], None, workspace=False, **kw)
    need = binding.osdn_precond_scan_workspace_bytes(2, T, 4, 128, dev["k"].dtype)
    assert need > 0
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")  # NaN garbage to start from
    kt1, d1 = osdn_precond_scan(dev["k"], dev["beta"], dev["r"], None, workspace=ws, **kw)
    kt2, d2 = osdn_precond_scan(dev["k"], dev["beta"], dev["r"], None, workspace=ws, **kw)
    torch.cuda.synchronize()
    assert torch.equal(kt0, kt1) and torch.equal(kt1, kt2)
    assert torch.equal(d0, d1) and torch.equal(d1, d2)
    kt_ref, d_ref = oracle.precond_scan(inp["k"], inp["beta"], inp["r"], None, eta=kw["eta"],
                                        d_min=w.d_min, d_max=w.d_max, eps=w.eps,
                                        beta_aware=w.beta_aware)
    assert_rel(d1, d_ref, 1e-5, what="d")


@pytest.mark.parametrize("eta", [0.3, 1.0])
def test_scan_blocks_alternating_pinned_and_free(eta):
    """Head gates of 0.3 and 1 in turns of two blocks: d collapses onto d_min (every coordinate
    pinned: the block needs no Gram, so none is formed for the next one) and then leaves it (every
    coordinate free: the Gram the block needs was skipped, and it runs the clipped sweeps until no
    step size moves).  Both ways, and the emission from the workspace, against the oracle."""
    w = W.WORKLOADS["layer_1p3b_apf"]
    B, H, T = 1, 2, 1024
    inp = W.make_prefill(w, B=B, H=H, T=T, seed=46)
    t = np.arange(T)
    r = torch.from_numpy(np.where((t // 128) % 2 == 0, 0.3, 1.0)[None, :, None].repeat(H, 2)).float().contiguous()
    dev = to_dev(inp)
    kw = dict(kt_dtype=torch.float32, eta=eta, d_min=w.d_min, d_max=w.d_max, eps=w.eps)
    kt0, d0 = osdn_precond_scan(dev["k"], dev["beta"], r.cuda(), None, workspace=False, **kw)
    kt1, d1 = osdn_precond_scan(dev["k"], dev["beta"], r.cuda(), None, **kw)
    torch.cuda.synchronize()
    assert torch.equal(kt0, kt1) and torch.equal(d0, d1)
    kt_ref, d_ref = oracle.precond_scan(inp["k"], inp["beta"], r, None, eta=eta, d_min=w.d_min, d_max=w.d_max,
                                        eps=w.eps)
    assert_rel(kt0, kt_ref, 1e-5, what="k_tilde")
    assert_rel(d0, d_ref, 1e-5, what="d")
