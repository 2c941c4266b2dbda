"""Comparison helpers shared by the GPU parity tests (tolerances as stated per test)."""
import numpy as np
import torch


def np64(x):
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def assert_rel(got, ref, rtol, floor=1e-30, what=""):
    """Elementwise |got - ref| <= rtol * |ref| + floor."""
    g, r = np64(got), np64(ref)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    err = np.abs(g - r)
    bad = err > rtol * np.abs(r) + floor
    if bad.any():
        i = np.unravel_index(np.argmax(err / (np.abs(r) + floor)), r.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements exceed rel {rtol}; "
                             f"worst at {i}: got {g[i]!r} ref {r[i]!r}")


def assert_maxabs(got, ref, atol, what=""):
    g, r = np64(got), np64(ref)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    err = np.abs(g - r)
    m = float(err.max()) if err.size else 0.0
    if m > atol:
        i = np.unravel_index(np.argmax(err), r.shape)
        raise AssertionError(f"{what}: max-abs error {m:.3e} > {atol:.1e} at {i}: got {g[i]!r} ref {r[i]!r}")
    return m


def to_dev(inp, device="cuda"):
    """Move a workloads.make_prefill dict to the GPU (None stays None)."""
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
