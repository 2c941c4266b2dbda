"""Seeded synthetic inputs for the OSDN forward path (phase-1 scan, chunk forward, decode step).

This module holds none of the method's arithmetic: only random draws, per-token L2
normalisation, the logistic squashing that turns normal draws into gates in (0, 1), and
rounding to the storage dtype.  Both the CUDA path and the fp64 oracle consume exactly the
tensors produced here (the oracle takes them upcast to float64), so input rounding is never
counted as error.

Workloads follow the shapes of "OSDN: Improving Delta Rule with Provable Online
Preconditioning in Linear Attention" (arXiv:2605.13473): head dim 128 for both the
340M model (width 1024, 8 heads; Table 4) and the 1.3B model (width 2048, 16 heads; Table 5),
chunk 64 and eta = 0.003, D = [0.5, 2]^K (Appendix F), 20K-token PG-19 extrapolation blocks
(Section 6 / Table 13).  The datasets and trained checkpoints are not used: every tensor is
drawn from a seeded generator with the distribution stated per workload.

Draw order for a prefill workload (numpy ``Generator(PCG64(seed))``, float64 draws):
q, k, v, beta, r (APF only), then the tiny-norm token indices (long-context only).
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np
import torch


@dataclass(frozen=True)
class PrefillWorkload:
    """A layer-shaped prefill problem: B sequences, H heads, T tokens, head dims K and V."""

    name: str
    B: int
    H: int
    T: int
    K: int
    V: int
    dtype: str                 # storage dtype of q, k, v: "f32" or "bf16"
    key_mode: str = "unit"     # "unit" | "raw_tiny" | "unit_tiny"
    apf: bool = False          # draw a retention gate r_{t,h} = sigmoid(N(2, 1))
    seed: int = 0
    chunk: int = 64
    eta: float = 0.003
    d_min: float = 0.5
    d_max: float = 2.0
    eps: float = 1e-6
    beta_aware: bool = True
    key_std: float = 0.5       # std of raw keys in the long-context workload
    tiny_frac: float = 0.01    # fraction of tokens per (b, h) with near-zero key norm
    tiny_norm: float = 1e-4

    @property
    def tokens(self) -> int:
        return self.B * self.T

    @property
    def heads(self) -> int:
        return self.B * self.H


@dataclass(frozen=True)
class DecodeWorkload:
    """Recurrent single-token decode: B sequences x H heads, fp32 state S (V x K) and d."""

    name: str
    B: int
    H: int
    K: int
    V: int
    steps: int
    seed: int = 4
    dtype: str = "bf16"
    s_std: float = 0.01
    eta: float = 0.003
    d_min: float = 0.5
    d_max: float = 2.0
    eps: float = 1e-6
    beta_aware: bool = True


# The five workloads of the hot path.  The long-context one comes in two forms: the
# verbatim draw (raw keys with std 0.5, which make the delta-rule transition expanding and
# the phase-2 values overflow; used for phase-1 parity and for timing) and the same draw with
# the regular keys L2-normalised (used for o/S parity).
WORKLOADS = {
    "tiny_f32": PrefillWorkload("tiny_f32", B=1, H=2, T=256, K=64, V=64, dtype="f32", seed=0),
    "layer_340m": PrefillWorkload("layer_340m", B=8, H=8, T=2048, K=128, V=128, dtype="bf16", seed=1),
    "layer_1p3b_apf": PrefillWorkload("layer_1p3b_apf", B=4, H=16, T=4096, K=128, V=128,
                                      dtype="bf16", apf=True, seed=2),
    "longctx_raw": PrefillWorkload("longctx_raw", B=1, H=16, T=20480, K=128, V=128, dtype="bf16",
                                   key_mode="raw_tiny", seed=3),
    "longctx_unit": PrefillWorkload("longctx_unit", B=1, H=16, T=20480, K=128, V=128, dtype="bf16",
                                    key_mode="unit_tiny", seed=3),
}
DECODE = DecodeWorkload("decode_b256_h16", B=256, H=16, K=128, V=128, steps=1024, seed=4)


def _torch_dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def _l2_normalise(x: np.ndarray) -> np.ndarray:
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
    return x / n


def _sigmoid(x: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-x))


def _round(x: np.ndarray, dtype: str) -> torch.Tensor:
    """float64 numpy -> torch tensor of the storage dtype (round to nearest even)."""
    t = torch.from_numpy(np.ascontiguousarray(x)).to(torch.float32)
    return t.to(_torch_dtype(dtype)) if dtype != "f32" else t


def make_prefill(w: PrefillWorkload, **overrides) -> dict:
    """Draw one prefill problem on the host.

    Returns a dict of CPU tensors: q, k, v [B,T,H,K|V] in ``w.dtype``; beta [B,T,H] fp32;
    r [B,T,H] fp32 or None; d0, S0 None (the workloads start from d = 1 and S = 0);
    ``tiny_idx`` the (b, h, t) positions whose key has norm ``tiny_norm`` (or None).
    ``overrides`` replace fields of the workload (for example a shorter T for a test).
    """
    if overrides:
        w = replace(w, **overrides)
    B, T, H, K, V = w.B, w.T, w.H, w.K, w.V
    rng = np.random.Generator(np.random.PCG64(w.seed))
    q = _l2_normalise(rng.standard_normal((B, T, H, K)))
    q_t = _round(q, w.dtype)
    del q
    k = rng.standard_normal((B, T, H, K))
    if w.key_mode == "raw_tiny":
        k *= w.key_std
    v = rng.standard_normal((B, T, H, V))
    v_t = _round(v, w.dtype)
    del v
    beta = _sigmoid(rng.standard_normal((B, T, H))).astype(np.float32)
    r = _sigmoid(2.0 + rng.standard_normal((B, T, H))).astype(np.float32) if w.apf else None
    tiny_idx = None
    if w.key_mode in ("raw_tiny", "unit_tiny"):
        n_tiny = max(1, int(round(T * w.tiny_frac)))
        picks = []
        for b in range(B):
            for h in range(H):
                picks.append(rng.choice(T, n_tiny, replace=False))
        if w.key_mode == "unit_tiny":
            k = _l2_normalise(k)
        tiny_idx = []
        i = 0
        for b in range(B):
            for h in range(H):
                ts = np.sort(picks[i])
                i += 1
                kk = k[b, ts, h, :]
                k[b, ts, h, :] = kk / np.sqrt(np.sum(kk * kk, axis=-1, keepdims=True)) * w.tiny_norm
                tiny_idx.extend((b, h, int(t)) for t in ts)
    elif w.key_mode == "unit":
        k = _l2_normalise(k)
    else:
        raise ValueError(f"unknown key_mode {w.key_mode!r}")
    k_t = _round(k, w.dtype)
    del k
    return {
        "q": q_t, "k": k_t, "v": v_t,
        "beta": torch.from_numpy(beta),
        "r": torch.from_numpy(r) if r is not None else None,
        "d0": None, "S0": None, "tiny_idx": tiny_idx, "workload": w,
    }


def make_random_state(B: int, H: int, K: int, V: int, seed: int, s_std: float = 0.01,
                      d_lo: float = 0.5, d_hi: float = 2.0):
    """Initial decode/continuation state: S ~ N(0, s_std^2) [B,H,V,K], d ~ U[d_lo, d_hi] [B,H,K]."""
    rng = np.random.Generator(np.random.PCG64([seed, 0xD5]))
    S = (rng.standard_normal((B, H, V, K)) * s_std).astype(np.float32)
    d = rng.uniform(d_lo, d_hi, size=(B, H, K)).astype(np.float32)
    return torch.from_numpy(S), torch.from_numpy(d)


def make_decode_steps(w: DecodeWorkload, steps: int, device="cpu", seed: Optional[int] = None) -> dict:
    """Per-step decode inputs for ``steps`` tokens, drawn with a seeded torch generator on
    ``device`` (the full decode workload is about 3 GB of bf16, so it is drawn where it is used).

    Returns q, k [steps,B,H,K] (unit norm), v [steps,B,H,V] in ``w.dtype`` and beta [steps,B,H]
    fp32 = sigmoid(N(0,1)).
    """
    g = torch.Generator(device=device)
    g.manual_seed(w.seed if seed is None else seed)
    dt = _torch_dtype(w.dtype)
    shape = (steps, w.B, w.H)
    out = {}
    q = torch.randn(*shape, w.K, generator=g, device=device, dtype=torch.float32)
    out["q"] = (q / q.norm(dim=-1, keepdim=True)).to(dt)
    del q
    k = torch.randn(*shape, w.K, generator=g, device=device, dtype=torch.float32)
    out["k"] = (k / k.norm(dim=-1, keepdim=True)).to(dt)
    del k
    out["v"] = torch.randn(*shape, w.V, generator=g, device=device, dtype=torch.float32).to(dt)
    out["beta"] = torch.sigmoid(torch.randn(*shape, generator=g, device=device, dtype=torch.float32))
    return out


def make_decode_state(w: DecodeWorkload, device="cpu", seed: Optional[int] = None):
    """Decode start state drawn on ``device``: S ~ N(0, s_std^2) [B,H,V,K], d ~ U[0.5, 2] [B,H,K]."""
    g = torch.Generator(device=device)
    g.manual_seed((w.seed if seed is None else seed) + 7919)
    S = torch.randn(w.B, w.H, w.V, w.K, generator=g, device=device, dtype=torch.float32) * w.s_std
    d = torch.rand(w.B, w.H, w.K, generator=g, device=device, dtype=torch.float32) * 1.5 + 0.5
    return S, d
