"""fp64 CPU reference of the OSDN layer backward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/`` may import this module (like the rest of ``oracle/``); the product path never
does, and it imports nothing from the product.

What it computes: the gradients of a scalar L = <do, o> + <dS, S_T> + <dd, d_T> + <dkt, k~>
with respect to the forward's inputs (q, k, v, beta, r, alpha, d0, S0), where the forward is the
token loop of "OSDN: Improving Delta Rule with Provable Online Preconditioning in Linear
Attention" restated in plain PyTorch fp64 CPU ops, one token at a time, in the order of the
definition (the same one ``osdn_oracle.c`` follows; ``tests/test_oracle_pins.py`` checks that the
two forwards agree):
  k~_t = d_t . k_t (emitted with the old d, Algorithm 1);
  d_{t+1} = clip(r_t d_t + eta b (1 - b <d_t, k_t^2>) / max(|k_t|^2, eps) k_t^2), b = beta_t or 1
    (Eqs. (4), (7); Appendix A.5 for one gate per coordinate);
  Sbar = alpha_t S_{t-1} (the gated variant, Appendix B.1; alpha = 1 without it);
  u_t = v_t - Sbar k_t;  S_t = Sbar + beta_t u_t k~_t^T;  o_t = scale S_t q_t (Eqs. (2), (5)).
The gradients come from reverse-mode automatic differentiation of that loop (a library routine
used as one step).  The clip passes the gradient where d_min <= x <= d_max and stops it outside:
a clipped coordinate has zero gradient (at the faces themselves the closed interval is this
module's reading).

Parity status: pinned -- the forward equals the C oracle's, and every gradient equals central
finite differences of the C oracle's forward (``tests/test_oracle_pins.py``).
"""
from __future__ import annotations

import numpy as np
import torch


def _t(x):
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu", torch.float64)
    return torch.as_tensor(np.asarray(x, dtype=np.float64))


def forward(q, k, v, beta, r=None, d0=None, S0=None, alpha=None, *, eta=0.003, d_min=0.5, d_max=2.0,
            eps=1e-6, beta_aware=True, scale=1.0):
    """The token loop on fp64 tensors (autograd-friendly).  q, k [B,T,H,K], v [B,T,H,V],
    beta / alpha [B,T,H], r [B,T,H] or [B,T,H,K].  Returns (o, S_T, d_T, k~)."""
    B, T, H, K = k.shape
    V = v.shape[-1]
    d = d0 if d0 is not None else torch.ones(B, H, K, dtype=k.dtype)
    S = S0 if S0 is not None else torch.zeros(B, H, V, K, dtype=k.dtype)
    per_key = r is not None and r.dim() == 4
    outs, kts = [], []
    for t in range(T):
        kk = k[:, t]
        kt = d * kk
        s = kk * kk
        nbar = torch.clamp(s.sum(-1), min=eps)
        b = beta[:, t] if beta_aware else torch.ones_like(beta[:, t])
        a = (d * s).sum(-1)
        g = eta * b * (1.0 - b * a) / nbar
        if r is None:
            rd = d
        else:
            rd = (r[:, t] if per_key else r[:, t][..., None]) * d
        d = torch.clamp(rd + g[..., None] * s, min=d_min, max=d_max)
        if alpha is not None:  # one gate per head (Appendix B.1) or per key channel (B.2)
            S = (alpha[:, t][..., None, :] if alpha.dim() == 4 else alpha[:, t][..., None, None]) * S
        u = v[:, t] - torch.einsum("bhvk,bhk->bhv", S, kk)
        S = S + beta[:, t][..., None, None] * u[..., :, None] * kt[..., None, :]
        outs.append(scale * torch.einsum("bhvk,bhk->bhv", S, q[:, t]))
        kts.append(kt)
    return torch.stack(outs, 1), S, d, torch.stack(kts, 1)


def layer_backward(q, k, v, beta, r=None, d0=None, S0=None, alpha=None, *, do=None, dS=None, dd=None,
                   dkt=None, eta=0.003, d_min=0.5, d_max=2.0, eps=1e-6, beta_aware=True, scale=1.0):
    """Gradients of L = <do, o> + <dS, S_T> + <dd, d_T> + <dkt, k~> (absent terms are zero).
    Returns a dict of numpy arrays: dq, dk, dv, dbeta, dr, dalpha, dd0, dS0 (None where the input
    was None), plus the forward's o, S, d, k_tilde."""
    names = ("q", "k", "v", "beta", "r", "d0", "S0", "alpha")
    vals = [_t(x) for x in (q, k, v, beta, r, d0, S0, alpha)]
    B, T, H, K = vals[1].shape
    V = vals[2].shape[-1]
    if vals[5] is None:
        vals[5] = torch.ones(B, H, K, dtype=torch.float64)
    if vals[6] is None:
        vals[6] = torch.zeros(B, H, V, K, dtype=torch.float64)
    leaves = [x.clone().requires_grad_(True) if x is not None else None for x in vals]
    o, S, d, kt = forward(*leaves[:7], leaves[7], eta=eta, d_min=d_min, d_max=d_max, eps=eps,
                          beta_aware=beta_aware, scale=scale)
    L = torch.zeros((), dtype=torch.float64)
    for out, up in ((o, do), (S, dS), (d, dd), (kt, dkt)):
        if up is not None:
            L = L + (out * _t(up)).sum()
    used = [x for x in leaves if x is not None]
    grads = torch.autograd.grad(L, used, allow_unused=True)
    gi = iter(grads)
    res = {}
    for n, x in zip(names, leaves):
        if x is None:
            res["d" + n] = None
            continue
        g = next(gi)
        res["d" + n] = (torch.zeros_like(x) if g is None else g).detach().numpy()
    if r is None:
        res["dr"] = None
    if alpha is None:
        res["dalpha"] = None
    if d0 is None:
        res["dd0"] = None
    if S0 is None:
        res["dS0"] = None
    res.update(o=o.detach().numpy(), S=S.detach().numpy(), d=d.detach().numpy(), k_tilde=kt.detach().numpy())
    return res
