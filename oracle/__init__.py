"""fp64 CPU oracle for the OSDN forward path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's ``cpu_baseline`` /
``--impl reference`` legs may import this package.  The product path (the CUDA library and its
Python binding) never imports it, and it imports nothing from the product.

The arithmetic lives in ``osdn_oracle.c`` (plain C, double precision, token by token, OpenMP over
independent heads).  This module only compiles it with gcc and marshals numpy arrays.

Parity status of each function (what pins it is in ``tests/test_oracle_pins.py``):
  precond_scan   pinned (surrogate-gradient identity, box invariant, special cases, fixtures)
  delta_phase2   pinned (textbook DeltaNet at d = 1, residual identity, chunk-form identity)
  osdn_forward   pinned (decoupling into the two phases, continuation, Cor. D.8 identity)
  decode_step    pinned (equals the forward on one token; decode x T equals forward on T)
  alpha [B,T,H,K] (one state gate per key channel, OSKDA): pinned (a textbook KDA recurrence in
                 its own K x V convention at eta = 0; equal channel gates reproduce the head gate)
  alpha (the OSGDN state gate, any of the three phase-2 functions): pinned (alpha = 1 is the
                 ungated rule; eta = 0 is a separately written Gated DeltaNet; the chunk form of
                 Eqs. (13)-(15) equals the recurrence; a zero gate forgets the state)
  backward.layer_backward (oracle/backward.py, the gradients of the layer forward by reverse-mode
                 differentiation of a plain fp64 PyTorch token loop): pinned (its forward equals
                 this library's; every gradient equals central finite differences of it)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "osdn_oracle.c"
_BUILD = _HERE / "_build"
_LIB_PATH = _BUILD / "libosdn_oracle.so"
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> Path:
    """Compile the oracle shared library with gcc (OpenMP, no FP contraction)."""
    with _lock:
        if _LIB_PATH.exists() and not force and _LIB_PATH.stat().st_mtime >= _SRC.stat().st_mtime:
            return _LIB_PATH
        _BUILD.mkdir(exist_ok=True)
        tmp = _BUILD / f"libosdn_oracle.{os.getpid()}.so"
        cmd = ["gcc", "-std=c11", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
               str(_SRC), "-o", str(tmp), "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        path = build()
        lib = ctypes.CDLL(str(path))
        i, d = ctypes.c_int, ctypes.c_double
        lib.oracle_precond_scan.argtypes = [_dp] * 3 + [i] + [_dp] * 4 + [i] * 4 + [d] * 4 + [i, i]
        lib.oracle_delta_phase2.argtypes = [_dp] * 6 + [i] + [_dp] * 3 + [i] * 5 + [d, i]
        lib.oracle_osdn_forward.argtypes = [_dp] * 5 + [i, _dp, i] + [_dp] * 8 + [i] * 5 + [d] * 4 + [i, d, i]
        lib.oracle_decode_step.argtypes = [_dp] * 5 + [i, _dp, i] + [_dp] * 3 + [i] * 4 + [d] * 4 + [i, d, i]
        for f in ("oracle_precond_scan", "oracle_delta_phase2", "oracle_osdn_forward",
                  "oracle_decode_step"):
            getattr(lib, f).restype = ctypes.c_int
        lib.oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _in(x):
    """Upcast an input (numpy array or torch tensor, any float dtype) to contiguous float64."""
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _p(a):
    return None if a is None else a.ctypes.data_as(_dp)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _per_key(r, k) -> int:
    """1 when r carries one retention per key coordinate (the layout of k), 0 for one per head."""
    if r is None:
        return 0
    if r.shape == k.shape:
        return 1
    if r.shape != k.shape[:-1]:
        raise ValueError(f"retention of shape {r.shape} fits neither {k.shape[:-1]} nor {k.shape}")
    return 0


def precond_scan(k, beta, r=None, d0=None, *, eta=0.003, d_min=0.5, d_max=2.0, eps=1e-6,
                 beta_aware=True, threads=0, return_a=False):
    """Phase 1 (Algorithm 1 / Eq. (4); Eq. (7) with r).  k [B,T,H,K] -> (k_tilde, d_out[, a]).
    r [B,T,H] is the per-head retention of Eq. (7); r [B,T,H,K] the vector retention diag(r_t)
    (Appendix A.5)."""
    k, beta, r, d0 = _in(k), _in(beta), _in(r), _in(d0)
    B, T, H, K = k.shape
    kt = np.empty_like(k)
    dout = np.empty((B, H, K))
    a = np.empty((B, T, H)) if return_a else None
    rc = _load().oracle_precond_scan(_p(k), _p(beta), _p(r), _per_key(r, k), _p(d0), _p(kt), _p(dout), _p(a),
                                     B, T, H, K, eta, d_min, d_max, eps, int(beta_aware), threads)
    if rc:
        raise ValueError("oracle_precond_scan: bad arguments")
    return (kt, dout, a) if return_a else (kt, dout)


def delta_phase2(q, k, k_tilde, v, beta, S0=None, *, alpha=None, scale=1.0, threads=0):
    """Phase 2 (Eq. (2)/(5)) token by token with the supplied write key -> (o, S_out).  alpha
    [B,T,H]: the OSGDN state gate (Appendix B.1, post-gate residual)."""
    q, k, kt, v, beta, S0, alpha = map(_in, (q, k, k_tilde, v, beta, S0, alpha))
    B, T, H, K = k.shape
    V = v.shape[-1]
    o = np.empty((B, T, H, V))
    S = np.empty((B, H, V, K))
    rc = _load().oracle_delta_phase2(_p(q), _p(k), _p(kt), _p(v), _p(beta), _p(alpha), _per_key(alpha, k), _p(S0),
                                     _p(o), _p(S),
                                     B, T, H, K, V, scale, threads)
    if rc:
        raise ValueError("oracle_delta_phase2: bad arguments")
    return o, S


def osdn_forward(q, k, v, beta, r=None, d0=None, S0=None, *, alpha=None, eta=0.003, d_min=0.5,
                 d_max=2.0, eps=1e-6, beta_aware=True, scale=1.0, threads=0):
    """Both phases interleaved per token.  Returns dict(o, S, d, k_tilde, a, u2).  alpha [B,T,H]:
    the OSGDN state gate (Appendix B.1)."""
    q, k, v, beta, r, d0, S0, alpha = map(_in, (q, k, v, beta, r, d0, S0, alpha))
    B, T, H, K = k.shape
    V = v.shape[-1]
    o = np.empty((B, T, H, V))
    S = np.empty((B, H, V, K))
    d = np.empty((B, H, K))
    kt = np.empty((B, T, H, K))
    a = np.empty((B, T, H))
    u2 = np.empty((B, T, H))
    rc = _load().oracle_osdn_forward(_p(q), _p(k), _p(v), _p(beta), _p(r), _per_key(r, k), _p(alpha),
                                     _per_key(alpha, k), _p(d0),
                                     _p(S0), _p(o),
                                     _p(S), _p(d), _p(kt), _p(a), _p(u2), B, T, H, K, V, eta,
                                     d_min, d_max, eps, int(beta_aware), scale, threads)
    if rc:
        raise ValueError("oracle_osdn_forward: bad arguments")
    return {"o": o, "S": S, "d": d, "k_tilde": kt, "a": a, "u2": u2}


def decode_step(q, k, v, beta, S, d, r=None, *, alpha=None, eta=0.003, d_min=0.5, d_max=2.0,
                eps=1e-6, beta_aware=True, scale=1.0, threads=0):
    """One decode token.  q, k [B,H,K], v [B,H,V], beta/r/alpha [B,H]; S [B,H,V,K], d [B,H,K] are
    copied, stepped and returned: (o, S_new, d_new)."""
    q, k, v, beta, r, alpha = map(_in, (q, k, v, beta, r, alpha))
    S = _in(S).copy()
    d = _in(d).copy()
    B, H, K = k.shape
    V = v.shape[-1]
    o = np.empty((B, H, V))
    rc = _load().oracle_decode_step(_p(q), _p(k), _p(v), _p(beta), _p(r), _per_key(r, k), _p(alpha),
                                    _per_key(alpha, k), _p(S), _p(d),
                                    _p(o),
                                    B, H, K, V, eta, d_min, d_max, eps, int(beta_aware), scale,
                                    threads)
    if rc:
        raise ValueError("oracle_decode_step: bad arguments")
    return o, S, d
