"""Thin ctypes binding over libosdn.so (include/osdn.h): argument marshalling only.

Every function here takes torch CUDA tensors, checks shapes/dtypes/contiguity, allocates any
output the caller did not pass (PyTorch is only the device-memory and stream provider), and
calls the C entry point of the same name on the current torch stream.  All arithmetic runs in
the library's CUDA kernels; there is no CPU or PyTorch fallback.  A missing library raises.
"""
from __future__ import annotations

import ctypes
import math
from pathlib import Path
from typing import Optional

import torch

_PKG = Path(__file__).resolve().parent
LIB_PATH = _PKG / "libosdn.so"

OSDN_F32, OSDN_BF16, OSDN_F16 = 0, 1, 2
_DTYPE_CODE = {torch.float32: OSDN_F32, torch.bfloat16: OSDN_BF16, torch.float16: OSDN_F16}
_STATUS = ["OSDN_OK", "OSDN_ERR_ARG", "OSDN_ERR_SHAPE", "OSDN_ERR_DTYPE", "OSDN_ERR_ALIGN",
           "OSDN_ERR_UNSUPPORTED", "OSDN_ERR_CUDA", "OSDN_ERR_TIMEOUT", "OSDN_ERR_CAPACITY",
           "OSDN_ERR_RANGE"]
OSDN_ERR_TIMEOUT, OSDN_ERR_RANGE = _STATUS.index("OSDN_ERR_TIMEOUT"), _STATUS.index("OSDN_ERR_RANGE")

_lib = None


class OsdnError(RuntimeError):
    """A non-OK status from the C ABI."""

    def __init__(self, fn: str, status: int, detail: str):
        self.status = status
        super().__init__(f"{fn}: {detail} (status {status})")


def lib() -> ctypes.CDLL:
    """Load libosdn.so (built in-tree by ``preconditioned_delta_rule_gb300.build.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not LIB_PATH.exists():
        raise ImportError(f"{LIB_PATH} is missing: build the CUDA library first "
                          "(python -m preconditioned_delta_rule_gb300.build)")
    L = ctypes.CDLL(str(LIB_PATH))
    vp, fp, i, f = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    sz = ctypes.c_size_t
    L.osdn_precond_scan.argtypes = [vp, i, fp, fp, i, fp, vp, i, fp, i, i, i, i, f, f, f, f, i, vp, sz, vp]
    L.osdn_precond_scan_workspace_bytes.argtypes = [i, i, i, i, i]
    L.osdn_precond_scan_workspace_bytes.restype = sz
    L.osdn_chunk_fwd.argtypes = [vp, vp, vp, vp, i, fp, fp, i, fp, vp, fp, i, i, i, i, i, i, f, vp, sz, vp]
    L.osdn_chunk_fwd_workspace_bytes.argtypes = [i, i, i, i, i, i, i]
    L.osdn_chunk_fwd_workspace_bytes.restype = sz
    L.osdn_chunk_fwd_static_ws.argtypes = [vp, vp, vp, vp, i, fp, fp, i, fp, vp, fp, i, i, i, i, i, i, f, vp]
    L.osdn_chunk_fwd_static_ws.restype = ctypes.c_int
    L.osdn_layer_fwd.argtypes = [vp, vp, vp, i, fp, fp, i, fp, i, fp, fp, vp, vp, fp, fp, i, i, i, i, i, i,
                                 f, f, f, f, f, i, vp, sz, vp]
    L.osdn_layer_fwd.restype = ctypes.c_int
    L.osdn_layer_fwd_workspace_bytes.argtypes = [i, i, i, i, i, i, i]
    L.osdn_layer_fwd_workspace_bytes.restype = sz
    L.osdn_chunk_fwd_gated_workspace_bytes.argtypes = [i, i, i, i, i, i, i, i]
    L.osdn_chunk_fwd_gated_workspace_bytes.restype = sz
    L.osdn_layer_fwd_gated_workspace_bytes.argtypes = [i, i, i, i, i, i, i, i]
    L.osdn_layer_fwd_gated_workspace_bytes.restype = sz
    ll = ctypes.c_longlong
    L.osdn_layer_fwd_varlen.argtypes = [vp, vp, vp, i, fp, fp, i, fp, i, vp, i, ll, i, fp, fp, vp, vp, fp, fp, i, i, i,
                                        i, f, f, f, f, f, i, vp, sz, vp]
    L.osdn_layer_fwd_varlen.restype = ctypes.c_int
    L.osdn_layer_fwd_varlen_workspace_bytes.argtypes = [i, i, i, i, i, i, i, i, i]
    L.osdn_layer_fwd_varlen_workspace_bytes.restype = sz
    L.osdn_layer_fwd_host.argtypes = [vp, vp, vp, i, fp, fp, i, fp, i, fp, fp, vp, fp, fp, i, i, i, i, i, i,
                                      f, f, f, f, f, i, i, vp, sz, vp, vp, vp]
    L.osdn_layer_fwd_host.restype = ctypes.c_int
    L.osdn_layer_fwd_host_workspace_bytes.argtypes = [i, i, i, i, i, i, i, i, i, i]
    L.osdn_layer_fwd_host_workspace_bytes.restype = sz
    L.osdn_layer_bwd.argtypes = [vp, vp, vp, i, fp, fp, i, fp, fp, fp, fp, fp, fp, fp, fp, fp, fp, fp, fp, fp,
                                 i, i, i, i, i, f, f, f, f, f, i, vp, sz, vp]
    L.osdn_layer_bwd.restype = ctypes.c_int
    L.osdn_layer_bwd_workspace_bytes.argtypes = [i, i, i, i, i]
    L.osdn_layer_bwd_workspace_bytes.restype = sz
    L.osdn_decode_step.argtypes = [vp, vp, vp, i, fp, fp, i, fp, i, fp, fp, vp, i, i, i, i, f, f, f, f, f, i, vp]
    L.osdn_check.argtypes = [vp]
    for fn in ("osdn_precond_scan", "osdn_chunk_fwd", "osdn_decode_step", "osdn_check"):
        getattr(L, fn).restype = ctypes.c_int
    L.osdn_status_string.argtypes = [ctypes.c_int]
    L.osdn_status_string.restype = ctypes.c_char_p
    L.osdn_version.restype = ctypes.c_int
    L.osdn_last_cuda_error.restype = ctypes.c_char_p
    L.osdn_set_poll_limit.argtypes = [ctypes.c_uint]
    L.osdn_set_poll_limit.restype = None
    _lib = L
    return L


def osdn_status_string(status: int) -> str:
    return lib().osdn_status_string(int(status)).decode()


def osdn_version() -> int:
    return int(lib().osdn_version())


def osdn_set_poll_limit(polls: int) -> None:
    """Failure-detection hook: poll limit of the fused layer's prep workers (0: the default)."""
    lib().osdn_set_poll_limit(int(polls))


def _raise(fn: str, st: int):
    if st != 0:
        detail = osdn_status_string(st)
        if st == 6:  # OSDN_ERR_CUDA: name the CUDA error
            detail += f" [{lib().osdn_last_cuda_error().decode()}]"
        raise OsdnError(fn, st, detail)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device, stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


_HOST = object()  # device argument of _check for host (CPU) arrays


def _check(name, t, shape, dtype=None, device=None):
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if device is _HOST:  # the host-buffer entry point's arrays
        if t.is_cuda:
            raise ValueError(f"{name} must be a host (CPU) tensor")
        device = torch.device("cpu")
    elif not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")


def _code(dtype) -> int:
    if dtype not in _DTYPE_CODE:
        raise ValueError(f"unsupported dtype {dtype}; use float32, bfloat16 or float16")
    return _DTYPE_CODE[dtype]


def _state_gate(alpha, head_shape, K, dev):
    """Check the state gate and say its layout: 0 for one gate per head (``head_shape``, OSGDN), 1
    for one per key channel (``head_shape + (K,)``, OSKDA)."""
    if alpha is None:
        return 0
    per_key = tuple(alpha.shape) == tuple(head_shape) + (K,)
    _check("alpha", alpha, tuple(head_shape) + ((K,) if per_key else ()), torch.float32, dev)
    return int(per_key)


def _retention(r, head_shape, K, dev):
    """Check the retention and say its layout: 0 for one gate per head (``head_shape``, Eq. (7)),
    1 for one per key coordinate (``head_shape + (K,)``, the vector retention diag(r_t))."""
    if r is None:
        return 0
    per_key = tuple(r.shape) == tuple(head_shape) + (K,)
    _check("r", r, tuple(head_shape) + ((K,) if per_key else ()), torch.float32, dev)
    return int(per_key)


def osdn_precond_scan(k, beta, r=None, d0=None, *, k_tilde=None, kt_dtype=None, d_out=None,
                      eta=0.003, d_min=0.5, d_max=2.0, eps=1e-6, beta_aware=True, workspace=None,
                      stream=None):
    """Phase 1 (Algorithm 1 / Eq. (4); APF Eq. (7) with r).  k [B,T,H,K] -> (k_tilde, d_out).
    r is [B,T,H] (one retention per head) or [B,T,H,K] (vector retention, one per coordinate).

    ``workspace``: None (default) uses a cached torch buffer of the size the library asks for;
    a uint8 CUDA tensor is used as given; False makes the scan kernel write k_tilde itself."""
    B, T, H, K = k.shape
    dev = k.device
    _check("k", k, (B, T, H, K), device=dev)
    _check("beta", beta, (B, T, H), torch.float32, dev)
    r_per_key = _retention(r, (B, T, H), K, dev)
    _check("d0", d0, (B, H, K), torch.float32, dev)
    if k_tilde is None:
        k_tilde = torch.empty((B, T, H, K), device=dev, dtype=kt_dtype or k.dtype)
    _check("k_tilde", k_tilde, (B, T, H, K), device=dev)
    if d_out is None:
        d_out = torch.empty((B, H, K), device=dev, dtype=torch.float32)
    _check("d_out", d_out, (B, H, K), torch.float32, dev)
    need = osdn_precond_scan_workspace_bytes(B, T, H, K, k.dtype)
    ws_ptr, ws_bytes = _resolve_workspace(workspace, dev, need, "scan", stream)
    st = lib().osdn_precond_scan(_ptr(k), _code(k.dtype), _ptr(beta), _ptr(r), r_per_key, _ptr(d0),
                                 _ptr(k_tilde), _code(k_tilde.dtype), _ptr(d_out), B, T, H, K,
                                 float(eta), float(d_min), float(d_max), float(eps),
                                 int(bool(beta_aware)), ws_ptr, ws_bytes, _stream(dev, stream))
    _raise("osdn_precond_scan", st)
    return k_tilde, d_out


_WS_CACHE = {}


def osdn_precond_scan_workspace_bytes(B, T, H, K, dtype=torch.bfloat16) -> int:
    return int(lib().osdn_precond_scan_workspace_bytes(B, T, H, K, _code(dtype)))


def osdn_chunk_fwd_workspace_bytes(B, T, H, K, V, chunk=64, dtype=torch.bfloat16, gated=0) -> int:
    """gated: 0 none, 1 one state gate per head, 2 one per key channel."""
    return int(lib().osdn_chunk_fwd_gated_workspace_bytes(B, T, H, K, V, chunk, _code(dtype), int(gated)))


def _workspace(device, nbytes, role, stream=None):
    """A cached uint8 device buffer of at least nbytes per (device, role, stream): torch
    allocates, the library never does.  Calls on one stream run in order, so they can share a
    buffer; each entry point and each stream has its own, so that no two calls that may run at
    the same time on the GPU share scratch."""
    s = stream if stream is not None else torch.cuda.current_stream(device)
    key = (device, role, s.cuda_stream)
    buf = _WS_CACHE.get(key)
    if buf is None or buf.numel() < nbytes:
        if buf is not None:  # the old buffer may still be in use by work queued on s
            buf.record_stream(s)
        buf = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device)
        _WS_CACHE[key] = buf
    return buf


def _resolve_workspace(workspace, device, need, role, stream=None):
    """(pointer, bytes) for a workspace argument: None = cached buffer, False = none, else a tensor."""
    if workspace is None:
        ws = _workspace(device, need, role, stream) if need else None
    elif workspace is False:
        ws = None
    else:
        ws = workspace
        if not (isinstance(ws, torch.Tensor) and ws.is_cuda and ws.is_contiguous()):
            raise ValueError("workspace must be a contiguous CUDA tensor")
    if ws is None:
        return None, 0
    return ctypes.c_void_p(ws.data_ptr()), ws.numel() * ws.element_size()


def osdn_chunk_fwd(q, k, k_tilde, v, beta, S0=None, *, alpha=None, o=None, S_out=None, chunk=64,
                   scale=1.0, workspace=None, stream=None):
    """Phase 2 (Eqs. (2), (5), (8)-(11)).  Returns (o [B,T,H,V], S_out [B,H,V,K] fp32).
    ``alpha`` [B,T,H] fp32: the OSGDN state gate (Appendix B.1, Eqs. (13)-(15)), or [B,T,H,K]: one
    gate per key channel (OSKDA, Appendix B.2); None for none.

    ``workspace``: None (default) uses a cached torch buffer of the size the library asks for;
    a uint8 CUDA tensor is used as given; False runs the no-scratch fused kernel."""
    B, T, H, K = k.shape
    V = v.shape[-1]
    dev, dt = k.device, k.dtype
    for name, t, shp in (("q", q, (B, T, H, K)), ("k", k, (B, T, H, K)),
                         ("k_tilde", k_tilde, (B, T, H, K)), ("v", v, (B, T, H, V))):
        _check(name, t, shp, dt, dev)
    _check("beta", beta, (B, T, H), torch.float32, dev)
    a_per_key = _state_gate(alpha, (B, T, H), K, dev)
    _check("S0", S0, (B, H, V, K), torch.float32, dev)
    if o is None:
        o = torch.empty((B, T, H, V), device=dev, dtype=dt)
    _check("o", o, (B, T, H, V), dt, dev)
    if S_out is None:
        S_out = torch.empty((B, H, V, K), device=dev, dtype=torch.float32)
    _check("S_out", S_out, (B, H, V, K), torch.float32, dev)
    gated = 0 if alpha is None else (2 if a_per_key else 1)
    need = osdn_chunk_fwd_workspace_bytes(B, T, H, K, V, chunk, dt, gated) if T > 0 else 0
    ws_ptr, ws_bytes = _resolve_workspace(workspace, dev, need, "chunk", stream)
    st = lib().osdn_chunk_fwd(_ptr(q), _ptr(k), _ptr(k_tilde), _ptr(v), _code(dt), _ptr(beta),
                              _ptr(alpha), a_per_key, _ptr(S0), _ptr(o), _ptr(S_out), B, T, H, K, V, int(chunk),
                              float(scale), ws_ptr, ws_bytes, _stream(dev, stream))
    _raise("osdn_chunk_fwd", st)
    return o, S_out


def osdn_decode_step(q, k, v, beta, S, d, r=None, *, alpha=None, o=None, eta=0.003, d_min=0.5,
                     d_max=2.0, eps=1e-6, scale=1.0, beta_aware=True, stream=None):
    """One decode token in place on S [B,H,V,K] and d [B,H,K].  Returns o [B,H,V].  r is [B,H]
    or [B,H,K] (vector retention); alpha [B,H] the OSGDN state gate (None: none)."""
    B, H, K = k.shape
    V = v.shape[-1]
    dev, dt = k.device, k.dtype
    _check("q", q, (B, H, K), dt, dev)
    _check("v", v, (B, H, V), dt, dev)
    _check("beta", beta, (B, H), torch.float32, dev)
    r_per_key = _retention(r, (B, H), K, dev)
    a_per_key = _state_gate(alpha, (B, H), K, dev)
    _check("S", S, (B, H, V, K), torch.float32, dev)
    _check("d", d, (B, H, K), torch.float32, dev)
    if o is None:
        o = torch.empty((B, H, V), device=dev, dtype=dt)
    _check("o", o, (B, H, V), dt, dev)
    st = lib().osdn_decode_step(_ptr(q), _ptr(k), _ptr(v), _code(dt), _ptr(beta), _ptr(r), r_per_key,
                                _ptr(alpha), a_per_key, _ptr(S), _ptr(d), _ptr(o), B, H, K, V, float(eta), float(d_min),
                                float(d_max), float(eps), float(scale), int(bool(beta_aware)),
                                _stream(dev, stream))
    _raise("osdn_decode_step", st)
    return o


def osdn_check(stream=None, device=None):
    """Synchronise the stream and raise on a recorded device-side timeout or CUDA error."""
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    _raise("osdn_check", lib().osdn_check(_stream(dev, stream)))


def osdn_layer_fwd_workspace_bytes(B, T, H, K, V, chunk=64, dtype=torch.bfloat16, gated=0) -> int:
    """gated: 0 none, 1 one state gate per head, 2 one per key channel."""
    return int(lib().osdn_layer_fwd_gated_workspace_bytes(B, T, H, K, V, chunk, _code(dtype), int(gated)))


def osdn_layer_fwd(q, k, v, beta, r=None, d0=None, S0=None, *, alpha=None, k_tilde=None, o=None,
                   S_out=None, d_out=None, chunk=64, eta=0.003, d_min=0.5, d_max=2.0, eps=1e-6,
                   scale=1.0, beta_aware=True, workspace=None, stream=None):
    """Phase 1 then phase 2 in one call.  Returns (o, S_out, d_out, k_tilde).  ``alpha`` [B,T,H]:
    the OSGDN state gate of phase 2 (Appendix B.1); None for the ungated rule.

    ``workspace``: None (default) uses a cached torch buffer of the size the library asks for;
    a uint8 CUDA tensor is used as given; False runs without scratch."""
    B, T, H, K = k.shape
    V = v.shape[-1]
    dev, dt = k.device, k.dtype
    for name, t, shp in (("q", q, (B, T, H, K)), ("k", k, (B, T, H, K)), ("v", v, (B, T, H, V))):
        _check(name, t, shp, dt, dev)
    _check("beta", beta, (B, T, H), torch.float32, dev)
    r_per_key = _retention(r, (B, T, H), K, dev)
    a_per_key = _state_gate(alpha, (B, T, H), K, dev)
    _check("d0", d0, (B, H, K), torch.float32, dev)
    _check("S0", S0, (B, H, V, K), torch.float32, dev)
    if k_tilde is None:
        k_tilde = torch.empty((B, T, H, K), device=dev, dtype=dt)
    _check("k_tilde", k_tilde, (B, T, H, K), dt, dev)
    if o is None:
        o = torch.empty((B, T, H, V), device=dev, dtype=dt)
    _check("o", o, (B, T, H, V), dt, dev)
    if S_out is None:
        S_out = torch.empty((B, H, V, K), device=dev, dtype=torch.float32)
    _check("S_out", S_out, (B, H, V, K), torch.float32, dev)
    if d_out is None:
        d_out = torch.empty((B, H, K), device=dev, dtype=torch.float32)
    _check("d_out", d_out, (B, H, K), torch.float32, dev)
    gated = 0 if alpha is None else (2 if a_per_key else 1)
    need = osdn_layer_fwd_workspace_bytes(B, T, H, K, V, chunk, dt, gated) if T > 0 and T % chunk == 0 else 0
    ws_ptr, ws_bytes = _resolve_workspace(workspace, dev, need, "layer", stream)
    st = lib().osdn_layer_fwd(_ptr(q), _ptr(k), _ptr(v), _code(dt), _ptr(beta), _ptr(r), r_per_key, _ptr(alpha),
                              a_per_key, _ptr(d0),
                              _ptr(S0), _ptr(k_tilde), _ptr(o), _ptr(S_out), _ptr(d_out), B, T, H, K,
                              V, int(chunk), float(eta), float(d_min), float(d_max), float(eps),
                              float(scale), int(bool(beta_aware)), ws_ptr, ws_bytes,
                              _stream(dev, stream))
    _raise("osdn_layer_fwd", st)
    return o, S_out, d_out, k_tilde


def osdn_layer_fwd_varlen_workspace_bytes(N, max_len, H, K, V, chunk=64, dtype=torch.bfloat16, r_mode=0,
                                          gated=0) -> int:
    """gated: 0 no state gate, 1 one per head, 2 one per key channel."""
    return int(lib().osdn_layer_fwd_varlen_workspace_bytes(N, max_len, H, K, V, chunk, _code(dtype), int(r_mode),
                                                           int(gated)))


_COPY_STREAMS = {}


def _copy_streams(device):
    """The two copy streams osdn_layer_fwd_host overlaps with the compute, one pair per device."""
    s = _COPY_STREAMS.get(device)
    if s is None:
        s = (torch.cuda.Stream(device), torch.cuda.Stream(device))
        _COPY_STREAMS[device] = s
    return s


def osdn_layer_fwd_host_workspace_bytes(B, T, H, K, V, chunk=64, dtype=torch.bfloat16, r_mode=0, gated=0,
                                        segments=4) -> int:
    return int(lib().osdn_layer_fwd_host_workspace_bytes(B, T, H, K, V, chunk, _code(dtype), r_mode, gated,
                                                         segments))


def osdn_layer_fwd_host(q, k, v, beta, r=None, d0=None, S0=None, *, alpha=None, o=None, S_out=None, d_out=None,
                        segments=4, chunk=64, eta=0.003, d_min=0.5, d_max=2.0, eps=1e-6, scale=1.0,
                        beta_aware=True, device=None, workspace=None, stream=None, synchronize=True):
    """The layer forward (both phases, the pages' chunk_osdn) from HOST tensors: the sequence runs
    as ``segments`` consecutive pieces whose input copies overlap the previous piece's compute,
    with (d, S) carried on the device.  q, k [B,T,H,K], v [B,T,H,V], beta [B,T,H], r [B,T,H] or
    [B,T,H,K], alpha [B,T,H] or [B,T,H,K], d0 [B,H,K], S0 [B,H,V,K]: CPU tensors (page-locked for
    the overlap).  Returns CPU tensors (o, S_out, d_out), page-locked when allocated here.  With
    ``synchronize`` False the outputs are valid once ``stream`` has passed the call, and the
    inputs must stay unchanged until then."""
    B, T, H, K = k.shape
    V = v.shape[-1]
    dt = k.dtype
    cpu = _HOST
    for name, t, shp in (("q", q, (B, T, H, K)), ("k", k, (B, T, H, K)), ("v", v, (B, T, H, V))):
        _check(name, t, shp, dt, cpu)
    _check("beta", beta, (B, T, H), torch.float32, cpu)
    r_per_key = _retention(r, (B, T, H), K, cpu)
    a_per_key = _state_gate(alpha, (B, T, H), K, cpu)
    _check("d0", d0, (B, H, K), torch.float32, cpu)
    _check("S0", S0, (B, H, V, K), torch.float32, cpu)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if o is None:
        o = torch.empty((B, T, H, V), dtype=dt, pin_memory=True)
    if S_out is None:
        S_out = torch.empty((B, H, V, K), dtype=torch.float32, pin_memory=True)
    if d_out is None:
        d_out = torch.empty((B, H, K), dtype=torch.float32, pin_memory=True)
    _check("o", o, (B, T, H, V), dt, cpu)
    _check("S_out", S_out, (B, H, V, K), torch.float32, cpu)
    _check("d_out", d_out, (B, H, K), torch.float32, cpu)
    r_mode = 0 if r is None else (2 if r_per_key else 1)
    g_mode = 0 if alpha is None else (2 if a_per_key else 1)
    need = osdn_layer_fwd_host_workspace_bytes(B, T, H, K, V, chunk, dt, r_mode, g_mode, segments) if T > 0 else 0
    ws_ptr, ws_bytes = _resolve_workspace(workspace, dev, need, "host", stream)
    h2d, d2h = _copy_streams(dev)
    st = lib().osdn_layer_fwd_host(_ptr(q), _ptr(k), _ptr(v), _code(dt), _ptr(beta), _ptr(r), r_per_key,
                                   _ptr(alpha), a_per_key, _ptr(d0), _ptr(S0), _ptr(o), _ptr(S_out), _ptr(d_out),
                                   B, T, H, K, V, int(chunk), float(eta),
                                   float(-math.inf if d_min is None else d_min),
                                   float(math.inf if d_max is None else d_max), float(eps), float(scale),
                                   int(bool(beta_aware)), int(segments), ws_ptr, ws_bytes, _stream(dev, stream),
                                   ctypes.c_void_p(h2d.cuda_stream), ctypes.c_void_p(d2h.cuda_stream))
    _raise("osdn_layer_fwd_host", st)
    if synchronize:
        (stream if stream is not None else torch.cuda.current_stream(dev)).synchronize()
    return o, S_out, d_out


def osdn_layer_fwd_varlen(q, k, v, beta, cu_seqlens, *, max_len=None, r=None, alpha=None, d0=None, S0=None,
                          k_tilde=None, o=None, S_out=None, d_out=None, chunk=64, eta=0.003, d_min=0.5, d_max=2.0,
                          eps=1e-6, scale=1.0, beta_aware=True, workspace=None, stream=None):
    """The layer forward over N packed variable-length sequences.  q, k [total,H,K] and v [total,H,V]
    (a leading batch dimension of 1 is accepted), beta and alpha [total,H], r [total,H] or
    [total,H,K]; cu_seqlens: int32 CUDA tensor [N+1] of sequence offsets; d0 [N,H,K], S0 [N,H,V,K]
    per sequence.  ``max_len`` (the longest sequence) is read from cu_seqlens when None, which
    synchronises.  Returns (o [total,H,V], S_out [N,H,V,K], d_out [N,H,K], k_tilde [total,H,K])."""
    squeeze = k.dim() == 4
    if squeeze:
        if k.shape[0] != 1:
            raise ValueError("packed sequences take a leading batch dimension of 1 at most")
        q, k, v, beta = q[0], k[0], v[0], beta[0]
        r = None if r is None else r[0]
        alpha = None if alpha is None else alpha[0]
    total, H, K = k.shape
    V = v.shape[-1]
    dev, dt = k.device, k.dtype
    for name, t, shp in (("q", q, (total, H, K)), ("k", k, (total, H, K)), ("v", v, (total, H, V))):
        _check(name, t, shp, dt, dev)
    _check("beta", beta, (total, H), torch.float32, dev)
    r_per_key = _retention(r, (total, H), K, dev)
    a_per_key = _state_gate(alpha, (total, H), K, dev)
    _check("cu_seqlens", cu_seqlens, (cu_seqlens.shape[0],), torch.int32, dev)
    N = cu_seqlens.shape[0] - 1
    if N < 0:
        raise ValueError("cu_seqlens needs at least one entry")
    if max_len is None:
        max_len = int((cu_seqlens[1:] - cu_seqlens[:-1]).max().item()) if N > 0 else 0
    _check("d0", d0, (N, H, K), torch.float32, dev)
    _check("S0", S0, (N, H, V, K), torch.float32, dev)
    if k_tilde is None:
        k_tilde = torch.empty((total, H, K), device=dev, dtype=dt)
    _check("k_tilde", k_tilde, (total, H, K), dt, dev)
    if o is None:
        o = torch.empty((total, H, V), device=dev, dtype=dt)
    _check("o", o, (total, H, V), dt, dev)
    if S_out is None:
        S_out = torch.empty((N, H, V, K), device=dev, dtype=torch.float32)
    _check("S_out", S_out, (N, H, V, K), torch.float32, dev)
    if d_out is None:
        d_out = torch.empty((N, H, K), device=dev, dtype=torch.float32)
    _check("d_out", d_out, (N, H, K), torch.float32, dev)
    r_mode = 0 if r is None else 1 + r_per_key
    g_mode = 0 if alpha is None else 1 + a_per_key
    need = osdn_layer_fwd_varlen_workspace_bytes(N, max_len, H, K, V, chunk, dt, r_mode, g_mode) if N else 0
    if workspace is False:
        raise ValueError("osdn_layer_fwd_varlen needs a workspace")
    ws_ptr, ws_bytes = _resolve_workspace(workspace, dev, need, "varlen", stream)
    st = lib().osdn_layer_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _code(dt), _ptr(beta), _ptr(r), r_per_key, _ptr(alpha),
                                     a_per_key, _ptr(cu_seqlens), N, int(total), int(max_len), _ptr(d0), _ptr(S0), _ptr(k_tilde),
                                     _ptr(o), _ptr(S_out), _ptr(d_out), H, K, V, int(chunk), float(eta), float(d_min),
                                     float(d_max), float(eps), float(scale), int(bool(beta_aware)), ws_ptr, ws_bytes,
                                     _stream(dev, stream))
    _raise("osdn_layer_fwd_varlen", st)
    if squeeze:
        return o[None], S_out, d_out, k_tilde[None]
    return o, S_out, d_out, k_tilde


def osdn_layer_bwd_workspace_bytes(B, T, H, K, V) -> int:
    return int(lib().osdn_layer_bwd_workspace_bytes(B, T, H, K, V))


def osdn_layer_bwd(q, k, v, beta, do, r=None, d0=None, S0=None, *, dS=None, dd=None, eta=0.003, d_min=0.5,
                   d_max=2.0, eps=1e-6, scale=1.0, beta_aware=True, workspace=None, stream=None):
    """Gradients of a loss through osdn_layer_fwd's o, S_out and d_out: ``do`` [B,T,H,V] and the
    optional ``dS`` [B,H,V,K], ``dd`` [B,H,K] (fp32) are the loss's gradients with respect to them.
    Returns a dict of fp32 tensors dq, dk, dv, dbeta, dr (None without r), dd0, dS0."""
    B, T, H, K = k.shape
    V = v.shape[-1]
    dev, dt = k.device, k.dtype
    for name, t, shp in (("q", q, (B, T, H, K)), ("k", k, (B, T, H, K)), ("v", v, (B, T, H, V))):
        _check(name, t, shp, dt, dev)
    _check("beta", beta, (B, T, H), torch.float32, dev)
    r_per_key = _retention(r, (B, T, H), K, dev)
    _check("d0", d0, (B, H, K), torch.float32, dev)
    _check("S0", S0, (B, H, V, K), torch.float32, dev)
    _check("do", do, (B, T, H, V), torch.float32, dev)
    _check("dS", dS, (B, H, V, K), torch.float32, dev)
    _check("dd", dd, (B, H, K), torch.float32, dev)
    f32 = dict(device=dev, dtype=torch.float32)
    g = {"dq": torch.empty((B, T, H, K), **f32), "dk": torch.empty((B, T, H, K), **f32),
         "dv": torch.empty((B, T, H, V), **f32), "dbeta": torch.empty((B, T, H), **f32),
         "dr": None if r is None else torch.empty(tuple(r.shape), **f32),
         "dd0": torch.empty((B, H, K), **f32), "dS0": torch.empty((B, H, V, K), **f32)}
    need = osdn_layer_bwd_workspace_bytes(B, T, H, K, V)
    if workspace is False:
        raise ValueError("osdn_layer_bwd needs a workspace")
    ws_ptr, ws_bytes = _resolve_workspace(workspace, dev, need, "bwd", stream)
    st = lib().osdn_layer_bwd(_ptr(q), _ptr(k), _ptr(v), _code(dt), _ptr(beta), _ptr(r), r_per_key, None, _ptr(d0),
                              _ptr(S0), _ptr(do), _ptr(dS), _ptr(dd), _ptr(g["dq"]), _ptr(g["dk"]), _ptr(g["dv"]),
                              _ptr(g["dbeta"]), _ptr(g["dr"]), _ptr(g["dd0"]), _ptr(g["dS0"]), B, T, H, K, V,
                              float(eta), float(d_min), float(d_max), float(eps), float(scale),
                              int(bool(beta_aware)), ws_ptr, ws_bytes, _stream(dev, stream))
    _raise("osdn_layer_bwd", st)
    return g


def chunk_osdn(q, k, v, beta, precond_retention=None, initial_state=None, initial_d=None, *,
               chunk_size=64, eta=0.003, beta_aware=True, d_min=0.5, d_max=2.0, eps=1e-6,
               scale=1.0, workspace=None, stream=None):
    """Both phases of the layer forward (the pages' ``chunk_osdn`` signature, Listing 1) through
    osdn_layer_fwd.  ``scale`` defaults to 1 (o_t = S_t q_t as in the equations; pass K ** -0.5
    for the listing's query scaling).  Returns (o, S, d)."""
    o, S, d, _ = osdn_layer_fwd(q, k, v, beta, precond_retention, initial_d, initial_state,
                                chunk=chunk_size, eta=eta,
                                d_min=-math.inf if d_min is None else d_min,
                                d_max=math.inf if d_max is None else d_max, eps=eps, scale=scale,
                                beta_aware=beta_aware, workspace=workspace, stream=stream)
    return o, S, d
