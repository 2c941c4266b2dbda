"""Host-only checks of the C ABI (no GPU needed): the library loads, exports every entry point
that include/osdn.h declares, and rejects bad arguments on the host before any launch.

Every call here is built to be REJECTED by validation (or to have nothing to do), so no kernel
is ever launched with the fake device addresses used below.
"""
import ctypes
import math
import os
import re

import pytest
import torch

from preconditioned_delta_rule_gb300 import binding
from preconditioned_delta_rule_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
A = 0x10000  # a fake, 16-byte-aligned "device address" (never dereferenced: see module doc)
OK, ARG, SHAPE, DTYPE, ALIGN, UNSUP = 0, 1, 2, 3, 4, 5


@pytest.fixture(scope="module")
def L():
    build()
    return binding.lib()


def header_functions():
    src = open(os.path.join(ROOT, "include", "osdn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(osdn_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = header_functions()
    assert {"osdn_precond_scan", "osdn_chunk_fwd", "osdn_decode_step"} <= set(names)
    for n in names:
        assert hasattr(L, n), f"libosdn.so does not export {n}"


def test_status_strings_and_version(L):
    for code in range(10):
        s = binding.osdn_status_string(code)
        assert s.startswith(binding._STATUS[code])
    assert "unknown" in binding.osdn_status_string(99)
    assert binding.osdn_version() >= 100


def scan(L, **kw):
    a = dict(k=A, kdt=1, beta=A, r=None, d0=None, kt=A, ktdt=1, dout=A, B=2, T=64, H=2, K=128,
             eta=0.003, dmin=0.5, dmax=2.0, eps=1e-6, ba=1)
    a.update(kw)
    return L.osdn_precond_scan(a["k"], a["kdt"], a["beta"], a["r"], a.get("rpk", 0), a["d0"], a["kt"], a["ktdt"],
                               a["dout"], a["B"], a["T"], a["H"], a["K"], a["eta"], a["dmin"],
                               a["dmax"], a["eps"], a["ba"], a.get("ws"), a.get("wsb", 0), None)


def chunk(L, **kw):
    a = dict(q=A, k=A, kt=A, v=A, dt=1, beta=A, S0=None, o=A, Sout=A, B=2, T=128, H=2, K=128,
             V=128, C=64, scale=1.0)
    a.update(kw)
    return L.osdn_chunk_fwd(a["q"], a["k"], a["kt"], a["v"], a["dt"], a["beta"], a.get("alpha"), a.get("apk", 0), a["S0"],
                            a["o"],
                            a["Sout"], a["B"], a["T"], a["H"], a["K"], a["V"], a["C"], a["scale"],
                            a.get("ws"), a.get("wsb", 0), None)


def decode(L, **kw):
    a = dict(q=A, k=A, v=A, dt=1, beta=A, r=None, S=A, d=A, o=A, B=2, H=2, K=128, V=128,
             eta=0.003, dmin=0.5, dmax=2.0, eps=1e-6, scale=1.0, ba=1)
    a.update(kw)
    return L.osdn_decode_step(a["q"], a["k"], a["v"], a["dt"], a["beta"], a["r"], a.get("rpk", 0), a.get("alpha"),
                              a.get("apk", 0), a["S"], a["d"],
                              a["o"], a["B"], a["H"], a["K"], a["V"], a["eta"], a["dmin"],
                              a["dmax"], a["eps"], a["scale"], a["ba"], None)


@pytest.mark.parametrize("kw,want", [
    (dict(k=None), ARG), (dict(beta=None), ARG), (dict(kt=None), ARG), (dict(dout=None), ARG),
    (dict(k=A + 8), ALIGN), (dict(r=A + 4), ALIGN), (dict(d0=A + 2), ALIGN),
    (dict(K=96), UNSUP), (dict(K=0), SHAPE), (dict(B=-1), SHAPE), (dict(T=-1), SHAPE),
    (dict(kdt=7), DTYPE), (dict(ktdt=-1), DTYPE), (dict(ws=A + 4, wsb=1 << 20), ALIGN),
    (dict(eta=-0.1), ARG), (dict(eta=math.nan), ARG), (dict(eps=0.0), ARG),
    (dict(dmin=2.0, dmax=0.5), ARG), (dict(dmin=math.nan), ARG), (dict(rpk=2), ARG),
    (dict(r=A + 4, rpk=1), ALIGN), (dict(B=0), OK), (dict(H=0), OK),
])
def test_scan_validation(L, kw, want):
    assert scan(L, **kw) == want


@pytest.mark.parametrize("kw,want", [
    (dict(q=None), ARG), (dict(kt=None), ARG), (dict(o=None), ARG), (dict(Sout=None), ARG),
    (dict(v=A + 8), ALIGN), (dict(S0=A + 4), ALIGN),
    (dict(T=100), SHAPE), (dict(C=0), SHAPE), (dict(C=32), UNSUP), (dict(K=256), UNSUP),
    (dict(V=48), UNSUP), (dict(dt=5), DTYPE), (dict(scale=math.inf), ARG),
    (dict(ws=A + 8, wsb=1 << 20), ALIGN), (dict(alpha=A + 4), ALIGN), (dict(apk=2), ARG), (dict(B=0), OK),
])
def test_chunk_validation(L, kw, want):
    assert chunk(L, **kw) == want


@pytest.mark.parametrize("kw,want", [
    (dict(S=None), ARG), (dict(d=None), ARG), (dict(o=None), ARG), (dict(q=A + 1), ALIGN),
    (dict(K=32), UNSUP), (dict(dt=3), DTYPE), (dict(eps=-1.0), ARG), (dict(scale=math.nan), ARG),
    (dict(rpk=-1), ARG), (dict(alpha=A + 8), ALIGN), (dict(apk=-1), ARG), (dict(H=0), OK),
])
def test_decode_validation(L, kw, want):
    assert decode(L, **kw) == want


def test_binding_rejects_host_tensors(L):
    k = torch.zeros(1, 64, 1, 64, dtype=torch.bfloat16)
    beta = torch.zeros(1, 64, 1)
    with pytest.raises(ValueError, match="CUDA tensor"):
        binding.osdn_precond_scan(k, beta)


def test_workspace_size_query(L):
    f = L.osdn_chunk_fwd_workspace_bytes
    assert f(8, 2048, 8, 128, 128, 64, 1) == 8 * 8 * 32 * 33280
    assert f(1, 64, 1, 128, 128, 64, 2) == 33280
    assert f(1, 64, 1, 64, 64, 64, 1) == 0      # shapes the tensor-core path does not cover
    assert f(1, 64, 1, 128, 128, 64, 0) == 0    # fp32 inputs use the CUDA-core kernel
    assert f(1, 100, 1, 128, 128, 64, 1) == 0   # T not a multiple of the chunk


def test_scan_workspace_size_query(L):
    f = L.osdn_precond_scan_workspace_bytes
    assert f(8, 2048, 8, 128, 1) == 4 * 8 * 8 * (2048 + 32 * 256)
    assert f(1, 100, 2, 128, 2) == 4 * 2 * (100 + 2 * 256)   # ragged tail: ceil(100 / 64) blocks
    assert f(1, 64, 1, 64, 1) == 0      # K = 64 runs the warp-per-head scan, no workspace
    assert f(1, 64, 1, 128, 0) == 0     # fp32 keys likewise
    assert f(1, 0, 1, 128, 1) == 0


def layer(L, **kw):
    a = dict(q=A, k=A, v=A, dt=1, beta=A, r=None, d0=None, S0=None, kt=A, o=A, Sout=A, dout=A, B=2, T=128,
             H=2, K=128, V=128, C=64, eta=0.003, dmin=0.5, dmax=2.0, eps=1e-6, scale=1.0, ba=1)
    a.update(kw)
    return L.osdn_layer_fwd(a["q"], a["k"], a["v"], a["dt"], a["beta"], a["r"], a.get("rpk", 0), a.get("alpha"),
                            a.get("apk", 0), a["d0"], a["S0"], a["kt"],
                            a["o"], a["Sout"], a["dout"], a["B"], a["T"], a["H"], a["K"], a["V"], a["C"],
                            a["eta"], a["dmin"], a["dmax"], a["eps"], a["scale"], a["ba"], a.get("ws"),
                            a.get("wsb", 0), None)


@pytest.mark.parametrize("kw,want", [
    (dict(kt=None), ARG), (dict(dout=None), ARG), (dict(Sout=None), ARG), (dict(o=None), ARG),
    (dict(q=A + 2), ALIGN), (dict(ws=A + 8, wsb=1 << 20), ALIGN), (dict(K=96), UNSUP), (dict(C=32), UNSUP),
    (dict(T=100), SHAPE), (dict(dt=5), DTYPE), (dict(eta=-1.0), ARG), (dict(scale=math.inf), ARG),
    (dict(rpk=3), ARG), (dict(alpha=A + 12), ALIGN), (dict(apk=5), ARG), (dict(B=0), OK),
])
def test_layer_validation(L, kw, want):
    assert layer(L, **kw) == want


def test_layer_workspace_size_query(L):
    f = L.osdn_layer_fwd_workspace_bytes
    scan = 4 * 8 * 8 * (2048 + 32 * 256)
    chunk = 8 * 8 * 32 * 33280
    got = f(8, 2048, 8, 128, 128, 64, 1)
    assert got >= scan + chunk + 4               # both workspaces and a chunk counter
    assert got < scan + chunk + 1024
    assert f(1, 64, 1, 64, 64, 64, 0) == 0        # fp32, K = 64: no workspace is used
    assert f(1, 100, 1, 128, 128, 64, 1) == 0     # T not a multiple of the chunk


def varlen(L, **kw):
    a = dict(q=A, k=A, v=A, dt=1, beta=A, r=None, rpk=0, alpha=None, cu=A, N=3, total=300, maxlen=128, d0=None,
             S0=None, kt=A, o=A, Sout=A, dout=A, H=2, K=128, V=128, C=64, eta=0.003, dmin=0.5, dmax=2.0, eps=1e-6,
             scale=1.0, ba=1, ws=A, wsb=1 << 40)
    a.update(kw)
    return L.osdn_layer_fwd_varlen(a["q"], a["k"], a["v"], a["dt"], a["beta"], a["r"], a["rpk"], a["alpha"],
                                   a.get("apk", 0), a["cu"],
                                   a["N"], a["total"], a["maxlen"], a["d0"], a["S0"], a["kt"], a["o"], a["Sout"],
                                   a["dout"], a["H"], a["K"], a["V"], a["C"], a["eta"], a["dmin"], a["dmax"], a["eps"],
                                   a["scale"], a["ba"], a["ws"], a["wsb"], None)


@pytest.mark.parametrize("kw,want", [
    (dict(cu=None), ARG), (dict(ws=None), ARG), (dict(wsb=1024), ARG), (dict(cu=A + 4), ALIGN),
    (dict(q=A + 2), ALIGN), (dict(alpha=A + 8), ALIGN), (dict(dout=None), ARG), (dict(K=96), UNSUP),
    (dict(C=32), UNSUP), (dict(N=-1), SHAPE), (dict(total=-1), SHAPE), (dict(maxlen=-1), SHAPE),
    (dict(dt=9), DTYPE), (dict(rpk=2), ARG), (dict(eta=math.nan), ARG), (dict(N=0), OK), (dict(H=0), OK),
])
def test_varlen_validation(L, kw, want):
    assert varlen(L, **kw) == want


def test_gated_workspace_size_queries(L):
    """gated = 2 (one gate per key channel) keeps Q . Gamma, K~ . Gamma_C / Gamma and Gamma_C per
    chunk besides the images: 66048 bytes per chunk of each head; gated 0 and 1 as the plain query."""
    f, f0 = L.osdn_chunk_fwd_gated_workspace_bytes, L.osdn_chunk_fwd_workspace_bytes
    assert f(8, 2048, 8, 128, 128, 64, 1, 0) == f0(8, 2048, 8, 128, 128, 64, 1) == 8 * 8 * 32 * 33280
    assert f(8, 2048, 8, 128, 128, 64, 1, 1) == 8 * 8 * 32 * 33280
    assert f(8, 2048, 8, 128, 128, 64, 1, 2) == 8 * 8 * 32 * 66048
    assert f(8, 2048, 8, 128, 128, 64, 1, 3) == 0 and f(8, 2048, 8, 128, 128, 64, 1, -1) == 0
    g, g0 = L.osdn_layer_fwd_gated_workspace_bytes, L.osdn_layer_fwd_workspace_bytes
    assert g(8, 2048, 8, 128, 128, 64, 1, 0) == g0(8, 2048, 8, 128, 128, 64, 1)
    scan = 4 * 8 * 8 * (2048 + 32 * 256)
    assert g(8, 2048, 8, 128, 128, 64, 1, 2) == (scan + 255) // 256 * 256 + 8 * 8 * 32 * 66048
    assert g(8, 2048, 8, 128, 128, 64, 1, 3) == 0


def test_varlen_workspace_size_query(L):
    f = L.osdn_layer_fwd_varlen_workspace_bytes
    lay = L.osdn_layer_fwd_workspace_bytes
    up = lambda x: (x + 255) // 256 * 256
    N, H, Tp = 4, 8, 320                       # max_len 300 rounds up to 320
    rows = N * Tp
    pad = 3 * up(rows * H * 128 * 2) + 2 * up(rows * H * 128 * 2) + up(rows * H * 4)
    assert f(N, 300, H, 128, 128, 64, 1, 0, 0) == up(pad) + lay(N, Tp, H, 128, 128, 64, 1)
    assert f(N, 300, H, 128, 128, 64, 1, 1, 1) == up(pad + 2 * up(rows * H * 4)) + lay(N, Tp, H, 128, 128, 64, 1)
    assert f(N, 0, H, 128, 128, 64, 1, 0, 0) > 0   # all empty: one chunk of padding each
    assert f(0, 300, H, 128, 128, 64, 1, 0, 0) == 0
    assert f(N, 300, H, 128, 128, 64, 1, 3, 0) == 0
    # one gate per key channel: the batched layer's workspace is the channel-gated one
    layg = L.osdn_layer_fwd_gated_workspace_bytes
    assert f(N, 300, H, 128, 128, 64, 1, 0, 2) == up(pad + up(rows * H * 128 * 4)) + layg(N, Tp, H, 128, 128, 64, 1, 2)
    assert f(N, 300, H, 128, 128, 64, 1, 0, 3) == 0


def host_layer(L, **kw):
    a = dict(q=A, k=A, v=A, dt=1, beta=A, r=None, rpk=0, alpha=None, apk=0, d0=None, S0=None, o=A, Sout=A, dout=A,
             B=2, T=256, H=2, K=128, V=128, C=64, eta=0.003, dmin=0.5, dmax=2.0, eps=1e-6, scale=1.0, ba=1, seg=4,
             ws=ctypes.c_void_p(1 << 20), wsb=1 << 40)
    a.update(kw)
    return L.osdn_layer_fwd_host(a["q"], a["k"], a["v"], a["dt"], a["beta"], a["r"], a["rpk"], a["alpha"], a["apk"],
                                 a["d0"], a["S0"], a["o"], a["Sout"], a["dout"], a["B"], a["T"], a["H"], a["K"],
                                 a["V"], a["C"], a["eta"], a["dmin"], a["dmax"], a["eps"], a["scale"], a["ba"],
                                 a["seg"], a["ws"], a["wsb"], None, None, None)


@pytest.mark.parametrize("kw,want", [
    (dict(seg=0), ARG), (dict(seg=3), SHAPE), (dict(seg=8), SHAPE), (dict(T=100, seg=1), SHAPE),
    (dict(ws=None), ARG), (dict(wsb=1024), ARG), (dict(ws=ctypes.c_void_p((1 << 20) + 128)), ALIGN),
    (dict(q=None), ARG), (dict(Sout=None), ARG), (dict(K=96), UNSUP), (dict(C=32), UNSUP), (dict(dt=9), DTYPE),
    (dict(rpk=2), ARG), (dict(apk=2), ARG), (dict(dmin=3.0), ARG), (dict(eta=math.nan), ARG), (dict(B=-1), SHAPE),
    (dict(eta=math.inf), ARG), (dict(eps=0.0), ARG), (dict(eps=math.inf), ARG), (dict(scale=math.inf), ARG),
    (dict(dmin=math.nan), ARG), (dict(B=0), OK), (dict(H=0), OK),
])
def test_host_layer_validation(L, kw, want):
    """Every argument error is returned before any CUDA call (host buffers need no alignment)."""
    assert host_layer(L, **kw) == want


def test_host_layer_workspace_size_query(L):
    f = L.osdn_layer_fwd_host_workspace_bytes
    lay = L.osdn_layer_fwd_workspace_bytes
    up = lambda x: (x + 255) // 256 * 256
    B, T, H, seg = 8, 2048, 8, 4
    rows = B * (T // seg) * H
    state = 2 * (up(B * H * 128 * 4) + up(B * H * 128 * 128 * 4))
    slot = 5 * up(rows * 128 * 2) + up(rows * 4)  # q, k, v, k~, o and beta
    assert f(B, T, H, 128, 128, 64, 1, 0, 0, seg) == state + 2 * slot + lay(B, T // seg, H, 128, 128, 64, 1)
    assert f(B, T, H, 128, 128, 64, 1, 2, 1, seg) == (state + 2 * (slot + up(rows * 128 * 4) + up(rows * 4))
                                                      + lay(B, T // seg, H, 128, 128, 64, 1))
    assert f(B, T, H, 128, 128, 64, 1, 0, 0, 3) == 0      # 2048 / 3 is not whole
    assert f(B, T, H, 128, 128, 64, 1, 0, 0, 64) == 0     # 32 tokens: not a whole chunk
    assert f(B, 0, H, 128, 128, 64, 1, 0, 0, 1) == 0
    assert f(B, T, H, 128, 128, 64, 1, 3, 0, seg) == 0


def test_host_binding_rejects_device_side_arguments(L):
    k = torch.zeros(1, 64, 1, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="shape"):
        binding.osdn_layer_fwd_host(k, k, k, torch.zeros(1, 64, 2))
