"""Build the OSDN CUDA library (libosdn.so) in-tree for sm_103a with nvcc.

Each .cu file is compiled to an object in parallel, then linked into one shared library with
the CUDA runtime linked statically, so the library needs only the NVIDIA driver at run time.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
BUILD = PKG / "_build"
LIB = PKG / "libosdn.so"
SOURCES = ["api.cu", "scan.cu", "scan_block.cu", "decode.cu", "chunk_simt.cu", "chunk_tc.cu", "chunk_static_ws.cu", "varlen.cu", "bwd.cu", "host_pipeline.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the OSDN CUDA library cannot be built")
    return cand


def _flags(extra=()):
    return [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
            f"-I{ROOT / 'include'}", f"-I{CSRC}", *extra]


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> Path:
    srcs = [CSRC / s for s in SOURCES]
    deps = srcs + [CSRC / "common.cuh", ROOT / "include" / "osdn.h"] + sorted(CSRC.glob("*.cuh"))
    if LIB.exists() and not force and LIB.stat().st_mtime >= max(p.stat().st_mtime for p in deps):
        return LIB
    BUILD.mkdir(exist_ok=True)
    nv = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(src: Path):
        obj = BUILD / (src.stem + ".o")
        cmd = [nv, *_flags(extra), "-c", str(src), "-o", str(obj)]
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src.name}:\n{p.stderr}")
        return obj, p.stderr

    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose or ptxas_info:
        for obj, log in results:
            if log.strip():
                print(f"--- {obj.name}\n{log}")
    tmp = BUILD / f"libosdn.{os.getpid()}.so"
    cmd = [nv, *ARCH, "-shared", "-cudart", "static", "-o", str(tmp), *[str(o) for o, _ in results]]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"link failed:\n{p.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
