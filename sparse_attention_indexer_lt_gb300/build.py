"""Compile the CUDA library in-tree: ``liblt_topk.so`` next to this file.

Each translation unit is compiled for sm_103a in parallel, then linked with
the shared CUDA runtime (so the process shares one runtime with PyTorch).
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
CSRC = PKG / "csrc"
INCLUDE = PKG.parent / "include"
BUILD = PKG / "_build"
LIB = PKG / "liblt_topk.so"
SOURCES = ["lt_api.cu", "lt_topk_kernels.cu", "lt_stream_kernels.cu", "lt_blocked_256_f32.cu",
           "lt_blocked_256_bf16.cu", "lt_blocked_512_f32.cu", "lt_blocked_512_bf16.cu", "lt_listed_kernels.cu", "lt_compress.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", f"-I{INCLUDE}"]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not Path(exe).exists():
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build liblt_topk.so")
    return exe


def source_hash() -> str:
    """Hash of the CUDA sources and the C header (ties a profile to the code it measured)."""
    import hashlib
    h = hashlib.sha256()
    for f in sorted(list(CSRC.glob("*")) + list(INCLUDE.glob("*.h"))):
        h.update(f.name.encode())
        h.update(f.read_bytes())
    return h.hexdigest()[:16]


def _deps_mtime() -> float:
    files = list(CSRC.glob("*")) + list(INCLUDE.glob("*.h"))
    return max(f.stat().st_mtime for f in files)


def build(force: bool = False, verbose: bool = False) -> Path:
    if not force and LIB.exists() and LIB.stat().st_mtime >= _deps_mtime():
        return LIB
    BUILD.mkdir(exist_ok=True)
    exe = nvcc()

    def compile_one(src: str) -> Path:
        obj = BUILD / (Path(src).stem + ".o")
        cmd = [exe, *ARCH, *FLAGS, "-c", str(CSRC / src), "-o", str(obj)]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB.with_name(f"{LIB.name}.tmp{os.getpid()}")
    cmd = [exe, *ARCH, "-shared", "-cudart", "shared", "-o", str(tmp), *map(str, objs)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
