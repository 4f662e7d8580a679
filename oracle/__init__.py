"""CPU oracle for the indexer top-k and its two-level variant (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never imports, links or
calls it, and it never imports the CUDA library.

Scores may also be given as bf16 bit patterns (the ``*_bf16`` functions): they
are widened to the fp32 numbers they denote (exact) and ranked as those.

The arithmetic lives in ``lt_oracle.cpp`` (a per-row ``std::stable_sort`` by
score descending, ties by index ascending; the two-level variant in the page's
literal step order). This module only compiles it with the host compiler and
marshals numpy arrays through ``ctypes``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "lt_oracle.cpp"
_LIB = _HERE / "liblt_oracle.so"
_lib = None


def build(force: bool = False) -> Path:
    """Compile ``liblt_oracle.so`` next to its source (host C++ only)."""
    if force or not _LIB.exists() or _LIB.stat().st_mtime < _SRC.stat().st_mtime:
        tmp = _LIB.with_suffix(f".so.tmp{os.getpid()}")
        subprocess.run(
            ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", "-o", str(tmp), str(_SRC)],
            check=True,
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(str(_LIB))
        i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
        lib.lt_oracle_topk.argtypes = [vp, vp, i64, i64, i64, vp, vp, i32]
        lib.lt_oracle_topk.restype = ctypes.c_int
        lib.lt_oracle_topk_blocked.argtypes = [vp, vp, i64, i64, i64, i64, i64, vp, vp, vp, i32]
        lib.lt_oracle_topk_blocked.restype = ctypes.c_int
        lib.lt_oracle_topk_candidates.argtypes = [vp, vp, i64, i64, i64, vp, i64, i64, vp, vp, i32]
        lib.lt_oracle_topk_candidates.restype = ctypes.c_int
        _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _prep(scores, lengths):
    s = np.ascontiguousarray(np.asarray(scores, dtype=np.float32))
    if s.ndim == 1:
        s = s[None, :]
    if s.ndim != 2:
        raise ValueError("scores must be 1-D or 2-D")
    ln = None
    if lengths is not None:
        ln = np.ascontiguousarray(np.asarray(lengths, dtype=np.int32).reshape(-1))
        if ln.shape[0] != s.shape[0]:
            raise ValueError("lengths must have one entry per row")
    return s, ln


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def widen_bf16(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> the fp32 numbers they denote.

    A bf16 number is the upper half of an fp32 (sign, the same 8 exponent
    bits, the leading 7 fraction bits), so the fp32 it denotes has those 16
    bits on top and zeros below; the conversion is exact. Scores given as
    bf16 are ranked as these fp32 numbers (the same selection rules apply).
    """
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def topk_bf16(bits, lengths, k: int, nthreads: int | None = None):
    """topk over bf16 scores (uint16 bit patterns): the fp32 numbers they denote."""
    return topk(widen_bf16(bits), lengths, k, nthreads)


def topk_blocked_bf16(bits, lengths, block: int, k_blocks: int, k: int, nthreads: int | None = None):
    """topk_blocked over bf16 scores (uint16 bit patterns)."""
    return topk_blocked(widen_bf16(bits), lengths, block, k_blocks, k, nthreads)


def topk_candidates_bf16(bits, lengths, cand_blocks, block: int, k: int, nthreads: int | None = None):
    """topk_candidates over bf16 scores (uint16 bit patterns)."""
    return topk_candidates(widen_bf16(bits), lengths, cand_blocks, block, k, nthreads)


def topk(scores, lengths, k: int, nthreads: int | None = None):
    """Per-row top-k: (idx int32 [rows, k], val float32 [rows, k])."""
    s, ln = _prep(scores, lengths)
    rows, stride = s.shape
    idx = np.empty((rows, k), dtype=np.int32)
    val = np.empty((rows, k), dtype=np.float32)
    rc = _load().lt_oracle_topk(_ptr(s), _ptr(ln), rows, stride, int(k), _ptr(idx), _ptr(val),
                                int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError("lt_oracle_topk: invalid argument")
    return idx, val


def topk_blocked(scores, lengths, block: int, k_blocks: int, k: int, nthreads: int | None = None):
    """Two-level top-k: (idx [rows, k], val [rows, k], blocks int32 [rows, k_blocks])."""
    s, ln = _prep(scores, lengths)
    rows, stride = s.shape
    idx = np.empty((rows, k), dtype=np.int32)
    val = np.empty((rows, k), dtype=np.float32)
    blk = np.empty((rows, k_blocks), dtype=np.int32)
    rc = _load().lt_oracle_topk_blocked(_ptr(s), _ptr(ln), rows, stride, int(block), int(k_blocks),
                                        int(k), _ptr(idx), _ptr(val), _ptr(blk),
                                        int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError("lt_oracle_topk_blocked: invalid argument")
    return idx, val, blk


def topk_candidates(scores, lengths, cand_blocks, block: int, k: int, nthreads: int | None = None):
    """Top-k among the positions of the listed blocks: (idx int32 [rows, k], val float32 [rows, k]).

    cand_blocks: int [rows, n_cand]; ids outside [0, nblocks) are ignored and
    repeated ids count once.
    """
    s, ln = _prep(scores, lengths)
    rows, stride = s.shape
    cb = np.ascontiguousarray(np.asarray(cand_blocks, dtype=np.int32))
    if cb.ndim == 1:
        cb = cb[None, :]
    if cb.ndim != 2 or cb.shape[0] != rows:
        raise ValueError("cand_blocks must be [rows, n_cand]")
    idx = np.empty((rows, k), dtype=np.int32)
    val = np.empty((rows, k), dtype=np.float32)
    rc = _load().lt_oracle_topk_candidates(_ptr(s), _ptr(ln), rows, stride, int(block), _ptr(cb),
                                           cb.shape[1], int(k), _ptr(idx), _ptr(val),
                                           int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError("lt_oracle_topk_candidates: invalid argument")
    return idx, val
