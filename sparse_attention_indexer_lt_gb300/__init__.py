"""GB300-native indexer top-k (Lightning TopK) -- Python binding.

Thin ``ctypes`` binding of ``liblt_topk.so`` (see ``include/lt_topk.h``). It
only checks and marshals arguments: device pointers, sizes and the current
CUDA stream go to the C ABI, and every step of the selection runs in the
library's sm_103a kernels. There is no CPU path: if the library is missing or
the tensors are not on a CUDA device, the call raises.

    idx, val = topk(scores, lengths, k=512)
    idx, val, blocks = topk_blocked(scores, lengths, block=8, k_blocks=2048, k=512)

Scores may be float32 or bfloat16 (the bf16 entry points); values come back
as float32 either way (a bf16 score widens to fp32 exactly).
"""
from __future__ import annotations

import ctypes
from pathlib import Path

import torch

__all__ = ["topk", "topk_blocked", "topk_candidates", "compress", "compress_decode", "plan", "DTYPE_F32", "DTYPE_BF16", "load", "library_path", "LtError", "NUM_COUNTERS",
           "status_string", "version", "PlanInfo", "KERNEL_AUTO", "KERNEL_RESIDENT", "KERNEL_STREAM",
           "KERNEL_LISTED", "plan_candidates"]

_LIB_PATH = Path(__file__).resolve().parent / "liblt_topk.so"
_lib = None
NUM_COUNTERS = 7
DTYPE_F32, DTYPE_BF16 = 0, 1
KERNEL_AUTO, KERNEL_RESIDENT, KERNEL_STREAM, KERNEL_LISTED = 0, 1, 2, 3
_KERNEL_NAMES = {KERNEL_RESIDENT: "resident", KERNEL_STREAM: "stream", KERNEL_LISTED: "listed"}


class PlanInfo(ctypes.Structure):
    """Mirror of lt_plan_info."""
    _fields_ = [("kernel", ctypes.c_int32), ("cluster_size", ctypes.c_int32),
                ("threads_per_cta", ctypes.c_int32), ("smem_bytes", ctypes.c_int32),
                ("grid_ctas", ctypes.c_int32), ("ring_stages", ctypes.c_int32),
                ("one_round", ctypes.c_int32)]


class LtError(RuntimeError):
    """A non-zero lt_status from the library."""

    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status_string(status)} (status {status})")
        self.status = status


def library_path() -> Path:
    return _LIB_PATH


def load() -> ctypes.CDLL:
    """Load liblt_topk.so (built in-tree by ``build.build()``); raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not _LIB_PATH.exists():
        raise RuntimeError(
            f"{_LIB_PATH} is not built; run `python -m sparse_attention_indexer_lt_gb300.build` "
            "(needs nvcc) -- there is no fallback implementation")
    lib = ctypes.CDLL(str(_LIB_PATH))
    i32, i64, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
    lib.lt_topk.argtypes = [vp, vp, i32, i64, i32, vp, vp, vp]
    lib.lt_topk.restype = ctypes.c_int
    lib.lt_topk_ex.argtypes = [vp, i32, vp, i32, i64, i32, vp, vp, i32, i32, i32, i32, vp, vp, vp]
    lib.lt_topk_ex.restype = ctypes.c_int
    lib.lt_topk_blocked.argtypes = [vp, vp, i32, i64, i32, i32, i32, vp, vp, vp, vp]
    lib.lt_topk_blocked.restype = ctypes.c_int
    lib.lt_topk_blocked_ex.argtypes = [vp, i32, vp, i32, i64, i32, i32, i32, vp, vp, vp, i32, i32, i32, vp,
                                       vp, vp]
    lib.lt_topk_blocked_ex.restype = ctypes.c_int
    lib.lt_topk_candidates.argtypes = [vp, vp, i32, i64, i32, vp, i32, i32, vp, vp, vp]
    lib.lt_topk_candidates.restype = ctypes.c_int
    lib.lt_topk_candidates_ex.argtypes = [vp, i32, vp, i32, i64, i32, vp, i32, i32, vp, vp, i32, i32, i32,
                                          vp, vp, vp]
    lib.lt_topk_candidates_ex.restype = ctypes.c_int
    for name in ("lt_topk_bf16", "lt_topk_blocked_bf16", "lt_topk_candidates_bf16"):
        f = getattr(lib, name)
        f.argtypes = getattr(lib, name[:-5]).argtypes
        f.restype = ctypes.c_int
    lib.lt_topk_plan.argtypes = [i32, i64, i32, i32, i32, i32, i32, i32, i32, i32, vp]
    lib.lt_topk_plan.restype = ctypes.c_int
    lib.lt_topk_candidates_plan.argtypes = [i32, i64, i32, i32, i32, i32, i32, i32, i32, i32, vp]
    lib.lt_topk_candidates_plan.restype = ctypes.c_int
    lib.lt_status_string.argtypes = [ctypes.c_int]
    lib.lt_status_string.restype = ctypes.c_char_p
    lib.lt_compress.argtypes = [vp, vp, vp, vp, i32, i64, i32, i32, vp, i32, vp]
    lib.lt_compress.restype = ctypes.c_int
    lib.lt_compress_decode.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, vp, i32, vp]
    lib.lt_compress_decode.restype = ctypes.c_int
    lib.lt_test_inject.argtypes = [i32, i32]
    lib.lt_test_inject.restype = ctypes.c_int
    lib.lt_version.argtypes = []
    lib.lt_version.restype = i32
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().lt_status_string(int(status)).decode()


def version() -> int:
    return int(load().lt_version())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


_DTYPES = {torch.float32: DTYPE_F32, torch.bfloat16: DTYPE_BF16}


def _device_of(scores: torch.Tensor) -> torch.device:
    """The device that runs the call: the scores' own, or for pinned host
    scores (read by the kernel over the host link) the current one."""
    return scores.device if scores.is_cuda else torch.device("cuda", torch.cuda.current_device())


def _check_scores(scores: torch.Tensor):
    if not isinstance(scores, torch.Tensor) or not (scores.is_cuda or scores.is_pinned()):
        raise TypeError("scores must be a CUDA tensor or a pinned host tensor")
    if scores.dtype not in _DTYPES:
        raise TypeError("scores must be float32 or bfloat16")
    if scores.dim() != 2:
        raise ValueError("scores must be 2-D [rows, positions]")
    rows, n = scores.shape
    if n < 1:
        raise ValueError("scores must have at least one position per row")
    if rows > 0 and scores.stride(1) != 1:
        raise ValueError("scores rows must be contiguous (stride(1) == 1)")
    if rows > 1 and scores.stride(0) != n:
        raise ValueError("scores must have contiguous rows (stride(0) == number of positions)")
    return rows, n


def _usable(t: torch.Tensor, device: torch.device) -> bool:
    """On the call's device, or page-locked host memory the kernels reach over the host link."""
    return t.device == device or (t.device.type == "cpu" and t.is_pinned())


def _check_lengths(lengths, rows, device):
    if lengths is None:
        return None
    if not isinstance(lengths, torch.Tensor) or not _usable(lengths, device):
        raise TypeError("lengths must be a tensor on the scores' device or in pinned host memory")
    if lengths.dtype != torch.int32 or lengths.numel() != rows or not lengths.is_contiguous():
        raise ValueError("lengths must be a contiguous int32 tensor with one entry per row")
    return lengths


def _out(t, shape, dtype, device, name):
    if t is None:
        return torch.empty(shape, dtype=dtype, device=device)
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not _usable(t, device) or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {tuple(shape)} on {device} "
                         "or in pinned host memory")
    return t


def _counters(c, device):
    if c is None:
        return None
    if c.dtype != torch.int32 or c.numel() < NUM_COUNTERS or c.device != device:
        raise ValueError(f"counters must be an int32 tensor with >= {NUM_COUNTERS} entries on {device}")
    return c


def topk(scores: torch.Tensor, lengths: torch.Tensor | None = None, k: int = 512, *,
         out_idx: torch.Tensor | None = None, out_val: torch.Tensor | None = None,
         with_values: bool = True, force_cluster: int = 0, force_threads: int = 0,
         force_exact: bool = False, force_kernel: int = KERNEL_AUTO,
         counters: torch.Tensor | None = None, trace: torch.Tensor | None = None,
         stream: torch.cuda.Stream | None = None):
    """Per-row top-k by (score desc, index asc) of float32 or bfloat16 scores; returns
    (idx int32 [rows, k], val float32 [rows, k] or None)."""
    lib = load()
    rows, n = _check_scores(scores)
    dev = _device_of(scores)
    lengths = _check_lengths(lengths, rows, dev)
    out_idx = _out(out_idx, (rows, k), torch.int32, dev, "out_idx")
    if with_values:
        out_val = _out(out_val, (rows, k), torch.float32, dev, "out_val")
    else:
        out_val = None
    counters = _counters(counters, dev)
    with torch.cuda.device(dev):
        s = (stream or torch.cuda.current_stream(dev)).cuda_stream
        st = lib.lt_topk_ex(_ptr(scores), _DTYPES[scores.dtype], _ptr(lengths), rows, max(n, 1), int(k), _ptr(out_idx),
                            _ptr(out_val), int(force_cluster), int(force_threads),
                            int(bool(force_exact)), int(force_kernel), _ptr(counters), _ptr(trace),
                            ctypes.c_void_p(s))
    if st != 0:
        raise LtError("lt_topk", st)
    return out_idx, out_val


def topk_blocked(scores: torch.Tensor, lengths: torch.Tensor | None = None, block: int = 8,
                 k_blocks: int = 2048, k: int = 512, *, out_idx: torch.Tensor | None = None,
                 out_val: torch.Tensor | None = None, out_blocks: torch.Tensor | None = None,
                 with_values: bool = True, with_blocks: bool = True, force_cluster: int = 0,
                 force_threads: int = 0, force_exact: bool = False,
                 counters: torch.Tensor | None = None, trace: torch.Tensor | None = None,
                 stream: torch.cuda.Stream | None = None):
    """Two-level top-k; returns (idx [rows, k], val [rows, k] or None, blocks [rows, k_blocks] or None)."""
    lib = load()
    rows, n = _check_scores(scores)
    dev = _device_of(scores)
    lengths = _check_lengths(lengths, rows, dev)
    out_idx = _out(out_idx, (rows, k), torch.int32, dev, "out_idx")
    out_val = _out(out_val, (rows, k), torch.float32, dev, "out_val") if with_values else None
    out_blocks = _out(out_blocks, (rows, k_blocks), torch.int32, dev, "out_blocks") if with_blocks else None
    counters = _counters(counters, dev)
    with torch.cuda.device(dev):
        s = (stream or torch.cuda.current_stream(dev)).cuda_stream
        st = lib.lt_topk_blocked_ex(_ptr(scores), _DTYPES[scores.dtype], _ptr(lengths), rows, max(n, 1), int(block),
                                    int(k_blocks), int(k), _ptr(out_idx), _ptr(out_val),
                                    _ptr(out_blocks), int(force_cluster), int(force_threads),
                                    int(bool(force_exact)), _ptr(counters), _ptr(trace), ctypes.c_void_p(s))
    if st != 0:
        raise LtError("lt_topk_blocked", st)
    return out_idx, out_val, out_blocks


def topk_candidates(scores: torch.Tensor, cand_blocks: torch.Tensor, lengths: torch.Tensor | None = None,
                    block: int = 8, k: int = 512, *, out_idx: torch.Tensor | None = None,
                    out_val: torch.Tensor | None = None, with_values: bool = True, force_cluster: int = 0,
                    force_threads: int = 0, force_exact: bool = False,
                    counters: torch.Tensor | None = None, trace: torch.Tensor | None = None,
                    stream: torch.cuda.Stream | None = None):
    """Top-k among the positions of the listed blocks (cand_blocks int32 [rows, n_cand] on the same
    device; ids outside the row's blocks are ignored, repeats count once); returns
    (idx [rows, k], val [rows, k] or None)."""
    lib = load()
    rows, n = _check_scores(scores)
    dev = _device_of(scores)
    lengths = _check_lengths(lengths, rows, dev)
    if (not isinstance(cand_blocks, torch.Tensor) or not _usable(cand_blocks, dev)
            or cand_blocks.dtype != torch.int32 or cand_blocks.dim() != 2 or cand_blocks.shape[0] != rows
            or not cand_blocks.is_contiguous()):
        raise ValueError("cand_blocks must be a contiguous int32 tensor [rows, n_cand] on the scores' device "
                         "or in pinned host memory")
    out_idx = _out(out_idx, (rows, k), torch.int32, dev, "out_idx")
    out_val = _out(out_val, (rows, k), torch.float32, dev, "out_val") if with_values else None
    counters = _counters(counters, dev)
    with torch.cuda.device(dev):
        s = (stream or torch.cuda.current_stream(dev)).cuda_stream
        st = lib.lt_topk_candidates_ex(_ptr(scores), _DTYPES[scores.dtype], _ptr(lengths), rows, max(n, 1), int(block),
                                       _ptr(cand_blocks), int(cand_blocks.shape[1]), int(k), _ptr(out_idx),
                                       _ptr(out_val), int(force_cluster), int(force_threads),
                                       int(bool(force_exact)), _ptr(counters), _ptr(trace),
                                       ctypes.c_void_p(s))
    if st != 0:
        raise LtError("lt_topk_candidates", st)
    return out_idx, out_val


def _check_kv(name, t, device, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.device != device or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor on {device}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}")


def compress(kv: torch.Tensor, score: torch.Tensor, bias: torch.Tensor, ratio: int,
             lengths: torch.Tensor | None = None, *, out: torch.Tensor | None = None,
             stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """Fused KV compressor: kv, score [rows, T, d] (float32 or bfloat16, the same), bias float32
    [ratio, d]; returns out [rows, T // ratio, d] in kv's dtype, with block g of row r written when
    g < L_r // ratio (see include/lt_compress.h)."""
    lib = load()
    if kv.dim() != 3 or score.shape != kv.shape or score.dtype != kv.dtype or kv.dtype not in _DTYPES:
        raise ValueError("kv and score must be [rows, T, d] tensors of one dtype (float32 or bfloat16)")
    dev = kv.device
    _check_kv("kv", kv, dev)
    _check_kv("score", score, dev)
    _check_kv("bias", bias, dev, torch.float32)
    rows, T, d = kv.shape
    if tuple(bias.shape) != (ratio, d):
        raise ValueError(f"bias must be [{ratio}, {d}]")
    lengths = _check_lengths(lengths, rows, dev)
    out = _out(out, (rows, T // ratio, d), kv.dtype, dev, "out")
    with torch.cuda.device(dev):
        s = (stream or torch.cuda.current_stream(dev)).cuda_stream
        st = lib.lt_compress(_ptr(kv), _ptr(score), _ptr(bias), _ptr(lengths), rows, max(T, 1), d, int(ratio),
                             _ptr(out), _DTYPES[kv.dtype], ctypes.c_void_p(s))
    if st != 0:
        raise LtError("lt_compress", st)
    return out


def compress_decode(kv_new: torch.Tensor, score_new: torch.Tensor, bias: torch.Tensor, ring_kv: torch.Tensor,
                    ring_score: torch.Tensor, pos: torch.Tensor, out: torch.Tensor, *,
                    stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """One decode step of the compressor: kv_new, score_new [seqs, d]; rings [seqs, ratio, d]
    (updated in place); pos int32 [seqs]; out [seqs, d] written for the sequences whose new token
    completes a block."""
    lib = load()
    dev = kv_new.device
    seqs, d = kv_new.shape
    ratio = ring_kv.shape[1]
    for n, t in (("kv_new", kv_new), ("score_new", score_new), ("ring_kv", ring_kv), ("ring_score", ring_score),
                 ("out", out)):
        _check_kv(n, t, dev, kv_new.dtype)
    _check_kv("bias", bias, dev, torch.float32)
    _check_kv("pos", pos, dev, torch.int32)
    if (kv_new.dtype not in _DTYPES or score_new.shape != (seqs, d) or ring_kv.shape != (seqs, ratio, d)
            or ring_score.shape != (seqs, ratio, d) or tuple(bias.shape) != (ratio, d) or out.shape != (seqs, d)
            or pos.numel() != seqs):
        raise ValueError("compress_decode: inconsistent shapes or dtype")
    with torch.cuda.device(dev):
        s = (stream or torch.cuda.current_stream(dev)).cuda_stream
        st = lib.lt_compress_decode(_ptr(kv_new), _ptr(score_new), _ptr(bias), _ptr(ring_kv), _ptr(ring_score),
                                    _ptr(pos), seqs, d, int(ratio), _ptr(out), _DTYPES[kv_new.dtype],
                                    ctypes.c_void_p(s))
    if st != 0:
        raise LtError("lt_compress_decode", st)
    return out


def plan(rows: int, row_stride: int, k: int, *, blocked: bool = False, block: int = 8,
         k_blocks: int = 2048, force_cluster: int = 0, force_threads: int = 0,
         force_kernel: int = KERNEL_AUTO, aligned: bool = True, device: int | None = None) -> dict:
    """The launch the planner would make: {'kernel', 'cluster', 'threads', 'smem', 'grid', 'stages',
    'one_round'}."""
    lib = load()
    info = PlanInfo()
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        st = lib.lt_topk_plan(int(rows), int(row_stride), int(k), int(bool(blocked)), int(block),
                              int(k_blocks), int(force_cluster), int(force_threads), int(force_kernel),
                              int(bool(aligned)), ctypes.byref(info))
    if st != 0:
        raise LtError("lt_topk_plan", st)
    return {"kernel": _KERNEL_NAMES.get(info.kernel, str(info.kernel)), "cluster": info.cluster_size,
            "threads": info.threads_per_cta, "smem": info.smem_bytes, "grid": info.grid_ctas,
            "stages": info.ring_stages, "one_round": bool(info.one_round)}


def plan_candidates(rows: int, row_stride: int, block: int, n_cand: int, k: int, *,
                    dtype: torch.dtype = torch.float32, force_cluster: int = 0, force_threads: int = 0,
                    force_exact: bool = False, aligned: bool = True, device: int | None = None) -> dict:
    """The launch topk_candidates would make ('kernel' is 'listed' for the kernel
    that reads only the listed blocks); keys as for plan()."""
    lib = load()
    info = PlanInfo()
    if dtype not in _DTYPES:
        raise ValueError(f"scores must be float32 or bfloat16, got {dtype}")
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        st = lib.lt_topk_candidates_plan(int(rows), int(row_stride), int(block), int(n_cand), int(k),
                                         _DTYPES[dtype], int(force_cluster), int(force_threads),
                                         int(bool(force_exact)), int(bool(aligned)), ctypes.byref(info))
    if st != 0:
        raise LtError("lt_topk_candidates_plan", st)
    return {"kernel": _KERNEL_NAMES.get(info.kernel, str(info.kernel)), "cluster": info.cluster_size,
            "threads": info.threads_per_cta, "smem": info.smem_bytes, "grid": info.grid_ctas,
            "stages": info.ring_stages, "one_round": bool(info.one_round)}
