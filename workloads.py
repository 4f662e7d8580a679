"""Seeded synthetic inputs for the indexer top-k (shared by the tests and the bench).

This module draws random numbers and lays them out; it holds none of the
selection arithmetic. Both the CUDA path and the CPU oracle consume what it
returns, so parity never depends on it.

Workloads (the pages give the Lightning TopK figure for a context of a
million tokens at batch size 1, and CSA compresses 4:1, so one row at 1M
tokens has 262,144 compressed positions; the rest are the batched shapes the
deployment implies):

  c1_single_4096     1 x 4096, N(0,1) rounded to bf16 (ties occur), k=512
  c2_decode_262144   1 x 262144, N(0,1) -> bf16, plus U(2,6) on 1% of the
                     positions (2621, chosen without replacement), k=512
  c3_ragged_64       64 x 262144, lengths uniform in [2048, 262144],
                     N(0,1) -> bf16, k=512
  c4_prefill_4096    4096 x 32768, row r has length floor((126976 + r + 1)/4),
                     N(0,1) fp32, k=512
  c5_blocked_16      16 x 262144, N(0,1) fp32, blocks of 8, top-2048 blocks,
                     then top-512 positions inside them
  c6_listed_16       the c5 rows; per row 2048 distinct 8-blocks drawn
                     uniformly (listed_blocks), top-512 among their positions

RNG: ``torch.Generator('cpu').manual_seed(seed)``; draw order lengths, scores,
tail positions, tail addends.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    rows: int
    row_stride: int
    k: int
    blocked: bool = False
    block: int = 8
    k_blocks: int = 2048
    description: str = ""


CONFIGS = {
    "c1_single_4096": Workload("c1_single_4096", 1, 4096, 512,
                               description="1 row x 4096, N(0,1)->bf16, k=512"),
    "c2_decode_262144": Workload("c2_decode_262144", 1, 262144, 512,
                                 description="BS=1 decode at 1M tokens (262144 compressed), "
                                             "N(0,1)->bf16 + U(2,6) on 1%, k=512"),
    "c3_ragged_64": Workload("c3_ragged_64", 64, 262144, 512,
                             description="64 ragged rows, L~U[2048,262144], N(0,1)->bf16, k=512"),
    "c4_prefill_4096": Workload("c4_prefill_4096", 4096, 32768, 512,
                                description="causal prefill chunk, 4096 rows x 32768, "
                                            "L_r=floor((126977+r)/4), N(0,1) fp32, k=512"),
    "c5_blocked_16": Workload("c5_blocked_16", 16, 262144, 512, blocked=True, block=8,
                              k_blocks=2048,
                              description="two-level: 16 rows x 262144 fp32, top-2048 of "
                                          "32768 8-blocks, then top-512"),
    "c6_listed_16": Workload("c6_listed_16", 16, 262144, 512, block=8, k_blocks=2048,
                             description="listed candidates: the c5 rows, top-512 among 2048 "
                                         "given 8-blocks per row"),
}


def _bf16(x: torch.Tensor) -> torch.Tensor:
    # fp32 -> bf16 round-to-nearest-even -> fp32 (layout of the inputs, not the method)
    return x.to(torch.bfloat16).float()


def make(name: str, seed: int = 0):
    """Return (scores float32 [rows, stride] CPU, lengths int32 [rows] CPU or None, workload)."""
    w = CONFIGS[name]
    g = torch.Generator("cpu").manual_seed(seed)
    lengths = None
    if name == "c1_single_4096":
        scores = _bf16(torch.randn(w.rows, w.row_stride, generator=g))
    elif name == "c2_decode_262144":
        scores = _bf16(torch.randn(w.rows, w.row_stride, generator=g))
        n_tail = round(0.01 * w.row_stride)
        pos = torch.randperm(w.row_stride, generator=g)[:n_tail]
        add = torch.rand(n_tail, generator=g) * 4.0 + 2.0
        scores[0, pos] += add  # fp32 sum, not re-rounded
    elif name == "c3_ragged_64":
        lengths = torch.randint(2048, w.row_stride + 1, (w.rows,), generator=g, dtype=torch.int32)
        scores = _bf16(torch.randn(w.rows, w.row_stride, generator=g))
    elif name == "c4_prefill_4096":
        r = torch.arange(w.rows, dtype=torch.int64)
        lengths = ((126976 + r + 1) // 4).to(torch.int32)
        scores = torch.randn(w.rows, w.row_stride, generator=g)
    elif name in ("c5_blocked_16", "c6_listed_16"):
        scores = torch.randn(w.rows, w.row_stride, generator=g)
    else:  # pragma: no cover
        raise KeyError(name)
    return scores.contiguous(), lengths, w


def random_rows(rows: int, stride: int, seed: int, *, dist: str = "normal",
                lengths: str | None = None, min_len: int = 0):
    """Small seeded inputs for parity tests.

    dist: "normal" (fp32), "bf16" (ties), "coarse" (8 distinct values: heavy ties),
          "equal" (all 1.0), "asc"/"desc" (strictly monotone), "special" (mix of
          +-inf, +-0, denormals, NaN and ordinary numbers), "tail" (bf16 + U(2,6) on 1%).
    lengths: None (all full) or "ragged" (uniform in [min_len, stride]).
    """
    g = torch.Generator("cpu").manual_seed(seed)
    ln = None
    if lengths == "ragged":
        ln = torch.randint(min_len, stride + 1, (rows,), generator=g, dtype=torch.int32)
    if dist == "normal":
        x = torch.randn(rows, stride, generator=g)
    elif dist == "bf16":
        x = _bf16(torch.randn(rows, stride, generator=g))
    elif dist == "coarse":
        x = torch.randint(-4, 4, (rows, stride), generator=g).float() * 0.5
    elif dist == "equal":
        x = torch.ones(rows, stride)
    elif dist == "asc":
        x = torch.arange(stride, dtype=torch.float32).repeat(rows, 1) * 1e-3
    elif dist == "desc":
        x = -torch.arange(stride, dtype=torch.float32).repeat(rows, 1) * 1e-3
    elif dist == "special":
        pool = torch.tensor([
            float("inf"), float("-inf"), 0.0, -0.0, float("nan"), -float("nan"),
            1e-45, -1e-45, 1.17549435e-38, -1.17549435e-38, 3.0e38, -3.0e38,
            1.0, -1.0, 2.5, -2.5,
        ], dtype=torch.float32)
        pick = torch.randint(0, pool.numel(), (rows, stride), generator=g)
        x = pool[pick]
        # a second NaN payload, so value copies are checked bit for bit
        nanmask = torch.rand(rows, stride, generator=g) < 0.02
        xi = x.view(torch.int32)
        xi[nanmask] = 0x7FC00123
    elif dist == "tail":
        x = _bf16(torch.randn(rows, stride, generator=g))
        n_tail = max(1, round(0.01 * stride))
        for r in range(rows):
            pos = torch.randperm(stride, generator=g)[:n_tail]
            x[r, pos] += torch.rand(n_tail, generator=g) * 4.0 + 2.0
    else:
        raise KeyError(dist)
    return x.contiguous(), ln


def to_bf16(scores: torch.Tensor) -> torch.Tensor:
    """The bf16 form of a workload's scores (round to nearest even; exact for the
    bf16-rounded configs). A layout of the inputs, not part of the method."""
    return scores.to(torch.bfloat16).contiguous()


def bf16_bits(t: torch.Tensor):
    """The uint16 bit patterns of a CPU bf16 tensor, as a numpy array."""
    import numpy as np
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def random_bf16_special(rows: int, stride: int, seed: int):
    """bf16 bit patterns drawn from a pool of special values (+-0, +-inf,
    subnormals, NaNs with payloads, the largest finite) and ordinary numbers."""
    g = torch.Generator("cpu").manual_seed(seed)
    pool = torch.tensor([0x0000, 0x8000, 0x7F80, 0xFF80, 0x0001, 0x8001, 0x007F, 0x7FC0, 0xFFC1, 0x7FA0,
                         0x7F7F, 0xFF7F, 0x3F80, 0xBF80, 0x4049, 0xC0A0, 0x3F81, 0x3F80], dtype=torch.int32)
    pick = torch.randint(0, pool.numel(), (rows, stride), generator=g)
    return pool[pick].to(torch.int16).view(torch.bfloat16).contiguous()


@dataclass(frozen=True)
class CompressWorkload:
    name: str
    rows: int
    tokens: int
    dim: int
    ratio: int
    description: str = ""


# The compressor at a million-token context, prefill: one row of 2^20 tokens,
# 512 channels, bf16 KV and scores; 4:1 (CSA) and 128:1 (HCA).
COMPRESS_CONFIGS = {
    "compress_csa_1m": CompressWorkload("compress_csa_1m", 1, 1 << 20, 512, 4,
                                        "1 row x 2^20 tokens x 512 channels, bf16, 4:1"),
    "compress_hca_1m": CompressWorkload("compress_hca_1m", 1, 1 << 20, 512, 128,
                                        "1 row x 2^20 tokens x 512 channels, bf16, 128:1"),
}


def compress_inputs(rows: int, tokens: int, dim: int, ratio: int, seed: int, device="cpu",
                    dtype=torch.float32, score_scale: float = 1.0):
    """Seeded compressor inputs: kv ~ N(0,1), score ~ N(0, score_scale^2) (gate
    logits), bias ~ N(0, 0.25) float32 [ratio, dim]. On a CUDA device the
    device's own generator draws them (large inputs); the values depend only
    on the seed and the device type."""
    g = torch.Generator(device).manual_seed(seed)
    kv = torch.randn(rows, tokens, dim, generator=g, device=device)
    sc = torch.randn(rows, tokens, dim, generator=g, device=device) * score_scale
    bias = torch.randn(ratio, dim, generator=g, device=device) * 0.5
    return kv.to(dtype).contiguous(), sc.to(dtype).contiguous(), bias.float().contiguous()


def read_bytes(lengths, rows: int, stride: int) -> int:
    """Bytes a read-once pass touches: 4 bytes per valid position."""
    if lengths is None:
        return 4 * rows * stride
    return 4 * int(torch.clamp(lengths.to(torch.int64), 0, stride).sum().item())


def l2_rotation_copies(bytes_per_copy: int, l2_bytes: int) -> int:
    """Number of distinct input copies whose total exceeds twice the L2 size."""
    return max(1, math.ceil(2 * l2_bytes / max(1, bytes_per_copy)) + 1)


def listed_blocks(name: str, seed: int = 0) -> torch.Tensor:
    """The block list of a listed-candidates workload: per row, k_blocks distinct
    block ids drawn uniformly from the row's blocks, ascending (the form an
    earlier layer publishes; which blocks does not change the work)."""
    w = CONFIGS[name]
    g = torch.Generator("cpu").manual_seed(1000 + seed)
    nb = (w.row_stride + w.block - 1) // w.block
    rows = [torch.sort(torch.randperm(nb, generator=g)[:w.k_blocks]).values for _ in range(w.rows)]
    return torch.stack(rows).to(torch.int32).contiguous()
