"""Seeded random cases over every entry point, against the oracle bit for bit.

Each case draws its shape (rows, stride, ragged or full lengths), its score
distribution, k, the score type and, for the two-level and listed calls, the
block size, k_blocks and the block lists from a fixed seed, so a failing case
replays exactly (its parameters are in the assertion message). The shapes
cross the planner's boundaries: one and many CTAs per row, one and several
register rounds, clusters of 1 to 16, rows shorter than k.
"""
import numpy as np
import pytest
import torch

import workloads
from _gpu import parity_blocked, parity_bf16, parity_candidates, parity_topk

pytestmark = pytest.mark.gpu

DISTS = ["normal", "bf16", "coarse", "special", "equal", "asc", "desc", "tail"]
KS = [1, 5, 64, 300, 512, 1024, 2048]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_attention_indexer_lt_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _case(i):
    rng = np.random.default_rng(7919 * i + 17)
    rows = int(rng.choice([1, 2, 3, 16, 64, 200, 600]))
    max_stride = max(1, 3_000_000 // rows)
    stride = int(min(max_stride, rng.choice([1, 7, 100, 513, 4096, 9000, 40000, 131072, 262144])))
    dist = str(rng.choice(DISTS))
    k = int(rng.choice(KS))
    ragged = bool(rng.integers(0, 2))
    bf16 = bool(rng.integers(0, 4) == 0) and dist not in ("special",)
    seed = int(rng.integers(0, 1 << 30))
    return rng, rows, stride, dist, k, ragged, bf16, seed


def _inputs(rows, stride, dist, ragged, seed):
    S, L = workloads.random_rows(rows, stride, seed=seed, dist=dist, lengths="ragged" if ragged else None)
    return S, (None if L is None else L.numpy())


def _lists(rng, rows, nblocks, n):
    out = []
    for _ in range(rows):
        m = min(n, nblocks)
        ids = rng.choice(nblocks, size=m, replace=False).astype(np.int32)
        extra = np.concatenate([ids[: int(rng.integers(0, 4))], np.full(int(rng.integers(0, 3)), -1, np.int32),
                                (nblocks + rng.integers(0, 9, size=int(rng.integers(0, 2)))).astype(np.int32)])
        out.append(rng.permutation(np.concatenate([ids, extra]).astype(np.int32)))
    width = max(1, max(len(r) for r in out))
    return np.stack([np.pad(r, (0, width - len(r)), constant_values=-1) for r in out]).astype(np.int32)


@pytest.mark.parametrize("i", range(96))
def test_random_topk(i):
    rng, rows, stride, dist, k, ragged, bf16, seed = _case(i)
    S, L = _inputs(rows, stride, dist, ragged, seed)
    what = f"topk case {i}: rows={rows} stride={stride} dist={dist} k={k} ragged={ragged} bf16={bf16}"
    if bf16:
        parity_bf16(S.to(torch.bfloat16), L, k, what=what)
    else:
        parity_topk(S.numpy(), L, k, what=what)


@pytest.mark.parametrize("i", range(64))
def test_random_blocked(i):
    rng, rows, stride, dist, k, ragged, bf16, seed = _case(1000 + i)
    block = int(rng.choice([4, 8, 16, 32]))
    k_blocks = int(rng.choice([1, 16, 300, 1024, 2048]))
    S, L = _inputs(rows, stride, dist, ragged, seed)
    what = (f"blocked case {i}: rows={rows} stride={stride} dist={dist} block={block} "
            f"k_blocks={k_blocks} k={k} ragged={ragged} bf16={bf16}")
    if bf16:
        parity_bf16(S.to(torch.bfloat16), L, k, what=what, kind="blocked", block=block, k_blocks=k_blocks)
    else:
        parity_blocked(S.numpy(), L, block, k_blocks, k, what=what)


@pytest.mark.parametrize("i", range(64))
def test_random_candidates(i):
    rng, rows, stride, dist, k, ragged, bf16, seed = _case(2000 + i)
    block = int(rng.choice([4, 8, 16, 32]))
    nblocks = (stride + block - 1) // block
    n = int(rng.choice([1, 10, 300, 2048, 4096]))
    S, L = _inputs(rows, stride, dist, ragged, seed)
    cand = _lists(rng, rows, nblocks, n)
    what = (f"candidates case {i}: rows={rows} stride={stride} dist={dist} block={block} n={n} k={k} "
            f"ragged={ragged} bf16={bf16}")
    if bf16:
        parity_bf16(S.to(torch.bfloat16), L, k, what=what, kind="candidates", block=block, cand=cand)
    else:
        parity_candidates(S.numpy(), L, cand, block, k, what=what)
