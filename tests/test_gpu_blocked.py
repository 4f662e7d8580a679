"""GPU parity of lt_topk_blocked (two-level selection) against the literal oracle."""
import numpy as np
import pytest
import torch

import workloads
from _gpu import counters, parity_blocked

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_attention_indexer_lt_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def test_blocked_workload_parity():
    S, L, w = workloads.make("c5_blocked_16")
    c = counters()
    parity_blocked(S.numpy(), None, w.block, w.k_blocks, w.k, what="c5", counters=c)
    cnt = c.cpu().numpy()
    assert cnt[0] == 2 * w.rows and cnt[1] == 0, cnt  # both stages, fast path


def test_blocked_workload_exact_path():
    S, L, w = workloads.make("c5_blocked_16")
    parity_blocked(S[:4].numpy(), None, w.block, w.k_blocks, w.k, what="c5/exact", force_exact=True)


@pytest.mark.parametrize("ft", [256, 512])
@pytest.mark.parametrize("block", [4, 8, 16, 32])
@pytest.mark.parametrize("dist", ["normal", "coarse", "special", "equal", "asc"])
def test_blocked_small(block, dist, ft):
    S, L = workloads.random_rows(3, 30000, seed=block * 7 + len(dist), dist=dist, lengths="ragged")
    for kb, k in [(16, 512), (300, 100), (2048, 512), (64, 64)]:
        parity_blocked(S.numpy(), L.numpy(), block, kb, k, what=f"{dist} B={block} kb={kb} k={k} t={ft}",
                       force_threads=ft)


@pytest.mark.parametrize("ft", [256, 512])
@pytest.mark.parametrize("fc", [1, 2, 4, 8, 16])
def test_blocked_forced_plans(fc, ft):
    S, L = workloads.random_rows(2, 262144, seed=31, dist="bf16", lengths="ragged", min_len=1)
    parity_blocked(S.numpy(), L.numpy(), 8, 2048, 512, what=f"cluster {fc}x{ft}", force_cluster=fc,
                   force_threads=ft)
    parity_blocked(S.numpy(), L.numpy(), 8, 200, 512, what=f"cluster {fc}x{ft} kb<k", force_cluster=fc,
                   force_threads=ft)


@pytest.mark.parametrize("ft", [256, 512])
def test_blocked_workload_both_cta_shapes(ft):
    S, L, w = workloads.make("c5_blocked_16")
    parity_blocked(S.numpy(), None, w.block, w.k_blocks, w.k, what=f"c5/{ft}", force_threads=ft)


def test_blocked_edge_lengths():
    stride = 5000
    lens = [0, 1, 7, 8, 9, 15, 16, 17, 100, 4095, 4096, 4999, 5000]
    S, _ = workloads.random_rows(len(lens), stride, seed=33, dist="bf16")
    S = S.numpy().copy()
    for r, l in enumerate(lens):
        S[r, l:] = np.inf
    for kb, k in [(1, 8), (3, 20), (2048, 512)]:
        parity_blocked(S, np.array(lens, np.int32), 8, kb, k, what=f"edges kb={kb} k={k}")


def test_blocked_optional_outputs():
    import oracle
    import sparse_attention_indexer_lt_gb300 as lt
    S, _ = workloads.random_rows(2, 20000, seed=34, dist="normal")
    idx, val, blk = lt.topk_blocked(S.cuda(), None, 8, 100, 50, with_values=False, with_blocks=False)
    torch.cuda.synchronize()
    assert val is None and blk is None
    oi, _, _ = oracle.topk_blocked(S.numpy(), None, 8, 100, 50)
    assert np.array_equal(idx.cpu().numpy(), oi)
