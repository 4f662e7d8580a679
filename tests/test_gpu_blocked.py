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


def test_blocked_split_without_kept_blocks_runs_one_stage():
    """k_blocks >= k and no out_blocks: only the plain top-k group runs (one count
    per row), and its result still equals the literal two-level oracle."""
    import oracle
    import sparse_attention_indexer_lt_gb300 as lt
    S, L = workloads.random_rows(6, 50000, seed=35, dist="bf16", lengths="ragged", min_len=100)
    c = counters()
    idx, val, blk = lt.topk_blocked(S.cuda(), L.cuda(), 8, 2048, 512, with_blocks=False, counters=c)
    torch.cuda.synchronize()
    assert blk is None
    oi, ov, _ = oracle.topk_blocked(S.numpy(), L.numpy(), 8, 2048, 512)
    assert np.array_equal(idx.cpu().numpy(), oi)
    assert np.array_equal(val.cpu().numpy().view(np.uint32), ov.view(np.uint32))
    assert c.cpu().numpy()[0] + c.cpu().numpy()[1] == 6


@pytest.mark.parametrize("kb,k", [(2048, 512), (100, 512)])
def test_blocked_split_and_sequential_exact_paths(kb, k):
    """Forced streaming radix select in both the side-by-side (kb >= k) and the
    one-after-the-other (kb < k) launches."""
    S, L = workloads.random_rows(3, 90000, seed=36, dist="coarse", lengths="ragged", min_len=1)
    parity_blocked(S.numpy(), L.numpy(), 8, kb, k, what=f"exact kb={kb}", force_exact=True)
