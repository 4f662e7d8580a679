"""GPU parity of lt_topk_candidates (top-k among the positions of a given block
list) against the CPU oracle, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _gpu import counters, parity_candidates

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_attention_indexer_lt_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _random_lists(rng, rows, nblocks, n, pads=0, repeats=0, beyond=0):
    out = []
    for _ in range(rows):
        ids = rng.choice(nblocks, size=min(n, nblocks), replace=False).astype(np.int32)
        extra = [ids[:repeats], np.full(pads, -1, np.int32), nblocks + rng.integers(0, 50, size=beyond)]
        row = np.concatenate([ids] + [np.asarray(e, np.int32) for e in extra])
        out.append(rng.permutation(row))
    width = max(len(r) for r in out)
    return np.stack([np.pad(r, (0, width - len(r)), constant_values=-1) for r in out]).astype(np.int32)


def test_workload_lists_from_an_earlier_layer():
    """The c5 rows restricted to the blocks another score matrix (an earlier
    layer) kept: the cross-layer use."""
    S, _, w = workloads.make("c5_blocked_16")
    S_prev = workloads.make("c5_blocked_16", seed=1)[0]
    _, _, kept = oracle.topk_blocked(S_prev.numpy(), None, w.block, w.k_blocks, w.k)
    c = counters()
    parity_candidates(S.numpy(), None, kept, w.block, w.k, what="c5 rows, earlier layer's blocks", counters=c)
    cnt = c.cpu().numpy()
    assert cnt[0] == w.rows and cnt[1] == 0, cnt  # every row on the fast path


def test_own_kept_blocks_reproduce_the_two_level_result():
    S, L = workloads.random_rows(4, 60000, seed=41, dist="bf16", lengths="ragged", min_len=1)
    S = S.numpy()
    L = L.numpy()
    for kb, k in [(300, 100), (2048, 512), (64, 512)]:
        i2, v2, kept = oracle.topk_blocked(S, L, 8, kb, k)
        gi, gv = parity_candidates(S, L, kept, 8, k, what=f"kept kb={kb} k={k}")
        assert np.array_equal(gi, i2) and np.array_equal(gv.view(np.uint32), v2.view(np.uint32))


@pytest.mark.parametrize("ft", [0, 256, 512])
@pytest.mark.parametrize("block", [4, 8, 16, 32])
@pytest.mark.parametrize("dist", ["normal", "bf16", "coarse", "special", "equal"])
def test_small_lists(block, dist, ft):
    """ft 0: a cluster of CTAs per row shares each list; 512: one CTA per
    row; 256: the whole-row scan of the two-level kernel."""
    rng = np.random.default_rng(block * 31 + len(dist))
    stride = 30000
    S, L = workloads.random_rows(3, stride, seed=block + len(dist), dist=dist, lengths="ragged", min_len=0)
    nb = (stride + block - 1) // block
    for n, k in [(20, 64), (500, 512), (3000, 512), (nb, 2048)]:
        cand = _random_lists(rng, 3, nb, n, pads=5, repeats=7, beyond=3)
        parity_candidates(S.numpy(), L.numpy(), cand, block, k, what=f"{dist} B={block} n={n} k={k} t={ft}",
                          force_threads=ft)


@pytest.mark.parametrize("ft", [256, 512])
@pytest.mark.parametrize("fc", [1, 2, 4, 8, 16])
def test_forced_plans_and_exact_path(fc, ft):
    rng = np.random.default_rng(fc * 7 + ft)
    S, L = workloads.random_rows(2, 262144, seed=43, dist="bf16", lengths="ragged", min_len=1)
    nb = 262144 // 8
    cand = _random_lists(rng, 2, nb, 2048, pads=3)
    kw = dict(force_cluster=fc, force_threads=ft)
    parity_candidates(S.numpy(), L.numpy(), cand, 8, 512, what=f"cluster {fc}x{ft}", **kw)
    parity_candidates(S.numpy(), L.numpy(), cand, 8, 512, what=f"cluster {fc}x{ft} exact", force_exact=True, **kw)


@pytest.mark.parametrize("rows", [1, 5, 20, 40, 80])
def test_listed_rows_by_cluster_size(rows):
    """The automatic plan shares a row's list over clusters of 8, 4, 2 or 1
    CTAs as the row count grows (every cluster size once)."""
    rng = np.random.default_rng(rows)
    stride = 65536
    S, L = workloads.random_rows(rows, stride, seed=rows + 60, dist="bf16", lengths="ragged", min_len=stride // 4)
    cand = _random_lists(rng, rows, stride // 8, 2048, pads=9, repeats=40, beyond=2)
    c = counters()
    parity_candidates(S.numpy(), L.numpy(), cand, 8, 512, what=f"{rows} rows", counters=c)
    cnt = c.cpu().numpy()
    assert cnt[0] == rows and cnt[1] == 0, cnt
    parity_candidates(S.numpy(), L.numpy(), cand[:, :300], 8, 2048, what=f"{rows} rows, k > listed positions")


def test_empty_and_short_lists():
    S, L = workloads.random_rows(3, 5000, seed=44, dist="normal", lengths="ragged")
    none = np.full((3, 4), -1, np.int32)
    gi, gv = parity_candidates(S.numpy(), L.numpy(), none, 8, 16, what="only pads")
    assert np.all(gi == -1) and np.all(np.isneginf(gv))
    empty = np.zeros((3, 0), np.int32)
    gi, _ = parity_candidates(S.numpy(), L.numpy(), empty, 8, 16, what="n_cand = 0")
    assert np.all(gi == -1)
    one = np.array([[0], [3], [624]], np.int32)  # fewer candidate positions than k
    parity_candidates(S.numpy(), L.numpy(), one, 8, 64, what="one block each")


def test_unaligned_rows():
    rng = np.random.default_rng(45)
    S, L = workloads.random_rows(3, 40001, seed=45, dist="bf16", lengths="ragged")
    cand = _random_lists(rng, 3, (40001 + 7) // 8, 700)
    parity_candidates(S.numpy(), L.numpy(), cand, 8, 512, what="stride 40001")


@pytest.mark.parametrize("block", [4, 8])
def test_short_lists_on_rows_longer_than_a_bitmap(block):
    """A short list (the kernel that reads only the listed blocks) on rows of
    2^20 positions, more blocks than a bitmap of the row can hold: the unique
    ids come from a hash set; repeats, pads and ids past the row included."""
    rng = np.random.default_rng(51 + block)
    rows, stride = 3, 1 << 20
    S, L = workloads.random_rows(rows, stride, seed=52, dist="bf16", lengths="ragged", min_len=stride // 2)
    nb = stride // block
    n = (512 * 8 * 4 // block) // 2
    lists = _random_lists(rng, rows, nb, n, pads=7, repeats=n // 3, beyond=5)[:, : 512 * 8 * 4 // block]
    c = counters()
    parity_candidates(S.numpy(), L.numpy(), lists, block, 512, what=f"long rows, short list, block {block}",
                      counters=c)
    parity_candidates(S.numpy(), L.numpy(), lists, block, 2048, what=f"long rows, short list, k=2048, block {block}")


def test_long_lists_on_rows_longer_than_a_bitmap():
    """A long list (whole-row scan) on rows of 2^20 positions: every CTA of the
    row's cluster holds a bitmap of its own slice and the listed positions
    are summed over the cluster."""
    import sparse_attention_indexer_lt_gb300 as lt
    rng = np.random.default_rng(53)
    rows, stride, block = 2, 1 << 20, 8
    S, L = workloads.random_rows(rows, stride, seed=54, dist="tail", lengths="ragged", min_len=stride // 2)
    nb = stride // block
    lists = _random_lists(rng, rows, nb, 20000, pads=3, repeats=100, beyond=4)
    parity_candidates(S.numpy(), L.numpy(), lists, block, 512, what="long rows, long list")
    for fc in (4, 8, 16):
        parity_candidates(S.numpy(), L.numpy(), lists, block, 512, what=f"long rows, long list, cluster {fc}",
                          force_cluster=fc)
    # one CTA would need a bitmap of 131072 blocks: refused
    with pytest.raises(lt.LtError):
        lt.topk_candidates(S.cuda(), torch.as_tensor(lists).cuda(), L.cuda(), block, 512, force_cluster=1)


def test_listed_plan_query():
    """lt_topk_candidates_plan reports the launch the call makes."""
    import sparse_attention_indexer_lt_gb300 as lt
    pl = lt.plan_candidates(16, 262144, 8, 2048, 512)
    assert pl["kernel"] == "listed" and pl["cluster"] in (2, 4, 8) and pl["threads"] == 256, pl
    assert pl["grid"] == 16 * pl["cluster"], pl
    pl = lt.plan_candidates(200, 262144, 8, 2048, 512)
    assert pl["kernel"] == "listed" and pl["cluster"] == 1 and pl["threads"] == 512, pl
    pl = lt.plan_candidates(16, 262144, 8, 2048, 512, force_cluster=2)
    assert pl["kernel"] == "resident" and pl["cluster"] == 2, pl  # the whole-row scan
    pl = lt.plan_candidates(16, 262144, 8, 5000, 512)
    assert pl["kernel"] == "resident", pl  # longer than one register round of blocks
    pl = lt.plan_candidates(3, 1 << 20, 4, 100, 512)
    assert pl["kernel"] == "listed" and pl["cluster"] == 1, pl  # hash-set rows: one CTA each
