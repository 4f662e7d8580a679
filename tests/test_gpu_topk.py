"""GPU parity of lt_topk against the CPU oracle (bit-exact indices and value bits)."""
import zlib

import numpy as np
import pytest
import torch

import workloads
from _gpu import counters, gpu_topk, parity_topk

pytestmark = pytest.mark.gpu

# 1: register-resident kernel, 2: streamed kernel (bulk copies into a shared-memory ring)
KERNELS = [1, 2]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_attention_indexer_lt_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


@pytest.mark.parametrize("name", ["c1_single_4096", "c2_decode_262144", "c3_ragged_64", "c4_prefill_4096"])
def test_workload_parity_and_fast_path(name):
    S, L, w = workloads.make(name)
    c = counters()
    parity_topk(S.numpy(), None if L is None else L.numpy(), w.k, what=name, counters=c)
    cnt = c.cpu().numpy()
    assert cnt[0] + cnt[1] == w.rows
    # the seeded workloads never need the streaming radix select (beyond a
    # rare guessed threshold from an earlier row that did not fit: counted in [5])
    assert cnt[1] == cnt[5] and cnt[5] <= w.rows // 200, cnt


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("name", ["c1_single_4096", "c2_decode_262144", "c3_ragged_64", "c4_prefill_4096"])
def test_workload_parity_each_kernel(name, kernel):
    S, L, w = workloads.make(name)
    c = counters()
    parity_topk(S.numpy(), None if L is None else L.numpy(), w.k, what=f"{name}/kernel {kernel}",
                counters=c, force_kernel=kernel)
    cnt = c.cpu().numpy()
    assert cnt[0] == w.rows and cnt[1] == 0 and cnt[4] == 0, cnt


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("name", ["c1_single_4096", "c2_decode_262144", "c3_ragged_64"])
def test_workload_parity_exact_path(name, kernel):
    S, L, w = workloads.make(name)
    c = counters()
    parity_topk(S.numpy(), None if L is None else L.numpy(), w.k, what=name + "/exact",
                force_exact=True, counters=c, force_kernel=kernel)
    assert c.cpu().numpy()[1] == w.rows


def test_prefill_rows_exact_path_subset():
    S, L, w = workloads.make("c4_prefill_4096")
    sel = list(range(0, 4096, 97))
    parity_topk(S[sel].numpy(), L[sel].numpy(), w.k, what="c4 subset/exact", force_exact=True)


def stable_seed(*parts) -> int:
    """A seed fixed by the case's parameters (the same in every process, unlike
    Python's randomised string hash)."""
    return zlib.crc32("/".join(map(str, parts)).encode()) % 1000


DISTS = ["normal", "bf16", "coarse", "equal", "asc", "desc", "special", "tail"]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dist", DISTS)
@pytest.mark.parametrize("shape", [(3, 1000), (2, 5000), (2, 40000), (1, 300000)])
def test_small_distributions(dist, shape, kernel):
    rows, stride = shape
    S, L = workloads.random_rows(rows, stride, seed=stable_seed(dist, stride), dist=dist,
                                 lengths="ragged", min_len=0)
    for k in (1, 64, 512):
        parity_topk(S.numpy(), L.numpy(), k, what=f"{dist}{shape} k={k}", force_kernel=kernel)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("k", [1, 512, 2048])
def test_edge_lengths_and_poisoned_padding(k, kernel):
    stride = 20000
    lens = [0, 1, 2, 3, 4, 5, 7, 8, 9, k - 1, k, k + 1, 1023, 1024, 1025, 8191, 8192, 8193,
            16383, 16384, 16385, stride - 1, stride]
    lens = [max(0, min(stride, x)) for x in lens]
    S, _ = workloads.random_rows(len(lens), stride, seed=3, dist="bf16")
    S = S.numpy().copy()
    for r, l in enumerate(lens):
        S[r, l:] = np.inf  # never read: positions >= L must not be selected
    parity_topk(S, np.array(lens, np.int32), k, what=f"edges k={k}", force_kernel=kernel)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("ft", [256, 512])
@pytest.mark.parametrize("fc", [1, 2, 4, 8, 16])
def test_forced_plans_agree(fc, ft, kernel):
    kw = dict(force_cluster=fc, force_threads=ft, force_kernel=kernel)
    S, L = workloads.random_rows(4, 100000, seed=9, dist="bf16", lengths="ragged", min_len=1)
    parity_topk(S.numpy(), L.numpy(), 512, what=f"cluster {fc}x{ft}", **kw)
    # the resident kernel also gets an unaligned stride; the streamed one needs aligned rows
    S2, L2 = workloads.random_rows(3, 70001 if kernel == 1 else 70004, seed=10, dist="special",
                                   lengths="ragged")
    parity_topk(S2.numpy(), L2.numpy(), 300, what=f"cluster {fc}x{ft} special", **kw)
    parity_topk(S2.numpy(), L2.numpy(), 300, what=f"cluster {fc}x{ft} special exact", force_exact=True, **kw)
    S3, L3 = workloads.random_rows(5, 9000, seed=11, dist="coarse", lengths="ragged")
    parity_topk(S3.numpy(), L3.numpy(), 700, what=f"cluster {fc}x{ft} coarse", **kw)


@pytest.mark.parametrize("ft", [256, 512])
@pytest.mark.parametrize("name", ["c1_single_4096", "c2_decode_262144", "c3_ragged_64"])
def test_workloads_both_cta_shapes(name, ft):
    S, L, w = workloads.make(name)
    parity_topk(S.numpy(), None if L is None else L.numpy(), w.k, what=f"{name}/{ft}", force_threads=ft)


def test_unaligned_rows_take_the_scalar_path():
    S, L = workloads.random_rows(5, 30001, seed=4, dist="bf16", lengths="ragged")
    parity_topk(S.numpy(), L.numpy(), 512, what="stride 30001")
    # a row starting 4 bytes past a 16-byte boundary
    big = torch.randn(1, 50001, generator=torch.Generator().manual_seed(5))
    s = big.cuda()[:, 1:]
    import oracle
    import sparse_attention_indexer_lt_gb300 as lt
    idx, val = lt.topk(s, None, 512)
    oi, ov = oracle.topk(big[:, 1:].contiguous().numpy(), None, 512)
    assert np.array_equal(idx.cpu().numpy(), oi)
    assert np.array_equal(val.cpu().numpy().view(np.uint32), ov.view(np.uint32))
    # the streamed kernel needs 16-byte aligned rows and says so
    with pytest.raises(lt.LtError):
        lt.topk(s, None, 512, force_kernel=2)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("k", [1000, 2048])
def test_large_k(k, kernel):
    S, L = workloads.random_rows(3, 262144, seed=12, dist="bf16", lengths="ragged", min_len=1000)
    parity_topk(S.numpy(), L.numpy(), k, what=f"k={k}", force_kernel=kernel)


@pytest.mark.parametrize("kernel", KERNELS)
def test_rows_longer_than_one_register_pass(kernel):
    S, L = workloads.random_rows(2, 1048576, seed=13, dist="normal")
    parity_topk(S.numpy(), None, 512, what="1M positions", force_kernel=kernel)
    S, L = workloads.random_rows(2, 600000, seed=14, dist="tail", lengths="ragged")
    parity_topk(S.numpy(), L.numpy(), 512, what="600K ragged", force_cluster=4, force_kernel=kernel)


@pytest.mark.parametrize("ft", [256, 512])
@pytest.mark.parametrize("dist", ["desc", "coarse", "special", "normal", "equal"])
def test_streaming_filter_thresholds_of_any_sign(dist, ft):
    """Single-CTA rows of many register rounds (the sampled estimate and the
    streaming filter): negative and zero thresholds ("desc"), heavy ties
    ("coarse", "equal": the latter overflows onto the exact path), special
    values, and positive thresholds, which take the sign-bit key shortcut."""
    S, L = workloads.random_rows(6, 45000, seed=21 + len(dist), dist=dist, lengths="ragged",
                                 min_len=20000)
    for k in (64, 512, 2048):
        parity_topk(S.numpy(), L.numpy(), k, what=f"{dist} stream k={k} t={ft}", force_cluster=1,
                    force_threads=ft)


@pytest.mark.parametrize("ft", [256, 512])
def test_streamed_rows_walk_more_rows_than_ctas(ft):
    """Persistent CTAs: many short and empty rows, several rows per CTA, chunks of
    the next row in flight while a row is selected."""
    import sparse_attention_indexer_lt_gb300 as lt
    rows = 1500
    S, L = workloads.random_rows(rows, 6000, seed=16, dist="bf16", lengths="ragged", min_len=0)
    L = L.numpy().copy()
    L[::7] = 0
    c = counters()
    parity_topk(S.numpy(), L, 256, what=f"walk {ft}", force_kernel=2, force_threads=ft, counters=c)
    pl = lt.plan(rows, 6000, 256, force_kernel=2, force_threads=ft)
    assert pl["kernel"] == "stream" and pl["grid"] < rows and pl["stages"] >= 2
    assert c.cpu().numpy()[4] == 0


def test_determinism_repeated_runs():
    S, L, w = workloads.make("c3_ragged_64")
    s, l = S.cuda(), L.cuda()
    import sparse_attention_indexer_lt_gb300 as lt
    i0, v0 = lt.topk(s, l, 512)
    for _ in range(50):
        i1, v1 = lt.topk(s, l, 512)
        assert torch.equal(i0, i1) and torch.equal(v0.view(torch.int32), v1.view(torch.int32))


def test_values_optional_and_side_stream():
    import oracle
    import sparse_attention_indexer_lt_gb300 as lt
    S, _ = workloads.random_rows(8, 9000, seed=15, dist="normal")
    s = S.cuda()
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        idx, val = lt.topk(s, None, 128, with_values=False)
    st.synchronize()
    assert val is None
    oi, _ = oracle.topk(S.numpy(), None, 128)
    assert np.array_equal(idx.cpu().numpy(), oi)


def test_dependent_launch_orders_with_neighbouring_kernels():
    """The kernels start under programmatic dependent launch: a score row written
    by the kernel just before must be read complete, and a kernel just after that
    rewrites the scores must not change the result (no host synchronisation)."""
    import oracle
    import sparse_attention_indexer_lt_gb300 as lt
    S, _ = workloads.random_rows(4, 262144, seed=17, dist="tail")
    base = S.cuda()
    for threads in (0, 256, 512):
        scaled = base * 2.0                      # producer kernel, then top-k at once
        idx, val = lt.topk(scaled, None, 512, force_threads=threads)
        scaled.fill_(float("inf"))               # overwrites the scores right after
        idx2, _ = lt.topk(base * 2.0, None, 512, force_threads=threads)  # back to back
        torch.cuda.synchronize()
        oi, ov = oracle.topk((S * 2.0).numpy(), None, 512)
        assert np.array_equal(idx.cpu().numpy(), oi)
        assert np.array_equal(val.cpu().numpy().view(np.uint32), ov.view(np.uint32))
        assert np.array_equal(idx2.cpu().numpy(), oi)


@pytest.mark.parametrize("bf16", [False, True])
def test_batched_rows_start_from_earlier_rows(bf16):
    """The prefill batch: past the first wave, a row starts from the threshold
    the output of the row one wave earlier implies; the results are the
    oracle's, the guess almost always fits, and forcing the resident kernel
    (every row from its own estimate) gives the same outputs."""
    import sparse_attention_indexer_lt_gb300 as lt
    S, L, w = workloads.make("c4_prefill_4096")
    c = counters()
    if bf16:
        from _gpu import parity_bf16
        parity_bf16(workloads.to_bf16(S), L.numpy(), w.k, what="c4 bf16 hinted", counters=c)
    else:
        parity_topk(S.numpy(), L.numpy(), w.k, what="c4 hinted", counters=c)
    cnt = c.cpu().numpy()
    assert cnt[0] + cnt[1] == w.rows and cnt[1] == cnt[5], cnt  # only a missed guess takes the exact path
    assert cnt[6] > w.rows // 2, cnt  # most rows past the first two waves used a hint
    assert cnt[5] < w.rows // 100, cnt
    c.zero_()
    parity_topk(S.numpy(), L.numpy(), w.k, what="c4 own estimates", counters=c, force_kernel=lt.KERNEL_RESIDENT)
    assert c.cpu().numpy()[6] == 0 and c.cpu().numpy()[5] == 0


@pytest.mark.parametrize("dist", ["normal", "coarse", "special", "desc"])
def test_hinted_rows_redo_when_the_guess_misses(dist):
    """Rows whose scales alternate by a factor of 64 (the earlier row's values
    make the next row keep too few or too many), ragged and empty rows, ties
    and special values: a guess that misses takes the exact path; same
    results. Without values requested no hint is taken."""
    import sparse_attention_indexer_lt_gb300 as lt
    rows, stride = 1200, 9000
    S, L = workloads.random_rows(rows, stride, seed=stable_seed("hint", dist), dist=dist, lengths="ragged",
                                 min_len=0)
    S = S.numpy().copy()
    with np.errstate(over="ignore"):
        S[1::2] *= 64.0
    S[2::3] -= 5.0
    L = L.numpy().copy()
    L[::11] = 0
    L[1::13] = 300  # shorter than k: no estimate, no hint
    c = counters()
    for k in (64, 512):
        c.zero_()
        parity_topk(S, L, k, what=f"redo {dist} k={k}", counters=c)
        cnt = c.cpu().numpy()
        assert cnt[0] + cnt[1] == int((L > 0).sum()), cnt  # rows with K = 0 count nothing
        if dist == "normal":
            assert cnt[5] > 0 and cnt[6] > 0, cnt
    c.zero_()
    idx, val = gpu_topk(S, L, 512, with_values=False, counters=c)
    assert val is None and c.cpu().numpy()[6] == 0
    assert np.array_equal(idx, __import__("oracle").topk(S, L, 512)[0])


def test_hints_read_while_another_stream_rewrites_them():
    """Later rows of a batch take their threshold from an earlier row's output
    values. Here another stream keeps overwriting the values of the first rows
    while the launch runs, so the readings change under the rows that take
    them (and may differ between a CTA's warps): every index still matches the
    oracle, and so does every value the other stream does not touch."""
    import oracle
    import sparse_attention_indexer_lt_gb300 as lt
    rows, stride, k = 2400, 9000, 512
    S, L = workloads.random_rows(rows, stride, seed=stable_seed("rewrite"), dist="normal", lengths="ragged")
    S, L = S.numpy(), L.numpy()
    oi, ov = oracle.topk(S, L, k)
    dev = torch.device("cuda")
    s = torch.from_numpy(S).to(dev)
    l = torch.from_numpy(L).to(torch.int32).to(dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    n_rw = rows - 2 * sms * 3  # rows whose values later rows read
    assert n_rw > 0
    side = torch.cuda.Stream()
    for _ in range(3):
        out_idx = torch.empty(rows, k, dtype=torch.int32, device=dev)
        out_val = torch.empty(rows, k, dtype=torch.float32, device=dev)
        torch.cuda.synchronize()
        with torch.cuda.stream(side):
            for i in range(200):
                out_val[:n_rw].normal_()
        lt.topk(s, l, k, out_idx=out_idx, out_val=out_val)
        torch.cuda.synchronize()
        gi, gv = out_idx.cpu().numpy(), out_val.cpu().numpy()
        assert np.array_equal(gi, oi), np.nonzero((gi != oi).any(axis=1))[0][:8]
        assert np.array_equal(gv[n_rw:].view(np.uint32), ov[n_rw:].view(np.uint32))


@pytest.mark.parametrize("stride", [1, 2, 3, 5])
def test_tiny_rows(stride):
    """Rows of a handful of positions (unaligned, scalar loads), k above and
    below the row length, every plan the automatic planner picks for them."""
    for rows in (1, 7, 300):
        S, L = workloads.random_rows(rows, stride, seed=stable_seed("tiny", stride, rows), dist="coarse",
                                     lengths="ragged", min_len=0)
        for k in (1, 2, 4, 9):
            parity_topk(S.numpy(), L.numpy(), k, what=f"stride {stride} rows {rows} k {k}")
            parity_topk(S.numpy(), None, k, what=f"stride {stride} rows {rows} k {k} full")


def test_many_short_rows():
    """100,000 rows of 96 positions (one single-round CTA each, many waves),
    ragged, ties and special values mixed in."""
    rows, stride, k = 100000, 96, 16
    S, L = workloads.random_rows(rows, stride, seed=61, dist="special", lengths="ragged", min_len=0)
    c = counters()
    parity_topk(S.numpy(), L.numpy(), k, what="100K rows", counters=c)
    cnt = c.cpu().numpy()
    assert cnt[0] + cnt[1] == int((L.numpy() > 0).sum()), cnt
