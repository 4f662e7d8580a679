"""GPU parity of the bf16-score entry points against the oracle on the same bit
patterns (bit-exact indices, value bits and kept blocks)."""
import numpy as np
import pytest
import torch

import workloads
from _gpu import counters, parity_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_attention_indexer_lt_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


@pytest.mark.parametrize("name", ["c1_single_4096", "c2_decode_262144", "c3_ragged_64", "c4_prefill_4096"])
def test_workloads_in_bf16(name):
    S, L, w = workloads.make(name)
    c = counters()
    parity_bf16(workloads.to_bf16(S), None if L is None else L.numpy(), w.k, what=f"{name}/bf16", counters=c)
    cnt = c.cpu().numpy()
    assert cnt[0] + cnt[1] == w.rows


def test_blocked_workload_in_bf16():
    S, L, w = workloads.make("c5_blocked_16")
    parity_bf16(workloads.to_bf16(S), None, w.k, what="c5/bf16", kind="blocked", block=w.block,
                k_blocks=w.k_blocks)


def test_listed_workload_in_bf16():
    S, L, w = workloads.make("c6_listed_16")
    parity_bf16(workloads.to_bf16(S), None, w.k, what="c6/bf16", kind="listed", block=w.block,
                cand=workloads.listed_blocks("c6_listed_16").numpy())


@pytest.mark.parametrize("name", ["c1_single_4096", "c2_decode_262144", "c3_ragged_64"])
def test_exact_path_in_bf16(name):
    S, L, w = workloads.make(name)
    c = counters()
    parity_bf16(workloads.to_bf16(S), None if L is None else L.numpy(), w.k, what=f"{name}/bf16 exact",
                force_exact=True, counters=c)
    assert c.cpu().numpy()[1] == w.rows


@pytest.mark.parametrize("shape", [(3, 1000), (2, 40000), (1, 300000)])
@pytest.mark.parametrize("k", [1, 64, 512])
def test_special_patterns(shape, k):
    """Signed zeros, infinities, subnormals and NaNs with payloads, in ragged rows."""
    rows, stride = shape
    T = workloads.random_bf16_special(rows, stride, seed=stride + k)
    g = torch.Generator().manual_seed(stride)
    L = torch.randint(0, stride + 1, (rows,), generator=g, dtype=torch.int32).numpy()
    parity_bf16(T, L, k, what=f"special {shape} k={k}")
    parity_bf16(T, L, k, what=f"special {shape} k={k} blocked", kind="blocked", block=8, k_blocks=max(1, k // 2))


@pytest.mark.parametrize("k", [1, 512, 2048])
def test_edge_lengths_and_poisoned_padding(k):
    stride = 20000
    lens = [0, 1, 2, 3, 4, 5, 7, 8, 9, k - 1, k, k + 1, 1023, 1024, 1025, 8191, 8192, 8193,
            16383, 16384, 16385, stride - 1, stride]
    lens = [max(0, min(stride, x)) for x in lens]
    S, _ = workloads.random_rows(len(lens), stride, seed=31, dist="bf16")
    T = workloads.to_bf16(S)
    for r, l in enumerate(lens):
        T[r, l:] = float("inf")  # never read
    parity_bf16(T, np.array(lens, np.int32), k, what=f"bf16 edges k={k}")


@pytest.mark.parametrize("ft", [256, 512])
@pytest.mark.parametrize("fc", [1, 2, 4, 8, 16])
def test_forced_plans(fc, ft):
    S, L = workloads.random_rows(4, 100000, seed=33, dist="tail", lengths="ragged", min_len=1)
    parity_bf16(workloads.to_bf16(S), L.numpy(), 512, what=f"bf16 {fc}x{ft}", force_cluster=fc, force_threads=ft)
    S2, L2 = workloads.random_rows(3, 9000, seed=34, dist="coarse", lengths="ragged")
    parity_bf16(workloads.to_bf16(S2), L2.numpy(), 700, what=f"bf16 {fc}x{ft} coarse", force_cluster=fc,
                force_threads=ft)
    parity_bf16(workloads.to_bf16(S), L.numpy(), 256, what=f"bf16 {fc}x{ft} blocked", kind="blocked", block=8,
                k_blocks=128, force_cluster=fc, force_threads=ft)


def test_unaligned_rows_take_scalar_loads():
    """An odd row stride (rows not 8-byte aligned) and a row starting 2 bytes
    past an aligned address."""
    S, L = workloads.random_rows(5, 30001, seed=35, dist="bf16", lengths="ragged")
    parity_bf16(workloads.to_bf16(S), L.numpy(), 512, what="bf16 stride 30001")
    import oracle
    import sparse_attention_indexer_lt_gb300 as lt
    big = workloads.to_bf16(torch.randn(1, 50001, generator=torch.Generator().manual_seed(36)))
    s = big.cuda()[:, 1:]
    idx, val = lt.topk(s, None, 512)
    oi, ov = oracle.topk_bf16(workloads.bf16_bits(big[:, 1:]), None, 512)
    assert np.array_equal(idx.cpu().numpy(), oi)
    assert np.array_equal(val.cpu().numpy().view(np.uint32), ov.view(np.uint32))
    with pytest.raises(lt.LtError):
        lt.topk(big.cuda(), None, 512, force_kernel=2)  # the streamed kernel reads fp32 only


def test_long_rows():
    S, _ = workloads.random_rows(2, 1048576, seed=37, dist="normal")
    parity_bf16(workloads.to_bf16(S), None, 512, what="bf16 1M positions")


def test_plain_bf16_entry_points_through_the_c_abi():
    """lt_topk_bf16 / lt_topk_blocked_bf16 / lt_topk_candidates_bf16 called with
    device pointers and a stream through ctypes."""
    import ctypes
    import oracle
    import sparse_attention_indexer_lt_gb300 as lt
    lib = lt.load()
    S, L = workloads.random_rows(3, 70000, seed=38, dist="tail", lengths="ragged", min_len=1)
    T = workloads.to_bf16(S)
    bits = workloads.bf16_bits(T)
    Ln = L.numpy()
    s, l = T.cuda(), L.cuda()
    k, kb = 256, 512
    oi = torch.empty(3, k, dtype=torch.int32, device="cuda")
    ov = torch.empty(3, k, dtype=torch.float32, device="cuda")
    ob = torch.empty(3, kb, dtype=torch.int32, device="cuda")
    st = torch.cuda.Stream()
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    sp = ctypes.c_void_p(st.cuda_stream)
    assert lib.lt_topk_bf16(P(s), P(l), 3, 70000, k, P(oi), P(ov), sp) == 0
    st.synchronize()
    ei, ev = oracle.topk_bf16(bits, Ln, k)
    assert np.array_equal(oi.cpu().numpy(), ei) and np.array_equal(ov.cpu().numpy().view(np.uint32), ev.view(np.uint32))
    assert lib.lt_topk_blocked_bf16(P(s), P(l), 3, 70000, 8, kb, k, P(oi), P(ov), P(ob), sp) == 0
    st.synchronize()
    ei, ev, eb = oracle.topk_blocked_bf16(bits, Ln, 8, kb, k)
    assert np.array_equal(oi.cpu().numpy(), ei) and np.array_equal(ob.cpu().numpy(), eb)
    assert lib.lt_topk_candidates_bf16(P(s), P(l), 3, 70000, 8, P(ob), kb, k, P(oi), P(ov), sp) == 0
    st.synchronize()
    ei, ev = oracle.topk_candidates_bf16(bits, Ln, eb, 8, k)
    assert np.array_equal(oi.cpu().numpy(), ei) and np.array_equal(ov.cpu().numpy().view(np.uint32), ev.view(np.uint32))
