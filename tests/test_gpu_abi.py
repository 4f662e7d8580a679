"""The contract's own entry points on the GPU, called through ctypes with device
pointers and a stream, and the failure paths reachable without faulting a GPU."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

LT_TEST_FAIL_LAUNCHES, LT_TEST_STALL_STREAMED = 1, 2


@pytest.fixture(scope="module")
def lib():
    from sparse_attention_indexer_lt_gb300 import build, load
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return load()


def P(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def test_plain_entry_points_match_the_oracle(lib):
    """lt_topk, lt_topk_blocked and lt_topk_candidates (fp32) on a side stream."""
    rows, stride, k, kb = 3, 70000, 256, 512
    S, L = workloads.random_rows(rows, stride, seed=41, dist="tail", lengths="ragged", min_len=1)
    Sn, Ln = S.numpy(), L.numpy()
    s, l = S.cuda(), L.cuda()
    oi = torch.empty(rows, k, dtype=torch.int32, device="cuda")
    ov = torch.empty(rows, k, dtype=torch.float32, device="cuda")
    ob = torch.empty(rows, kb, dtype=torch.int32, device="cuda")
    st = torch.cuda.Stream()
    sp = ctypes.c_void_p(st.cuda_stream)

    def same(ei, ev):
        assert np.array_equal(oi.cpu().numpy(), ei)
        assert np.array_equal(ov.cpu().numpy().view(np.uint32), ev.view(np.uint32))

    assert lib.lt_topk(P(s), P(l), rows, stride, k, P(oi), P(ov), sp) == 0
    st.synchronize()
    same(*oracle.topk(Sn, Ln, k))
    assert lib.lt_topk_blocked(P(s), P(l), rows, stride, 8, kb, k, P(oi), P(ov), P(ob), sp) == 0
    st.synchronize()
    ei, ev, eb = oracle.topk_blocked(Sn, Ln, 8, kb, k)
    same(ei, ev)
    assert np.array_equal(ob.cpu().numpy(), eb)
    # the kept blocks as the published list of a later layer's call
    assert lib.lt_topk_candidates(P(s), P(l), rows, stride, 8, P(ob), kb, k, P(oi), P(ov), sp) == 0
    st.synchronize()
    same(*oracle.topk_candidates(Sn, Ln, eb, 8, k))
    # k_blocks < k: the stages run one after the other
    assert lib.lt_topk_blocked(P(s), P(l), rows, stride, 8, 16, k, P(oi), P(ov), None, sp) == 0
    st.synchronize()
    ei, ev, _ = oracle.topk_blocked(Sn, Ln, 8, 16, k)
    same(ei, ev)


def test_injected_launch_failure_returns_cuda_error_and_launches_nothing(lib):
    import sparse_attention_indexer_lt_gb300 as lt
    S, _ = workloads.random_rows(2, 5000, seed=42, dist="normal")
    s = S.cuda()
    oi = torch.full((2, 64), 7, dtype=torch.int32, device="cuda")
    assert lib.lt_test_inject(LT_TEST_FAIL_LAUNCHES, 3) == 0
    for call in (lambda: lib.lt_topk(P(s), None, 2, 5000, 64, P(oi), None, None),
                 lambda: lib.lt_topk_blocked(P(s), None, 2, 5000, 8, 128, 64, P(oi), None, None, None),
                 lambda: lib.lt_topk_candidates(P(s), None, 2, 5000, 8, None, 0, 64, P(oi), None, None)):
        assert call() == 3  # LT_ERR_CUDA
    torch.cuda.synchronize()
    assert bool((oi == 7).all()), "a failed launch wrote outputs"
    assert lib.lt_test_inject(99, 1) == 1 and lib.lt_test_inject(LT_TEST_FAIL_LAUNCHES, -1) == 1
    # the hook is spent: the next call works and the context is healthy
    idx, _ = lt.topk(s, None, 64)
    assert np.array_equal(idx.cpu().numpy(), oracle.topk(S.numpy(), None, 64)[0])


def test_streamed_kernel_wait_gives_up_and_returns(lib):
    """The streamed kernel's mbarrier waits are bounded: with the final copy of
    each CTA never issued, the wait for it gives up after a few polls, the row
    is counted in counters[4], and the kernel finishes; the next launch is
    correct again."""
    import sparse_attention_indexer_lt_gb300 as lt
    rows, stride = 40, 12000
    S, _ = workloads.random_rows(rows, stride, seed=43, dist="bf16")
    s = S.cuda()
    c = torch.zeros(lt.NUM_COUNTERS, dtype=torch.int32, device="cuda")
    assert lib.lt_test_inject(LT_TEST_STALL_STREAMED, 4) == 0
    lt.topk(s, None, 128, force_kernel=lt.KERNEL_STREAM, counters=c)
    torch.cuda.synchronize()
    pl = lt.plan(rows, stride, 128, force_kernel=lt.KERNEL_STREAM)
    assert c.cpu().numpy()[4] >= 1
    assert c.cpu().numpy()[4] <= pl["grid"] // pl["cluster"]
    # the hook applied to that launch only
    c.zero_()
    idx, val = lt.topk(s, None, 128, force_kernel=lt.KERNEL_STREAM, counters=c)
    torch.cuda.synchronize()
    oi, ov = oracle.topk(S.numpy(), None, 128)
    assert np.array_equal(idx.cpu().numpy(), oi)
    assert c.cpu().numpy()[4] == 0


def test_pinned_host_scores_read_in_place(lib):
    """Scores in page-locked host memory are read by the kernels in place (over
    the host link): every entry point and both score types give the oracle's
    answer; unregistered host memory is refused; the streamed kernel refuses
    host scores."""
    import sparse_attention_indexer_lt_gb300 as lt
    from _gpu import assert_same
    rows, stride, k = 5, 70000, 300
    S, L = workloads.random_rows(rows, stride, seed=47, dist="tail", lengths="ragged", min_len=1)
    Sn, Ln = S.numpy(), L.numpy()
    host = S.pin_memory()
    l = L.cuda()
    gi, gv = lt.topk(host, l, k)
    oi, ov = oracle.topk(Sn, Ln, k)
    assert_same(gi.cpu().numpy(), gv.cpu().numpy(), oi, ov, "pinned host, top-k")
    gi, gv = lt.topk(host, l, k, force_exact=True)
    assert_same(gi.cpu().numpy(), gv.cpu().numpy(), oi, ov, "pinned host, top-k exact")
    # many rows of several rounds (the batched 256-thread path, whose L2 prefetch host rows skip)
    S4, L4 = workloads.random_rows(400, 20000, seed=48, dist="normal", lengths="ragged", min_len=1)
    gi, gv = lt.topk(S4.pin_memory(), L4.cuda(), 512)
    oi4, ov4 = oracle.topk(S4.numpy(), L4.numpy(), 512)
    assert_same(gi.cpu().numpy(), gv.cpu().numpy(), oi4, ov4, "pinned host, batched rows")
    gi, gv, gb = lt.topk_blocked(host, l, 8, 512, k)
    oi, ov, ob = oracle.topk_blocked(Sn, Ln, 8, 512, k)
    assert_same(gi.cpu().numpy(), gv.cpu().numpy(), oi, ov, "pinned host, two-level")
    assert np.array_equal(gb.cpu().numpy(), ob)
    cand = np.sort(np.random.default_rng(49).choice(stride // 8, (rows, 900), replace=True), axis=1).astype(np.int32)
    gi, gv = lt.topk_candidates(host, torch.as_tensor(cand).cuda(), l, 8, k)
    oi, ov = oracle.topk_candidates(Sn, Ln, cand, 8, k)
    assert_same(gi.cpu().numpy(), gv.cpu().numpy(), oi, ov, "pinned host, listed candidates")
    # lengths and outputs in pinned host memory too (written in place by the kernel)
    hi = torch.empty(rows, k, dtype=torch.int32).pin_memory()
    hv = torch.empty(rows, k, dtype=torch.float32).pin_memory()
    hb = torch.empty(rows, 512, dtype=torch.int32).pin_memory()
    lt.topk(host, L.pin_memory(), k, out_idx=hi, out_val=hv)
    torch.cuda.synchronize()
    oi, ov = oracle.topk(Sn, Ln, k)
    assert_same(hi.numpy(), hv.numpy(), oi, ov, "pinned host scores, lengths and outputs")
    hv2 = torch.empty(rows, k, dtype=torch.float32).pin_memory()
    lt.topk_blocked(host, L.pin_memory(), 8, 512, k, out_idx=hi, out_val=hv2, out_blocks=hb)
    torch.cuda.synchronize()
    oi, ov, ob = oracle.topk_blocked(Sn, Ln, 8, 512, k)
    assert_same(hi.numpy(), hv2.numpy(), oi, ov, "pinned host, two-level outputs")
    assert np.array_equal(hb.numpy(), ob)
    lt.topk_candidates(host, torch.as_tensor(cand).pin_memory(), L.pin_memory(), 8, k, out_idx=hi, out_val=hv)
    torch.cuda.synchronize()
    oi, ov = oracle.topk_candidates(Sn, Ln, cand, 8, k)
    assert_same(hi.numpy(), hv.numpy(), oi, ov, "pinned host list and outputs")
    T = workloads.to_bf16(S)
    gi, gv = lt.topk(T.pin_memory(), l, k)
    oi, ov = oracle.topk_bf16(workloads.bf16_bits(T), Ln, k)
    assert_same(gi.cpu().numpy(), gv.cpu().numpy(), oi, ov, "pinned host, bf16")
    # unregistered host memory (a numpy buffer) and the streamed kernel
    out = torch.empty(rows, k, dtype=torch.int32, device="cuda")
    arr = np.ascontiguousarray(Sn)
    st = lib.lt_topk_ex(ctypes.c_void_p(arr.ctypes.data), 0, P(l), rows, stride, k, P(out), None, 0, 0, 0, 0,
                        None, None, None)
    assert st == 1
    st = lib.lt_topk_ex(P(host), 0, P(l), rows, stride, k, P(out), None, 0, 0, 0, 2, None, None, None)
    assert st == 2
    torch.cuda.synchronize()
    with pytest.raises(TypeError):
        lt.topk(S, l, k)  # a pageable CPU tensor
