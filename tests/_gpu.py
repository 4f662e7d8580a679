"""Helpers for the GPU parity tests: run the CUDA path through the C ABI on
seeded inputs and compare with the oracle bit for bit."""
import numpy as np
import torch

import oracle
import sparse_attention_indexer_lt_gb300 as lt
from _checks import check_invariants


def to_dev(S, L):
    s = torch.as_tensor(S).cuda()
    l = None if L is None else torch.as_tensor(L).to(torch.int32).cuda()
    return s, l


def gpu_topk(S, L, k, **kw):
    s, l = to_dev(S, L)
    idx, val = lt.topk(s, l, k, **kw)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), (val.cpu().numpy() if val is not None else None)


def gpu_blocked(S, L, block, k_blocks, k, **kw):
    s, l = to_dev(S, L)
    idx, val, blk = lt.topk_blocked(s, l, block, k_blocks, k, **kw)
    torch.cuda.synchronize()
    return (idx.cpu().numpy(), None if val is None else val.cpu().numpy(),
            None if blk is None else blk.cpu().numpy())


def assert_same(gi, gv, oi, ov, what=""):
    if not np.array_equal(gi, oi):
        bad = np.nonzero((gi != oi).any(axis=1))[0]
        r = int(bad[0])
        j = np.nonzero(gi[r] != oi[r])[0][:8]
        raise AssertionError(f"{what}: index mismatch in {bad.size} rows; row {r} slots {j.tolist()}: "
                             f"gpu {gi[r, j].tolist()} oracle {oi[r, j].tolist()}")
    if gv is not None:
        if not np.array_equal(gv.view(np.uint32), ov.view(np.uint32)):
            bad = np.nonzero((gv.view(np.uint32) != ov.view(np.uint32)).any(axis=1))[0]
            raise AssertionError(f"{what}: value bits differ in rows {bad[:8].tolist()}")


def parity_topk(S, L, k, what="", **kw):
    S = np.ascontiguousarray(np.asarray(S, dtype=np.float32))
    Ln = None if L is None else np.asarray(L, dtype=np.int32)
    gi, gv = gpu_topk(S, Ln, k, **kw)
    oi, ov = oracle.topk(S, Ln, k)
    assert_same(gi, gv, oi, ov, what)
    return gi, gv


def parity_blocked(S, L, block, k_blocks, k, what="", **kw):
    S = np.ascontiguousarray(np.asarray(S, dtype=np.float32))
    Ln = None if L is None else np.asarray(L, dtype=np.int32)
    gi, gv, gb = gpu_blocked(S, Ln, block, k_blocks, k, **kw)
    oi, ov, ob = oracle.topk_blocked(S, Ln, block, k_blocks, k)
    assert_same(gi, gv, oi, ov, what)
    if gb is not None and not np.array_equal(gb, ob):
        bad = np.nonzero((gb != ob).any(axis=1))[0]
        raise AssertionError(f"{what}: out_blocks differ in rows {bad[:8].tolist()}")
    return gi, gv, gb


def parity_candidates(S, L, cand, block, k, what="", **kw):
    S = np.ascontiguousarray(np.asarray(S, dtype=np.float32))
    Ln = None if L is None else np.asarray(L, dtype=np.int32)
    C = np.ascontiguousarray(np.asarray(cand, dtype=np.int32))
    s, l = to_dev(S, Ln)
    gi, gv = lt.topk_candidates(s, torch.as_tensor(C).cuda(), l, block, k, **kw)
    torch.cuda.synchronize()
    gi = gi.cpu().numpy()
    gv = None if gv is None else gv.cpu().numpy()
    oi, ov = oracle.topk_candidates(S, Ln, C, block, k)
    assert_same(gi, gv, oi, ov, what)
    return gi, gv


def parity_bf16(T, L, k, what="", kind="topk", block=8, k_blocks=2048, cand=None, **kw):
    """bf16 scores (a CPU torch.bfloat16 tensor) through the bf16 path and the
    oracle on the same bit patterns: indices, value bits and kept blocks agree."""
    import workloads
    bits = workloads.bf16_bits(T)
    Ln = None if L is None else np.asarray(L, dtype=np.int32)
    s = T.cuda()
    l = None if Ln is None else torch.as_tensor(Ln).cuda()
    if kind == "topk":
        gi, gv = lt.topk(s, l, k, **kw)
        oi, ov = oracle.topk_bf16(bits, Ln, k)
    elif kind == "blocked":
        gi, gv, gb = lt.topk_blocked(s, l, block, k_blocks, k, **kw)
        oi, ov, ob = oracle.topk_blocked_bf16(bits, Ln, block, k_blocks, k)
    else:
        C = np.ascontiguousarray(np.asarray(cand, dtype=np.int32))
        gi, gv = lt.topk_candidates(s, torch.as_tensor(C).cuda(), l, block, k, **kw)
        oi, ov = oracle.topk_candidates_bf16(bits, Ln, C, block, k)
    torch.cuda.synchronize()
    assert_same(gi.cpu().numpy(), None if gv is None else gv.cpu().numpy(), oi, ov, what)
    if kind == "blocked" and gb is not None:
        assert np.array_equal(gb.cpu().numpy(), ob), f"{what}: out_blocks differ"


def counters():
    return torch.zeros(lt.NUM_COUNTERS, dtype=torch.int32, device="cuda")
