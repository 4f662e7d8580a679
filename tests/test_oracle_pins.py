"""Pins for the CPU oracle: brute force, hand-worked cases, library routines,
invariants, special cases and the two-level identity. CPU only.

The oracle is the reference every GPU parity test compares against, so each of
its functions is checked here against something other than itself.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads
from _checks import (brute_blocked_row, brute_candidates_row, brute_topk_row, check_invariants, equal_outputs,
                     lexsort_topk_row)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f(v):
    return float(v)  # accepts "inf", "-inf", "nan", "-0.0" as strings


def _arr(vals):
    return np.array([_f(v) for v in vals], dtype=np.float32)


# ---------------------------------------------------------------- hand-worked cases

def _load(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return [json.loads(line) for line in fh if line.strip()]


@pytest.mark.parametrize("case", _load("topk_hand_cases.jsonl"), ids=lambda c: c["name"])
def test_hand_cases_topk(case):
    s = _arr(case["scores"])
    idx, val = oracle.topk(s[None, :], np.array([case["L"]], np.int32), case["k"], nthreads=1)
    assert idx[0].tolist() == case["idx"]
    want = _arr(case["val"])
    # bit-exact, including the sign of zero
    assert np.array_equal(np.where(np.isnan(val[0]), 0, val[0].view(np.uint32)),
                          np.where(np.isnan(want), 0, want.view(np.uint32)))
    assert np.array_equal(np.isnan(val[0]), np.isnan(want))


@pytest.mark.parametrize("case", _load("blocked_hand_cases.jsonl"), ids=lambda c: c["name"])
def test_hand_cases_blocked(case):
    s = _arr(case["scores"])
    idx, val, blk = oracle.topk_blocked(s[None, :], np.array([case["L"]], np.int32), case["block"],
                                        case["k_blocks"], case["k"], nthreads=1)
    assert idx[0].tolist() == case["idx"]
    assert blk[0].tolist() == case["blocks"]
    want = _arr(case["val"])
    assert np.array_equal(val[0], want)


# ---------------------------------------------------------------- brute force

ALPHABET = [0.0, 1.0, 2.0]


def test_exhaustive_small_alphabet():
    """Every row over {0,1,2} with n <= 7, every k in 1..n+1, against Python sorted."""
    rows = []
    for n in range(0, 8):
        for combo in itertools.product(ALPHABET, repeat=n):
            rows.append(list(combo) + [9.0] * (7 - n))  # 9.0 sits beyond L (poison)
    lens = []
    for n in range(0, 8):
        lens += [n] * (len(ALPHABET) ** n)
    S = np.array(rows, dtype=np.float32)
    Lv = np.array(lens, dtype=np.int32)
    for k in range(1, 9):
        idx, _ = oracle.topk(S, Lv, k)
        for r in range(S.shape[0]):
            assert idx[r].tolist() == brute_topk_row(S[r], int(Lv[r]), k), (r, k)


SPECIALS = [float("inf"), float("-inf"), 0.0, -0.0, float("nan"), 1.0, -1.0, 1e-45]


def test_random_specials_against_two_brute_forces():
    rng = np.random.default_rng(1)
    for trial in range(400):
        n = int(rng.integers(0, 13))
        s = np.array(rng.choice(SPECIALS, size=12), dtype=np.float32)
        k = int(rng.integers(1, 15))
        idx, val = oracle.topk(s[None, :], np.array([n], np.int32), k, nthreads=1)
        assert idx[0].tolist() == brute_topk_row(s, n, k), (s, n, k)
        assert idx[0].tolist() == lexsort_topk_row(s, n, k), (s, n, k)


def test_lexsort_on_seeded_tie_heavy_rows():
    S, _ = workloads.random_rows(6, 3000, seed=5, dist="coarse")
    S = S.numpy()
    idx, _ = oracle.topk(S, None, 700)
    for r in range(S.shape[0]):
        assert idx[r].tolist() == lexsort_topk_row(S[r], S.shape[1], 700)


# ---------------------------------------------------------------- library cross-checks

def test_values_match_library_sorts():
    """The multiset of top-k values does not depend on the tie rule."""
    S, _ = workloads.random_rows(8, 5000, seed=7, dist="bf16")
    S = S.numpy()
    k = 512
    _, val = oracle.topk(S, None, k)
    tv = torch.topk(torch.from_numpy(S), k, dim=1, sorted=True).values.numpy()
    ns = -np.sort(-S, axis=1)[:, :k]
    assert np.array_equal(val, tv)
    assert np.array_equal(val, ns)


def test_k1_is_first_argmax():
    S, _ = workloads.random_rows(16, 777, seed=11, dist="coarse")
    S = S.numpy()
    idx, _ = oracle.topk(S, None, 1)
    assert np.array_equal(idx[:, 0], np.argmax(S, axis=1))


def test_k_ge_L_is_stable_argsort():
    S, _ = workloads.random_rows(4, 300, seed=12, dist="coarse")
    S = S.numpy()
    idx, _ = oracle.topk(S, None, 300)
    assert np.array_equal(idx, np.argsort(-S, axis=1, kind="stable"))


def test_all_equal_and_monotone_rows():
    S, _ = workloads.random_rows(2, 1000, seed=0, dist="equal")
    idx, _ = oracle.topk(S.numpy(), None, 64)
    assert np.array_equal(idx, np.tile(np.arange(64), (2, 1)))
    S, _ = workloads.random_rows(2, 1000, seed=0, dist="asc")
    idx, _ = oracle.topk(S.numpy(), None, 64)
    assert np.array_equal(idx, np.tile(np.arange(999, 999 - 64, -1), (2, 1)))
    S, _ = workloads.random_rows(2, 1000, seed=0, dist="desc")
    idx, _ = oracle.topk(S.numpy(), None, 64)
    assert np.array_equal(idx, np.tile(np.arange(64), (2, 1)))


# ---------------------------------------------------------------- invariants on the workloads

@pytest.mark.parametrize("name", ["c1_single_4096", "c2_decode_262144", "c3_ragged_64"])
def test_invariants_on_workloads(name):
    S, L, w = workloads.make(name)
    S = S.numpy()
    Ln = None if L is None else L.numpy()
    idx, val = oracle.topk(S, Ln, w.k)
    assert check_invariants(S, Ln, w.k, idx, val) == []


def test_invariants_on_prefill_rows_subset():
    S, L, w = workloads.make("c4_prefill_4096")
    sel = [0, 1, 2047, 4095]
    Ssub = S[sel].numpy()
    Lsub = L[sel].numpy()
    idx, val = oracle.topk(Ssub, Lsub, w.k)
    assert check_invariants(Ssub, Lsub, w.k, idx, val) == []


def test_seed0_config1_threshold_has_ties():
    """Config 1 really exercises the tie fill: 509 above the threshold, 5 equal."""
    S, _, w = workloads.make("c1_single_4096")
    S = S.numpy()[0]
    idx, val = oracle.topk(S[None], None, 512)
    t = val[0, -1]
    assert (S > t).sum() == 509 and (S == t).sum() == 5
    ties = np.nonzero(S == t)[0]
    assert idx[0, 509:].tolist() == ties[:3].tolist()


# ---------------------------------------------------------------- two-level

def test_blocked_against_brute_force_small():
    rng = np.random.default_rng(3)
    for trial in range(300):
        B = int(rng.choice([1, 2, 3, 4, 8]))
        n = int(rng.integers(0, 40))
        s = np.array(rng.choice([0.0, 1.0, 2.0, -1.0, float("nan"), -0.0], size=40), dtype=np.float32)
        kb = int(rng.integers(1, 8))
        k = int(rng.integers(1, 20))
        idx, val, blk = oracle.topk_blocked(s[None], np.array([n], np.int32), B, kb, k, nthreads=1)
        bi, bb = brute_blocked_row(s, n, B, kb, k)
        assert idx[0].tolist() == bi, (s, n, B, kb, k)
        assert blk[0].tolist() == bb, (s, n, B, kb, k)


@pytest.mark.parametrize("dist", ["normal", "coarse", "bf16", "special"])
def test_blocked_equals_plain_when_kblocks_ge_k(dist):
    """With k_blocks >= k every block holding a plain top-k position is kept (the
    blocks ranked above it each hold a distinct, higher-ranked position), so the
    two-level result equals the plain top-k, ties included."""
    S, L = workloads.random_rows(8, 4096, seed=21, dist=dist, lengths="ragged")
    S = S.numpy()
    L = L.numpy()
    for kb, k in [(64, 64), (128, 64), (512, 100)]:
        i1, v1, _ = oracle.topk_blocked(S, L, 8, kb, k)
        i2, v2 = oracle.topk(S, L, k)
        assert equal_outputs(i1, v1, i2, v2)


def test_blocked_workload_rows_invariants():
    S, L, w = workloads.make("c5_blocked_16")
    S = S[:2].numpy()
    idx, val, blk = oracle.topk_blocked(S, None, w.block, w.k_blocks, w.k)
    assert check_invariants(S, None, w.k, idx, val) == []
    for r in range(2):
        b = blk[r]
        assert np.all(np.diff(b) > 0) and b.size == w.k_blocks
        # every output position lies in a kept block
        assert np.isin(idx[r] // w.block, b).all()


def test_candidates_against_brute_force_small():
    rng = np.random.default_rng(5)
    for trial in range(300):
        B = int(rng.choice([1, 2, 3, 4, 8]))
        n = int(rng.integers(0, 40))
        s = np.array(rng.choice([0.0, 1.0, 2.0, -1.0, float("nan"), -0.0], size=40), dtype=np.float32)
        nc = int(rng.integers(0, 12))
        listed = rng.integers(-2, 14, size=nc).astype(np.int32)  # pads, repeats, ids past the row
        k = int(rng.integers(1, 20))
        idx, val = oracle.topk_candidates(s[None], np.array([n], np.int32), listed[None], B, k, nthreads=1)
        assert idx[0].tolist() == brute_candidates_row(s, n, B, listed, k), (s, n, B, listed, k)
        assert check_invariants_subset(s, idx[0], val[0])


def check_invariants_subset(s, idx, val):
    """Picks are distinct, values are bit copies, pads are (-1, -inf) after the picks."""
    picks = idx[idx >= 0]
    n = picks.size
    return (np.unique(picks).size == n and np.all(idx[n:] == -1) and np.all(np.isneginf(val[n:]))
            and np.array_equal(val[:n].view(np.uint32), s[picks].view(np.uint32)))


@pytest.mark.parametrize("dist", ["normal", "coarse", "bf16", "special"])
def test_candidates_reproduce_both_other_functions(dist):
    """Special cases that reduce to the other two functions: listing every block
    gives the plain top-k; listing the blocks stage A kept gives the two-level
    result."""
    S, L = workloads.random_rows(6, 3000, seed=22, dist=dist, lengths="ragged")
    S = S.numpy()
    L = L.numpy()
    B = 8
    every = np.tile(np.arange((3000 + B - 1) // B, dtype=np.int32), (6, 1))
    for k in (1, 64, 300):
        i1, v1 = oracle.topk_candidates(S, L, every, B, k)
        i2, v2 = oracle.topk(S, L, k)
        assert equal_outputs(i1, v1, i2, v2)
    for kb, k in [(16, 100), (40, 64), (300, 512)]:
        i3, v3, blk = oracle.topk_blocked(S, L, B, kb, k)
        i4, v4 = oracle.topk_candidates(S, L, blk, B, k)
        assert equal_outputs(i3, v3, i4, v4)


def test_candidates_ignore_order_repeats_and_padding():
    rng = np.random.default_rng(6)
    S, L = workloads.random_rows(4, 5000, seed=23, dist="bf16", lengths="ragged")
    S = S.numpy()
    L = L.numpy()
    listed = np.stack([np.sort(rng.choice(625, size=50, replace=False)) for _ in range(4)]).astype(np.int32)
    i1, v1 = oracle.topk_candidates(S, L, listed, 8, 128)
    shuffled = np.stack([rng.permutation(r) for r in listed])
    noisy = np.concatenate([shuffled, listed[:, :10], np.full((4, 7), -1, np.int32),
                            np.full((4, 3), 10 ** 6, np.int32)], axis=1)
    i2, v2 = oracle.topk_candidates(S, L, noisy, 8, 128)
    assert equal_outputs(i1, v1, i2, v2)
    # no listed block: every slot is padding
    i3, v3 = oracle.topk_candidates(S, L, np.full((4, 5), -1, np.int32), 8, 16)
    assert np.all(i3 == -1) and np.all(np.isneginf(v3))


def test_listed_workload_lists_are_valid_inputs():
    """The c6 input generator: per row k_blocks distinct block ids of the row,
    ascending, reproducible from the seed."""
    w = workloads.CONFIGS["c6_listed_16"]
    c = workloads.listed_blocks("c6_listed_16").numpy()
    nb = (w.row_stride + w.block - 1) // w.block
    assert c.shape == (w.rows, w.k_blocks) and c.dtype == np.int32
    assert np.all(np.diff(c, axis=1) > 0) and c.min() >= 0 and c.max() < nb
    assert np.array_equal(c, workloads.listed_blocks("c6_listed_16").numpy())
    assert not np.array_equal(c, workloads.listed_blocks("c6_listed_16", seed=1).numpy())


# ---------------------------------------------------------------- the pins have teeth

def test_checkers_reject_planted_mistakes():
    """Corrupt a correct oracle output in the ways a buggy oracle would and check that
    the invariant checker or the brute force notices each one."""
    S, _, w = workloads.make("c1_single_4096")
    S = S.numpy()
    idx, val = oracle.topk(S, None, 512)
    assert check_invariants(S, None, 512, idx, val) == []
    # (a) tie broken by highest index instead of lowest
    t = val[0, -1]
    ties = np.nonzero(S[0] == t)[0]
    bad = idx.copy()
    bad[0, 509:] = ties[-3:][::-1]
    assert check_invariants(S, None, 512, bad, val) != []
    # (b) one element dropped (replaced by the 513th)
    order = np.lexsort((np.arange(S.shape[1]), -S[0].astype(np.float64)))
    bad = idx.copy()
    badv = val.copy()
    bad[0, 100] = order[512]
    badv[0, 100] = S[0, order[512]]
    assert check_invariants(S, None, 512, bad, badv) != []
    # (c) ascending instead of descending
    assert check_invariants(S, None, 512, idx[:, ::-1].copy(), val[:, ::-1].copy()) != []
    # (d) value bits not copied (-0 written as +0)
    z = np.array([[-0.0, 1.0]], dtype=np.float32)
    zi, zv = oracle.topk(z, None, 2)
    zv2 = zv.copy()
    zv2[0, 1] = 0.0
    assert check_invariants(z, None, 2, zi, zv) == []
    assert check_invariants(z, None, 2, zi, zv2) != []
    # (e) NaN ranked on top instead of at the bottom
    s = np.array([1.0, float("nan"), 2.0], dtype=np.float32)
    assert brute_topk_row(s, 3, 3) == [2, 0, 1]
    assert lexsort_topk_row(s, 3, 3) == [2, 0, 1]


# ---------------------------------------------------------------- bf16 scores

def _bf16_cases():
    return _load("bf16_values.jsonl")


@pytest.mark.parametrize("case", _bf16_cases(), ids=lambda c: c["bits"])
def test_bf16_widening_hand_values(case):
    """The oracle's bf16 widening gives the number worked out by hand from the
    format's fields (sign of zero and NaN-ness included)."""
    from _checks import bf16_value
    bits = int(case["bits"], 16)
    got = float(oracle.widen_bf16(np.array([bits], np.uint16))[0])
    want = _f(case["value"])
    assert bf16_value(bits) == want or (math.isnan(want) and math.isnan(bf16_value(bits)))
    if math.isnan(want):
        assert math.isnan(got)
    else:
        assert got == want and math.copysign(1.0, got) == math.copysign(1.0, want)


def test_bf16_widening_matches_field_decoding_and_torch_everywhere():
    """All 65536 patterns: the widened fp32 equals the field decoding and
    torch's own bf16 -> float32 conversion (bitwise for numbers)."""
    from _checks import bf16_value
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.widen_bf16(bits)
    lib = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    nan = np.isnan(got)
    assert np.array_equal(nan, np.isnan(lib))
    assert np.array_equal(got[~nan].view(np.uint32), lib[~nan].view(np.uint32))
    ref = np.array([bf16_value(int(b)) for b in bits], dtype=np.float64)
    assert np.array_equal(np.isnan(ref), nan)
    assert np.array_equal(got[~nan].astype(np.float64), ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


BF16_ALPHABET = [0x0000, 0x8000, 0x3F80, 0x3F81, 0xFF80, 0x7FC0, 0x0001]  # +0 -0 1 1+2^-7 -inf NaN 2^-133


def test_bf16_topk_brute_force_small_rows():
    """Every row of length <= 4 over a 7-pattern bf16 alphabet (ties, signed
    zeros, NaN, -inf, a subnormal), every k: the oracle on bf16 bits equals
    Python `sorted` over the field-decoded numbers, and its values are the
    decoded numbers."""
    from _checks import bf16_value
    for n in range(1, 5):
        for row in itertools.product(BF16_ALPHABET, repeat=n):
            bits = np.array(row, np.uint16)
            dec = [bf16_value(b) for b in row]
            for k in range(1, n + 2):
                idx, val = oracle.topk_bf16(bits[None, :], None, k, nthreads=1)
                want = brute_topk_row(dec, n, k)
                assert idx[0].tolist() == want, (row, k)
                for j, i in enumerate(want):
                    if i < 0:
                        assert val[0, j] == -np.inf
                    elif math.isnan(dec[i]):
                        assert np.isnan(val[0, j])
                    else:
                        assert float(val[0, j]) == dec[i] and np.signbit(val[0, j]) == (math.copysign(1, dec[i]) < 0)


def test_bf16_blocked_and_candidates_brute_force():
    """Two-level and listed-candidate oracles on bf16 bits against their Python
    restatements over the field-decoded numbers."""
    from _checks import bf16_value
    rng = np.random.default_rng(7)
    pool = np.array(BF16_ALPHABET + [0x4049, 0xC0A0, 0x7F80], np.uint16)
    for _ in range(200):
        n = int(rng.integers(1, 40))
        bits = pool[rng.integers(0, pool.size, n)]
        dec = [bf16_value(int(b)) for b in bits]
        B = int(rng.choice([4, 8]))
        kb = int(rng.integers(1, 6))
        k = int(rng.integers(1, 12))
        idx, _, blk = oracle.topk_blocked_bf16(bits[None, :], None, B, kb, k, nthreads=1)
        wi, wb = brute_blocked_row(dec, n, B, kb, k)
        assert idx[0].tolist() == wi and blk[0].tolist() == wb
        listed = rng.integers(-1, (n + B - 1) // B + 1, 5).astype(np.int32)
        ci, _ = oracle.topk_candidates_bf16(bits[None, :], None, listed[None, :], B, k, nthreads=1)
        assert ci[0].tolist() == brute_candidates_row(dec, n, B, listed.tolist(), k)
