"""Independent checkers used to pin the oracle and to validate GPU outputs.

Nothing here calls the oracle or the CUDA library: each checker restates the
selection rule in a different form (Python tuple sort, numpy lexsort, vectorised
invariants) so that a mistake in either implementation shows up as a mismatch.

Order used throughout: score descending, index ascending; -0.0 equals +0.0;
NaN ranks below every number and NaNs tie with each other.
"""
from __future__ import annotations

import math

import numpy as np


def _sort_key(x: float, i: int):
    if math.isnan(x):
        return (1, 0.0, i)
    return (0, -x, i)


def brute_topk_row(s, L: int, k: int):
    """Python `sorted` over (nan-flag, -score, index) tuples."""
    order = sorted(range(L), key=lambda i: _sort_key(float(s[i]), i))
    picked = order[:k]
    return picked + [-1] * (k - len(picked))


def lexsort_topk_row(s, L: int, k: int):
    """numpy lexsort on (index, -score); NaN sorts last in ascending order."""
    x = np.asarray(s[:L], dtype=np.float64)
    idx = np.arange(L)
    order = np.lexsort((idx, -x))
    picked = order[:k].tolist()
    return picked + [-1] * (k - len(picked))


def brute_blocked_row(s, L: int, B: int, k_blocks: int, k: int):
    """The two-level rule restated with Python tuples (blocks then positions)."""
    nb = (L + B - 1) // B
    bkeys = []
    for b in range(nb):
        vals = [float(s[i]) for i in range(b * B, min(L, (b + 1) * B))]
        best = min(vals, key=lambda v: _sort_key(v, 0)[:2])  # smallest sort key = largest score
        bkeys.append((_sort_key(best, b)))
    kept = sorted(range(nb), key=lambda b: bkeys[b])[:k_blocks]
    kept_sorted = sorted(kept)
    cand = [i for b in kept_sorted for i in range(b * B, min(L, (b + 1) * B))]
    order = sorted(cand, key=lambda i: _sort_key(float(s[i]), i))[:k]
    out_idx = order + [-1] * (k - len(order))
    out_blocks = kept_sorted + [-1] * (k_blocks - len(kept_sorted))
    return out_idx, out_blocks


def brute_candidates_row(s, L: int, B: int, listed, k: int):
    """Top-k among the positions of the listed blocks, restated with Python tuples:
    the listed ids that name a block of [0, L) form a set; its valid positions
    are ranked like brute_topk_row."""
    nb = (L + B - 1) // B
    blocks = {int(b) for b in listed if 0 <= int(b) < nb}
    cand = [i for i in range(L) if i // B in blocks]
    order = sorted(cand, key=lambda i: _sort_key(float(s[i]), i))[:k]
    return order + [-1] * (k - len(order))


def _rank_tuple(x: np.ndarray):
    """(nan, -x) as two arrays usable for lexicographic comparison."""
    nan = np.isnan(x)
    neg = np.where(nan, 0.0, -x.astype(np.float64))
    return nan.astype(np.int8), neg


def check_invariants(scores: np.ndarray, lengths, k: int, idx: np.ndarray, val: np.ndarray,
                     rows=None) -> list[str]:
    """Invariants every correct top-k output satisfies; returns a list of failures.

    * exactly min(k, L) picks, then (-1, -inf) padding;
    * picks distinct and inside [0, L);
    * val is a bit copy of scores[idx];
    * picks strictly decreasing in (score, -index) under the order above;
    * the last pick ranks above every position that was not picked.
    """
    errs: list[str] = []
    R, S = scores.shape
    rows = range(R) if rows is None else rows
    sbits = scores.view(np.uint32)
    for r in rows:
        L = S if lengths is None else int(min(max(int(lengths[r]), 0), S))
        K = min(k, L)
        ir, vr = idx[r], val[r]
        if np.any(ir[K:] != -1) or np.any(~np.isneginf(vr[K:])):
            errs.append(f"row {r}: bad padding")
            continue
        p = ir[:K].astype(np.int64)
        if np.any(p < 0) or np.any(p >= L):
            errs.append(f"row {r}: pick out of range")
            continue
        if np.unique(p).size != K:
            errs.append(f"row {r}: duplicate picks")
            continue
        if np.any(vr[:K].view(np.uint32) != sbits[r, p]):
            errs.append(f"row {r}: value bits differ from scores[idx]")
            continue
        if K == 0:
            continue
        x = scores[r, p]
        nan, neg = _rank_tuple(x)
        # consecutive pairs must be strictly increasing in (nan, -x, idx)
        a = (nan[:-1], neg[:-1], p[:-1])
        b = (nan[1:], neg[1:], p[1:])
        lt = (a[0] < b[0]) | ((a[0] == b[0]) & ((a[1] < b[1]) | ((a[1] == b[1]) & (a[2] < b[2]))))
        if not np.all(lt):
            errs.append(f"row {r}: output not ordered by (score desc, index asc)")
            continue
        if K < L:
            mask = np.ones(L, dtype=bool)
            mask[p] = False
            rest = np.nonzero(mask)[0]
            xr = scores[r, rest]
            nr, gr = _rank_tuple(xr)
            ln, lg = nan[-1], neg[-1]
            li = p[-1]
            above = (ln < nr) | ((ln == nr) & ((lg < gr) | ((lg == gr) & (li < rest))))
            if not np.all(above):
                errs.append(f"row {r}: a non-pick ranks above the last pick")
    return errs


def equal_outputs(idx_a, val_a, idx_b, val_b) -> bool:
    """Bit-exact equality of two (idx, val) outputs."""
    return (np.array_equal(np.asarray(idx_a), np.asarray(idx_b))
            and np.array_equal(np.asarray(val_a).view(np.uint32), np.asarray(val_b).view(np.uint32)))


def bf16_value(bits: int) -> float:
    """The number a bf16 bit pattern denotes, from the format's fields (1 sign
    bit, 8 exponent bits with bias 127, 7 fraction bits), not from a bit shift."""
    s = -1.0 if (bits >> 15) & 1 else 1.0
    e = (bits >> 7) & 0xFF
    f = bits & 0x7F
    if e == 0xFF:
        return s * math.inf if f == 0 else math.nan
    if e == 0:
        return s * math.ldexp(f / 128.0, -126)
    return s * math.ldexp(1.0 + f / 128.0, e - 127)
