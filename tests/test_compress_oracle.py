"""Pins for the compressor oracle: hand-worked cases, closed forms, a scalar
brute force, invariants, the ring-buffer decode form, and mutants of the
oracle (a dropped bias, the softmax over channels, the wrong bias row, a
dropped normalisation) that these checks must catch. CPU only."""
import json
import math
import os

import numpy as np
import pytest

from oracle import compress as oc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _cases():
    with open(os.path.join(GOLDEN, "compress_hand_cases.jsonl")) as fh:
        return [json.loads(x) for x in fh if x.strip()]


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_hand_cases(case):
    kv = np.array(case["kv"])[None]
    sc = np.array(case["score"])[None]
    y = oc.compress(kv, sc, np.array(case["bias"]), case["ratio"])
    assert np.allclose(y[0], np.array(case["y"]), rtol=1e-12, atol=1e-12)


def brute(kv, score, bias, ratio, L):
    """The definition with Python scalars: exp of the biased score over the sum
    of exps in the block (no max shift), math.fsum for the sums."""
    T, d = len(kv), len(kv[0])
    out = []
    for g in range(L // ratio):
        row = []
        for c in range(d):
            ex = [math.exp(score[g * ratio + j][c] + bias[j][c]) for j in range(ratio)]
            den = math.fsum(ex)
            row.append(math.fsum(ex[j] / den * kv[g * ratio + j][c] for j in range(ratio)))
        out.append(row)
    return out


def _rand(rows, T, d, ratio, seed, scale=1.0):
    g = np.random.default_rng(seed)
    return (g.standard_normal((rows, T, d)), scale * g.standard_normal((rows, T, d)),
            0.5 * g.standard_normal((ratio, d)))


@pytest.mark.parametrize("ratio", [1, 2, 3, 4, 8])
def test_scalar_brute_force(ratio):
    kv, sc, b = _rand(2, 19, 5, ratio, seed=ratio)
    L = [19, 11]
    y = oc.compress(kv, sc, b, ratio, lengths=L)
    for r in range(2):
        want = brute(kv[r].tolist(), sc[r].tolist(), b.tolist(), ratio, L[r])
        n = L[r] // ratio
        assert np.allclose(y[r, :n], np.array(want).reshape(n, 5), rtol=1e-13, atol=1e-13)
        assert np.isnan(y[r, n:]).all()


def test_ratio_one_is_the_identity():
    kv, sc, b = _rand(2, 7, 3, 1, seed=1, scale=5.0)
    assert np.allclose(oc.compress(kv, sc, b, 1), kv, rtol=0, atol=1e-15)


def test_equal_biased_scores_give_the_block_mean():
    kv, _, _ = _rand(1, 16, 4, 4, seed=2)
    b = np.tile(np.array([[0.3], [-1.0], [2.0], [0.7]]), (1, 4))
    sc = -np.tile(b, (4, 1))[None]  # score + bias = 0 everywhere
    y = oc.compress(kv, sc, b, 4)
    assert np.allclose(y[0], kv[0].reshape(4, 4, 4).mean(axis=1), rtol=1e-14, atol=1e-14)


def test_a_dominant_token_is_selected():
    kv, sc, b = _rand(1, 8, 3, 4, seed=3)
    sc[0, 6, :] += 200.0  # token 6 = position 2 of block 1
    y = oc.compress(kv, sc, b, 4)
    assert np.allclose(y[0, 1], kv[0, 6], rtol=0, atol=1e-60)


def test_shift_invariance_and_convexity():
    kv, sc, b = _rand(2, 32, 6, 8, seed=4, scale=3.0)
    y = oc.compress(kv, sc, b, 8)
    shift = np.repeat(np.random.default_rng(5).standard_normal((2, 4, 1, 6)) * 7, 8, axis=2).reshape(2, 32, 6)
    assert np.allclose(oc.compress(kv, sc + shift, b, 8), y, rtol=1e-12, atol=1e-12)
    blocks = kv.reshape(2, 4, 8, 6)
    assert (y >= blocks.min(axis=2) - 1e-12).all() and (y <= blocks.max(axis=2) + 1e-12).all()


def test_linear_in_kv_and_channels_independent():
    kv, sc, b = _rand(1, 12, 5, 4, seed=6)
    kv2 = np.random.default_rng(7).standard_normal(kv.shape)
    y = oc.compress(2.0 * kv - 3.0 * kv2, sc, b, 4)
    assert np.allclose(y, 2.0 * oc.compress(kv, sc, b, 4) - 3.0 * oc.compress(kv2, sc, b, 4), atol=1e-12)
    perm = np.array([3, 0, 4, 1, 2])
    y0 = oc.compress(kv, sc, b, 4)
    assert np.allclose(oc.compress(kv[..., perm], sc[..., perm], b[:, perm], 4), y0[..., perm], atol=1e-14)


def test_decode_ring_matches_the_prefill_form():
    """Feeding tokens one at a time through the ring gives, at each completed
    block, the prefill result of that block."""
    kv, sc, b = _rand(3, 24, 4, 8, seed=8)
    ref = oc.compress(kv, sc, b, 8)
    rk = np.zeros((3, 8, 4))
    rs = np.zeros((3, 8, 4))
    for t in range(24):
        y, done = oc.decode_step(kv[:, t], sc[:, t], b, rk, rs, np.full(3, t), 8)
        assert done.all() == (t % 8 == 7)
        if t % 8 == 7:
            assert np.allclose(y, ref[:, t // 8], rtol=1e-14, atol=1e-14)


# ---------------------------------------------------------------- planted mistakes

def _mutant(kind):
    def f(kv, score, bias, ratio, lengths=None):
        kv = np.asarray(kv, np.float64)
        rows, T, d = kv.shape
        n = T // ratio
        x = kv[:, :n * ratio].reshape(rows, n, ratio, d)
        v = np.asarray(score, np.float64)[:, :n * ratio].reshape(rows, n, ratio, d)
        if kind == "no_bias":
            pass
        elif kind == "bias_by_block":
            v = v + np.asarray(bias)[np.arange(n) % ratio][None, :, None, :]
        else:
            v = v + np.asarray(bias)[None, None]
        ax = 3 if kind == "softmax_over_channels" else 2
        e = np.exp(v - v.max(axis=ax, keepdims=True))
        w = e if kind == "unnormalised" else e / e.sum(axis=ax, keepdims=True)
        return (w * x).sum(axis=2)
    return f


@pytest.mark.parametrize("kind", ["no_bias", "bias_by_block", "softmax_over_channels", "unnormalised"])
def test_checks_catch_planted_mistakes(kind):
    """Each mutant fails the hand cases or the brute force; the oracle passes both."""
    bad = _mutant(kind)
    caught = False
    for case in _cases():
        kv = np.array(case["kv"])[None]
        sc = np.array(case["score"])[None]
        if not np.allclose(bad(kv, sc, np.array(case["bias"]), case["ratio"])[0], case["y"], atol=1e-9):
            caught = True
    kv, sc, b = _rand(1, 16, 3, 4, seed=9)
    want = np.array(brute(kv[0].tolist(), sc[0].tolist(), b.tolist(), 4, 16))
    if not np.allclose(bad(kv, sc, b, 4)[0], want, atol=1e-9):
        caught = True
    assert caught, kind
