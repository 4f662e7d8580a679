"""CPU oracle of the fused KV compressor (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module. It shares nothing with the CUDA library.

What it computes. Compressed sparse attention keeps one KV entry per block of
``ratio`` consecutive tokens (4 for CSA, 128 for HCA: AICon 2026 Shenzhen
speaker page, outline section 1.1). The compressor builds that entry in the
order the SGLang DeepSeek-V4 inference talk notes list for the unfused flow
(section 3.1, KV compression operator fusion), whose fused form the AICon page
calls FlashCompressor (outline section 3.1): read the block's KV vectors and
scores, add a learned bias, take a softmax over the block's tokens, form the
weighted sum ("dot") of the KV vectors, store it. The pages give the step
names only; the plainest reading, taken here:

    v[t, c]  = score[t, c] + bias[t mod ratio, c]              (add)
    w[t, c]  = exp(v[t, c]) / sum_{t' in block} exp(v[t', c])   (softmax over the block's tokens)
    y[g, c]  = sum_{t in block g} w[t, c] * kv[t, c]            (dot, then store)

per channel c, for every complete block g of a row (tokens g*ratio ..
g*ratio + ratio - 1 < L); an incomplete trailing block is not emitted (its
tokens are the state a decoder keeps until the block completes). A score given
per token rather than per channel is the special case of a score constant
across channels. The softmax is evaluated as exp(v - max_t v) / sum exp(...),
the same function, in float64.
"""
from __future__ import annotations

import numpy as np


def compress(kv, score, bias, ratio: int, lengths=None) -> np.ndarray:
    """kv, score: [rows, T, d] numbers (float32, or bf16 already widened);
    bias: [ratio, d]. Returns float64 [rows, T // ratio, d]; blocks at or past
    L_r // ratio are NaN (the method does not write them)."""
    kv = np.asarray(kv, dtype=np.float64)
    sc = np.asarray(score, dtype=np.float64)
    b = np.asarray(bias, dtype=np.float64)
    if kv.ndim != 3 or sc.shape != kv.shape or b.shape != (ratio, kv.shape[2]) or ratio < 1:
        raise ValueError("kv/score [rows, T, d], bias [ratio, d], ratio >= 1")
    rows, T, d = kv.shape
    y = np.full((rows, T // ratio, d), np.nan)
    for r in range(rows):
        L = T if lengths is None else int(min(max(int(lengths[r]), 0), T))
        n = L // ratio
        if n == 0:
            continue
        x = kv[r, :n * ratio].reshape(n, ratio, d)                 # read
        v = sc[r, :n * ratio].reshape(n, ratio, d) + b[None, :, :]  # add
        e = np.exp(v - v.max(axis=1, keepdims=True))                # softmax over the block's tokens
        w = e / e.sum(axis=1, keepdims=True)
        y[r, :n] = (w * x).sum(axis=1)                              # dot; the caller stores
    return y


def decode_step(kv_new, score_new, bias, ring_kv, ring_score, pos, ratio: int):
    """One decode step for a batch of sequences (the ring-buffer form of the same
    compressor). Token pos[s] of sequence s enters slot pos[s] mod ratio of its
    ring; when it completes a block (pos mod ratio == ratio - 1) the block's
    entry is produced from the ring exactly as ``compress`` does. Updates the
    rings in place; returns (y float64 [seqs, d], done bool [seqs])."""
    seqs, d = kv_new.shape
    y = np.full((seqs, d), np.nan)
    done = np.zeros(seqs, dtype=bool)
    for s in range(seqs):
        slot = int(pos[s]) % ratio
        ring_kv[s, slot] = kv_new[s]
        ring_score[s, slot] = score_new[s]
        if slot == ratio - 1:
            y[s] = compress(ring_kv[s][None], ring_score[s][None], bias, ratio)[0, 0]
            done[s] = True
    return y, done
