"""GPU parity of the fused KV compressor against the float64 oracle.

Tolerance (derived from the kernel's fp32 arithmetic, eps = 2^-24): the bias
add rounds once (eps |v|); each exponential is __expf, whose documented error
is at most 2 + floor(1.173 |u|) ulps (an ulp is at most 2 eps relative) for
the shifted argument u = v - max; every chunk of four tokens may rescale the
running sums once; the weight sum and the weighted sum add up `ratio` terms;
the final division rounds once. Summed per (block, channel):

    |y_gpu - y| <= eps * max_t |kv_t| * (2 ratio + 4 ceil(ratio / 4) + 7 max_t |v_t| + 20)

and a bf16 output adds its rounding, at most 2^-8 |y| (half an ulp of an
8-bit significand). A wrong weight or a dropped term is off by orders of
magnitude more.
"""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import compress as oc

pytestmark = pytest.mark.gpu
EPS = 2.0 ** -24


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_attention_indexer_lt_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _num(t):
    """A CPU float64 view of the numbers a tensor holds (bf16 widens exactly)."""
    return t.detach().cpu().float().double().numpy()


def check(y_gpu, kv, sc, bias, ratio, lengths, what):
    """Compare every written block with the oracle within the derived bound;
    unwritten blocks must still hold the sentinel."""
    kvn, scn, bn = _num(kv), _num(sc), _num(bias)
    ref = oc.compress(kvn, scn, bn, ratio, lengths)
    rows, T, d = kvn.shape
    nb = T // ratio
    got = _num(y_gpu)
    for r in range(rows):
        L = T if lengths is None else min(max(int(lengths[r]), 0), T)
        n = L // ratio
        if n:
            x = kvn[r, :n * ratio].reshape(n, ratio, d)
            v = scn[r, :n * ratio].reshape(n, ratio, d) + bn[None]
            tol = EPS * np.abs(x).max(axis=1) * (2 * ratio + 4 * math.ceil(ratio / 4) + 7 * np.abs(v).max(axis=1) + 20)
            if y_gpu.dtype == torch.bfloat16:
                tol = tol + 2.0 ** -8 * np.abs(ref[r, :n])
            err = np.abs(got[r, :n] - ref[r, :n])
            bad = err > tol
            assert not bad.any(), (f"{what}: row {r}: {int(bad.sum())} entries off; worst err "
                                   f"{float(err.max()):.3g} at tol {float(tol.flat[int(np.argmax(err - tol))]):.3g}")
        assert np.all(got[r, n:nb] == 12288.0), f"{what}: row {r}: blocks past L/ratio were written"


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("ratio", [1, 3, 4, 7, 128])
@pytest.mark.parametrize("dim", [12, 10, 512])
def test_small_shapes_ragged(dtype, ratio, dim):
    """Ragged rows (an empty one, one shorter than a block, incomplete trailing
    blocks), vector (dim % 4 == 0) and scalar layouts, odd ratios."""
    import sparse_attention_indexer_lt_gb300 as lt
    rows, T = 4, 300
    kv, sc, bias = workloads.compress_inputs(rows, T, dim, ratio, seed=ratio * 1000 + dim, dtype=dtype,
                                             score_scale=2.0)
    L = np.array([T, 0, min(ratio - 1, T), T - 5], np.int32)
    out = torch.full((rows, T // ratio, dim), 12288.0, dtype=dtype, device="cuda")
    lt.compress(kv.cuda(), sc.cuda(), bias.cuda(), ratio, torch.as_tensor(L).cuda(), out=out)
    torch.cuda.synchronize()
    check(out, kv, sc, bias, ratio, L, f"{dtype} ratio={ratio} dim={dim}")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("ratio", [64, 128])
@pytest.mark.parametrize("dim", [512, 1024])
def test_streamed_blocks(dtype, ratio, dim):
    """Blocks too large for one ring stage: two streamed side by side sharing
    each stage's bias rows (512 channels), or one at a time with its channel
    groups split over threads (1024); odd block counts leave a unit with one."""
    import sparse_attention_indexer_lt_gb300 as lt
    rows, T = 3, 700
    kv, sc, bias = workloads.compress_inputs(rows, T, dim, ratio, seed=ratio + dim, dtype=dtype, score_scale=2.0)
    L = np.array([T, T - ratio - 3, 2 * ratio + 1], np.int32)
    out = torch.full((rows, T // ratio, dim), 12288.0, dtype=dtype, device="cuda")
    lt.compress(kv.cuda(), sc.cuda(), bias.cuda(), ratio, torch.as_tensor(L).cuda(), out=out)
    torch.cuda.synchronize()
    check(out, kv, sc, bias, ratio, L, f"streamed {dtype} ratio={ratio} dim={dim}")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_unaligned_views_take_scalar_loads(dtype):
    import sparse_attention_indexer_lt_gb300 as lt
    kv, sc, bias = workloads.compress_inputs(2, 65, 16, 4, seed=5, dtype=dtype)
    big_kv = torch.zeros(2 * 65 * 16 + 1, dtype=dtype, device="cuda")
    big_sc = torch.zeros_like(big_kv)
    k2 = big_kv[1:].view(2, 65, 16)
    s2 = big_sc[1:].view(2, 65, 16)
    k2.copy_(kv.cuda())
    s2.copy_(sc.cuda())
    out = torch.full((2, 16, 16), 12288.0, dtype=dtype, device="cuda")
    lt.compress(k2, s2, bias.cuda(), 4, out=out)
    torch.cuda.synchronize()
    check(out, kv, sc, bias, 4, None, f"{dtype} unaligned")


def test_large_scores_stay_finite():
    """Scores far from zero: the running maximum keeps every exponent <= 0."""
    import sparse_attention_indexer_lt_gb300 as lt
    kv, sc, bias = workloads.compress_inputs(1, 512, 8, 128, seed=6, score_scale=40.0)
    out = torch.full((1, 4, 8), 12288.0, device="cuda")
    lt.compress(kv.cuda(), sc.cuda(), bias.cuda(), 128, out=out)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    check(out, kv, sc, bias, 128, None, "large scores")


@pytest.mark.parametrize("name", sorted(workloads.COMPRESS_CONFIGS))
def test_full_size_workloads_sampled(name):
    """The benchmark's million-token inputs (drawn on the device), the launch the
    benchmark times; 3000 sampled blocks compared with the oracle."""
    import sparse_attention_indexer_lt_gb300 as lt
    w = workloads.COMPRESS_CONFIGS[name]
    kv, sc, bias = workloads.compress_inputs(w.rows, w.tokens, w.dim, w.ratio, seed=0, device="cuda",
                                             dtype=torch.bfloat16)
    out = lt.compress(kv, sc, bias, w.ratio)
    torch.cuda.synchronize()
    nb = w.tokens // w.ratio
    g = torch.Generator().manual_seed(1)
    pick = torch.randperm(nb, generator=g)[:3000].sort().values
    tok = (pick[:, None] * w.ratio + torch.arange(w.ratio)[None]).reshape(-1).cuda()
    kv_s = kv[0, tok].view(1, -1, w.dim)
    sc_s = sc[0, tok].view(1, -1, w.dim)
    sub = torch.full((1, pick.numel(), w.dim), 12288.0, dtype=torch.bfloat16)
    sub[0] = out[0, pick.cuda()].cpu()
    check(sub, kv_s, sc_s, bias, w.ratio, None, name)
    del kv, sc, out
    torch.cuda.empty_cache()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("ratio", [4, 5, 128])
def test_decode_steps_match_prefill(dtype, ratio):
    """Tokens fed one per step through the two ring buffers: each completed
    block equals the prefill entry of that block (same kernel arithmetic); the
    sequences start at different positions, one is idle (pos < 0)."""
    import sparse_attention_indexer_lt_gb300 as lt
    seqs, d = 5, 16
    T = 2 * ratio + 3
    kv, sc, bias = workloads.compress_inputs(seqs, T, d, ratio, seed=ratio, dtype=dtype)
    kvd, scd, bd = kv.cuda(), sc.cuda(), bias.cuda()
    ref = lt.compress(kvd, scd, bd, ratio)
    ring_k = torch.zeros(seqs, ratio, d, dtype=dtype, device="cuda")
    ring_s = torch.zeros_like(ring_k)
    out = torch.full((seqs, d), 12288.0, dtype=dtype, device="cuda")
    for t in range(T):
        pos = torch.full((seqs,), t, dtype=torch.int32)
        pos[4] = -1
        out.fill_(12288.0)
        lt.compress_decode(kvd[:, t].contiguous(), scd[:, t].contiguous(), bd, ring_k, ring_s, pos.cuda(), out)
        torch.cuda.synchronize()
        o = out.cpu()
        if t % ratio == ratio - 1:
            assert torch.equal(o[:4], ref[:4, t // ratio].cpu()), f"step {t}"
        else:
            assert bool((o[:4] == 12288.0).all())
        assert bool((o[4] == 12288.0).all())
    # and the oracle's ring form agrees on the last completed block
    check_blocks = ref[:, (T // ratio) - 1].cpu()
    want = oc.compress(_num(kv[:, :(T // ratio) * ratio]), _num(sc[:, :(T // ratio) * ratio]), _num(bias), ratio)
    assert np.allclose(_num(check_blocks)[:4], want[:4, -1], rtol=2.0 ** -7, atol=1e-6)
