"""C-ABI checks that need no GPU: the library loads, exports every function the
header declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in sorted(os.listdir(os.path.join(ROOT, "include")))
           if h.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    from sparse_attention_indexer_lt_gb300 import build, load
    build.build()
    return load()


def declared_functions():
    text = "".join(open(h).read() for h in HEADERS)
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lt_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ["lt_topk", "lt_topk_blocked", "lt_topk_ex", "lt_topk_blocked_ex", "lt_topk_candidates",
              "lt_topk_candidates_ex", "lt_topk_plan", "lt_status_string", "lt_version", "lt_topk_bf16",
              "lt_topk_blocked_bf16", "lt_topk_candidates_bf16", "lt_test_inject", "lt_compress",
              "lt_compress_decode", "lt_topk_candidates_plan"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_status_strings_and_version(lib):
    assert lib.lt_status_string(0) == b"ok"
    assert b"invalid" in lib.lt_status_string(1)
    assert lib.lt_status_string(99) == b"unknown status"
    assert lib.lt_version() >= 100


P = ctypes.c_void_p


def _topk(lib, scores, lengths, rows, stride, k, oi, ov, fc=0, fk=0, dtype=0):
    return lib.lt_topk_ex(scores, dtype, lengths, rows, stride, k, oi, ov, fc, 0, 0, fk, None, None, None)


def test_invalid_arguments_rejected_without_launch(lib):
    fake = P(0x1000)  # never dereferenced: validation fails first
    assert _topk(lib, None, None, 1, 16, 4, fake, None) == 1  # scores NULL
    assert _topk(lib, fake, None, 1, 16, 4, None, None) == 1  # out_idx NULL
    assert _topk(lib, fake, None, -1, 16, 4, fake, None) == 1  # rows < 0
    assert _topk(lib, fake, None, 1, 0, 4, fake, None) == 1   # row_stride < 1
    assert _topk(lib, fake, None, 1, 16, 0, fake, None) == 1  # k < 1
    assert _topk(lib, fake, None, 1, 16, 4, fake, None, fc=3) == 1  # cluster not a power of two
    assert _topk(lib, fake, None, 1, 16, 4096, fake, None) == 2  # k > LT_MAX_K
    assert _topk(lib, fake, None, 1, (1 << 30) + 1, 4, fake, None) == 2  # row too long
    assert lib.lt_topk_ex(fake, 0, None, 1, 16, 4, fake, None, 0, 1024, 0, 0, None, None, None) == 1  # bad threads
    assert _topk(lib, fake, None, 1, 16, 4, fake, None, dtype=2) == 1  # unknown score type
    assert _topk(lib, fake, None, 1, 16, 4, fake, None, dtype=-1) == 1
    assert _topk(lib, fake, None, 1, 16, 4, fake, None, fk=3) == 1  # unknown kernel
    assert _topk(lib, fake, None, 1, 16, 4, fake, None, fk=-1) == 1
    # rows == 0 is a valid no-op
    assert _topk(lib, None, None, 0, 16, 4, None, None) == 0


def test_blocked_invalid_arguments(lib):
    fake = P(0x1000)
    g = lib.lt_topk_blocked_ex

    def f(*a, dtype=0):
        return g(a[0], dtype, *a[1:])

    assert f(fake, None, 1, 64, 0, 4, 4, fake, None, None, 0, 0, 0, None, None, None) == 1   # block < 1
    assert f(fake, None, 1, 64, 8, 0, 4, fake, None, None, 0, 0, 0, None, None, None) == 1   # k_blocks < 1
    assert f(fake, None, 1, 64, 6, 4, 4, fake, None, None, 0, 0, 0, None, None, None) == 2   # block unsupported
    assert f(fake, None, 1, 64, 8, 5000, 4, fake, None, None, 0, 0, 0, None, None, None) == 2
    assert f(fake, None, 1, 64, 8, 4, 4, fake, None, None, 0, 0, 0, None, None, None, dtype=5) == 1  # score type
    assert f(None, None, 0, 64, 8, 4, 4, None, None, None, 0, 0, 0, None, None, None) == 0


def test_candidates_invalid_arguments(lib):
    fake = P(0x1000)
    f = lib.lt_topk_candidates_ex

    def call(scores, rows, stride, block, cand, n_cand, k, oi, dtype=0):
        return f(scores, dtype, None, rows, stride, block, cand, n_cand, k, oi, None, 0, 0, 0, None, None, None)

    assert call(fake, 1, 64, 0, fake, 4, 4, fake) == 1          # block < 1
    assert call(fake, 1, 64, 8, fake, -1, 4, fake) == 1         # n_cand < 0
    assert call(fake, 1, 64, 8, None, 4, 4, fake) == 1          # no list for n_cand > 0
    assert call(fake, 1, 64, 8, fake, 4, 0, fake) == 1          # k < 1
    assert call(None, 1, 64, 8, fake, 4, 4, fake) == 1          # scores NULL
    assert call(fake, 1, 64, 6, fake, 4, 4, fake) == 2          # block unsupported
    assert call(fake, 1, 64, 8, fake, 4, 4096, fake) == 2       # k > LT_MAX_K
    assert call(fake, 1, 262148, 4, fake, 4, 4, fake) != 1      # more than 65536 blocks: valid (long rows)
    assert call(fake, 1, 64, 8, fake, 4, 4, fake, dtype=3) == 1  # unknown score type
    assert call(None, 0, 64, 8, None, 4, 4, None) == 0          # rows == 0: nothing to do


def test_compress_invalid_arguments(lib):
    fake = P(0x1000)
    f = lib.lt_compress
    assert f(fake, fake, fake, None, 1, 16, 8, 0, fake, 0, None) == 1      # ratio < 1
    assert f(fake, fake, fake, None, 1, 16, 0, 4, fake, 0, None) == 1      # dim < 1
    assert f(fake, fake, fake, None, 1, 0, 8, 4, fake, 0, None) == 1       # no tokens
    assert f(fake, fake, fake, None, -1, 16, 8, 4, fake, 0, None) == 1     # rows < 0
    assert f(fake, fake, fake, None, 1, 16, 8, 4, fake, 7, None) == 1      # unknown dtype
    assert f(None, fake, fake, None, 1, 16, 8, 4, fake, 0, None) == 1      # kv NULL
    assert f(fake, fake, None, None, 1, 16, 8, 4, fake, 0, None) == 1      # bias NULL
    assert f(fake, fake, fake, None, 1, 1 << 14, 8, 8192, fake, 0, None) == 2  # ratio > LT_MAX_RATIO
    assert f(None, None, None, None, 0, 16, 8, 4, None, 0, None) == 0      # rows == 0
    assert f(fake, fake, fake, None, 1, 3, 8, 4, fake, 0, None) == 0       # no complete block: no-op
    d = lib.lt_compress_decode
    assert d(fake, fake, fake, fake, fake, fake, 1, 8, 0, fake, 0, None) == 1   # ratio < 1
    assert d(fake, fake, fake, fake, None, fake, 1, 8, 4, fake, 0, None) == 1   # ring NULL
    assert d(fake, fake, fake, fake, fake, fake, 1, 8, 4, fake, 2, None) == 1   # dtype
    assert d(None, None, None, None, None, None, 0, 8, 4, None, 0, None) == 0   # no sequences


def test_plan_rejects_bad_arguments(lib):
    from sparse_attention_indexer_lt_gb300 import PlanInfo
    info = PlanInfo()
    f = lib.lt_topk_plan
    assert f(0, 64, 4, 0, 4, 1, 0, 0, 0, 1, ctypes.byref(info)) == 1      # rows < 1
    assert f(1, 64, 4, 0, 4, 1, 0, 0, 0, 1, None) == 1                    # no output struct
    assert f(1, 64, 4, 0, 4, 1, 0, 0, 7, 1, ctypes.byref(info)) == 1      # unknown kernel
    assert f(1, 64, 4, 1, 6, 4, 0, 0, 0, 1, ctypes.byref(info)) == 2      # block unsupported
    g = lib.lt_topk_candidates_plan
    assert g(0, 64, 8, 4, 4, 0, 0, 0, 0, 1, ctypes.byref(info)) == 1      # rows < 1
    assert g(1, 64, 8, -1, 4, 0, 0, 0, 0, 1, ctypes.byref(info)) == 1     # negative list length
    assert g(1, 64, 8, 4, 4, 5, 0, 0, 0, 1, ctypes.byref(info)) == 1      # unknown dtype
    assert g(1, 64, 8, 4, 4, 0, 3, 0, 0, 1, ctypes.byref(info)) == 1      # cluster size 3
    assert g(1, 64, 6, 4, 4, 0, 0, 0, 0, 1, ctypes.byref(info)) == 2      # block unsupported
    assert g(1, 64, 8, 4, 4, 0, 0, 0, 0, 1, None) == 1                    # no output struct


def test_valid_calls_without_a_device_report_a_cuda_error(lib):
    """With no usable GPU every valid call fails in the CUDA runtime: the plain
    entry points (fp32 and bf16) return LT_ERR_CUDA (3), having launched nothing."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present: the CUDA runtime does not fail here")
    fake = P(0x1000)
    assert lib.lt_topk(fake, None, 1, 16, 4, fake, None, None) == 3
    assert lib.lt_topk_bf16(fake, None, 1, 16, 4, fake, None, None) == 3
    assert lib.lt_topk_blocked(fake, None, 1, 16, 8, 4, 4, fake, None, None, None) == 3
    assert lib.lt_topk_blocked_bf16(fake, None, 1, 16, 8, 4, 4, fake, None, None, None) == 3
    assert lib.lt_topk_candidates(fake, None, 1, 16, 8, fake, 2, 4, fake, None, None) == 3
    assert lib.lt_topk_candidates_bf16(fake, None, 1, 16, 8, fake, 2, 4, fake, None, None) == 3


def test_binding_refuses_cpu_tensors():
    import torch
    import sparse_attention_indexer_lt_gb300 as lt
    with pytest.raises(TypeError):
        lt.topk(torch.zeros(2, 8), None, 2)
