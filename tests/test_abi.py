"""The C-ABI library builds, loads and exports every symbol include/csa2.h
declares; host-side argument validation returns the documented statuses
without touching a GPU (CPU only)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "csa2.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    path = __graft_entry__._build_module().build()
    return ctypes.CDLL(path)


def declared_functions():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(csa2_[a-z0-9_]+)\s*\(", txt)))


def test_header_declares_the_five_calls():
    names = declared_functions()
    for n in ["csa2_quantize_kv_fp4", "csa2_index_score", "csa2_build_pool", "csa2_topk", "csa2_sparse_attn_fp4"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_names_match_header(lib):
    import sparse_attention_fp4_quantize_gb300 as csa2
    assert set(csa2.exported_symbols()) == set(declared_functions())
    for n in ["csa2_quantize_kv_fp4", "csa2_index_score", "csa2_build_pool", "csa2_topk", "csa2_sparse_attn_fp4"]:
        assert callable(getattr(csa2, n))


def test_status_strings_and_version(lib):
    lib.csa2_status_string.restype = ctypes.c_char_p
    lib.csa2_status_string.argtypes = [ctypes.c_int]
    assert lib.csa2_status_string(0) == b"CSA2_OK"
    assert lib.csa2_status_string(3) == b"CSA2_ERR_WORKSPACE"
    assert lib.csa2_version() >= 100


def _last_error(lib):
    lib.csa2_last_error.restype = ctypes.c_char_p
    return lib.csa2_last_error().decode()


I64 = ctypes.c_int64
NULL = None


def test_quantize_rejects_bad_arguments_on_host(lib):
    f = lib.csa2_quantize_kv_fp4
    f.argtypes = [ctypes.c_void_p, I64, ctypes.c_int, I64, ctypes.c_void_p, I64, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    fake = ctypes.c_void_p(0x1000)
    assert f(fake, 4, 17, 17, NULL, 4, fake, fake, NULL, NULL) == 1          # D not a multiple of 16
    assert "D=17" in _last_error(lib)
    assert f(fake, 4, 64, 60, NULL, 4, fake, fake, NULL, NULL) == 1          # stride < D
    assert f(fake, 5, 64, 64, NULL, 4, fake, fake, NULL, NULL) == 1          # rows > n_slots
    assert f(ctypes.c_void_p(0x1008), 4, 64, 64, NULL, 4, fake, fake, NULL, NULL) == 1  # kv misaligned
    assert f(NULL, 0, 64, 64, NULL, 0, NULL, NULL, NULL, NULL) == 0          # empty: no-op


def test_rope_quantize_rejects_bad_arguments_on_host(lib):
    f = lib.csa2_rope_quantize_kv_fp4
    P = ctypes.c_void_p
    f.argtypes = [P, I64, ctypes.c_int, I64, P, P, I64, ctypes.c_int, P, I64, P, P, P, P]
    fake = P(0x1000)
    assert f(fake, 4, 576, 576, fake, fake, 16, 24, NULL, 4, fake, fake, NULL, NULL) == 1   # rope_dim % 16
    assert "rope_dim=24" in _last_error(lib)
    assert f(fake, 4, 576, 576, fake, fake, 0, 64, NULL, 4, fake, fake, NULL, NULL) == 1    # empty table
    assert f(fake, 4, 576, 576, fake, P(0x1004), 16, 64, NULL, 4, fake, fake, NULL, NULL) == 1  # table not 8-B aligned
    assert "misaligned" in _last_error(lib)
    assert f(fake, 4, 576, 576, P(0x1002), fake, 16, 64, NULL, 4, fake, fake, NULL, NULL) == 1  # pos misaligned
    assert f(NULL, 0, 576, 576, NULL, NULL, 16, 64, NULL, 0, NULL, NULL, NULL, NULL) == 0   # empty: no-op


def test_selftest_bounded_wait_rejects_bad_arguments_on_host(lib):
    f = lib.csa2_selftest_bounded_wait
    f.argtypes = [ctypes.c_uint32, ctypes.c_void_p, ctypes.c_void_p]
    assert f(16, NULL, NULL) == 1                          # err_flag required
    assert f(0, ctypes.c_void_p(0x1000), NULL) == 1         # max_polls 0
    assert f((1 << 22) + 1, ctypes.c_void_p(0x1000), NULL) == 1
    assert "max_polls" in _last_error(lib)


def test_dense_index_topk_rejects_bad_arguments_on_host(lib):
    P = ctypes.c_void_p
    f = lib.csa2_index_topk_dense
    f.argtypes = [ctypes.c_int, ctypes.c_int, I64, P, ctypes.c_int, P, P, ctypes.c_int, P, ctypes.c_int, P, P, P,
                  ctypes.c_size_t, P]
    wsb = lib.csa2_index_topk_dense_workspace_bytes
    wsb.argtypes = [ctypes.c_int, ctypes.c_int, I64, ctypes.c_int]
    wsb.restype = ctypes.c_size_t
    fake = P(0x1000)
    FP8, BF16 = 1, 0
    need = wsb(1, 64, 4096, 512)
    assert need == 64 * (4096 // 8) * 4                                                   # 4 B per 8 positions per query
    assert f(1, 64, 4096, fake, BF16, fake, fake, BF16, fake, 512, fake, NULL, fake, need, NULL) == 1   # bf16
    assert f(1, 64, 4096, fake, FP8, fake, fake, FP8, fake, 0, fake, NULL, fake, need, NULL) == 1       # K = 0
    assert f(1, 64, 4096, fake, FP8, fake, fake, FP8, fake, 4096, fake, NULL, fake, need, NULL) == 1    # K > 2048
    assert f(1, 64, 262145, fake, FP8, fake, fake, FP8, fake, 512, fake, NULL, fake, need, NULL) == 2   # N too large
    assert f(1, 64, 4096, fake, FP8, fake, fake, FP8, fake, 512, fake, NULL, fake, need - 1, NULL) == 3  # workspace
    assert f(1, 64, 4096, fake, FP8, fake, fake, FP8, NULL, 512, fake, NULL, fake, need, NULL) == 1     # kv_len null
    assert f(0, 64, 4096, NULL, FP8, NULL, NULL, FP8, NULL, 512, NULL, NULL, NULL, 0, NULL) == 0        # empty: no-op


def test_index_score_rejects_bad_arguments_on_host(lib):
    f = lib.csa2_index_score
    P = ctypes.c_void_p
    f.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, I64, P, ctypes.c_int, P, P, ctypes.c_int, P, P,
                  ctypes.c_int, P, P, P]
    fake = P(0x1000)
    assert f(2, 1, 1, 10, NULL, 1, NULL, NULL, 1, NULL, NULL, 0, NULL, NULL, NULL) == 0   # REUSE: no work
    assert f(7, 1, 1, 10, fake, 1, fake, fake, 1, fake, NULL, 0, fake, NULL, NULL) == 1   # bad mode
    assert f(0, 1, 1, 10, fake, 1, fake, fake, 0, fake, NULL, 0, fake, NULL, NULL) == 1   # q_dt != k_dt
    assert f(1, 1, 1, 10, fake, 1, fake, fake, 1, fake, NULL, 8, fake, NULL, NULL) == 1   # REINDEX w/o pool
    assert f(1, 1, 1, 10, fake, 1, fake, fake, 1, fake, fake, 4096, fake, NULL, NULL) == 1  # P > 2048
    assert f(0, 1, 1, 10, fake, 1, fake, fake, 1, fake, fake, 8, fake, NULL, NULL) == 1   # FULL with pool


def test_topk_and_pool_reject_bad_arguments_on_host(lib):
    P = ctypes.c_void_p
    t = lib.csa2_topk
    t.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, I64, P, P, P, ctypes.c_int, ctypes.c_int, P, P,
                  ctypes.c_size_t, P]
    fake = P(0x1000)
    assert t(2, 1, 1, 10, NULL, NULL, NULL, 0, 512, NULL, NULL, 0, NULL) == 0            # REUSE no-op
    assert t(0, 1, 1, 10, fake, NULL, NULL, 0, 0, fake, NULL, 0, NULL) == 1              # K = 0
    assert t(0, 1, 1, 10, fake, NULL, NULL, 0, 4096, fake, NULL, 0, NULL) == 1           # K > 2048
    assert t(1, 1, 1, 100, fake, NULL, fake, 8, 16, fake, NULL, 0, NULL) == 1            # M != 8P
    bp = lib.csa2_build_pool
    bp.argtypes = [ctypes.c_int, ctypes.c_int, I64, P, P, ctypes.c_int, ctypes.c_int, P, P, ctypes.c_size_t, P]
    assert bp(1, 1, 100, fake, fake, 2048, 4, fake, NULL, 0, NULL) == 1                 # G != 8
    assert bp(1, 1, 100, fake, fake, 4096, 8, fake, NULL, 0, NULL) == 1                 # P > 2048


def test_attention_rejects_bad_arguments_on_host(lib):
    P = ctypes.c_void_p
    f = lib.csa2_sparse_attn_fp4
    f.argtypes = [ctypes.c_int] * 6 + [P, P, P, I64, P, ctypes.c_int, P, ctypes.c_float, P, ctypes.c_int, P, P, P,
                                       ctypes.c_size_t, P]
    fake = P(0x1000)
    # unsupported head dims
    assert f(0, 1, 1, 64, 256, 192, fake, fake, fake, 10, fake, 512, NULL, 0.1, fake, 2, NULL, NULL, NULL, 0, NULL) == 2
    # bf16 output not supported
    assert f(0, 1, 1, 64, 576, 512, fake, fake, fake, 10, fake, 512, NULL, 0.1, fake, 0, NULL, NULL, NULL, 0, NULL) == 1
    # K out of range
    assert f(0, 1, 1, 64, 576, 512, fake, fake, fake, 10, fake, 0, NULL, 0.1, fake, 2, NULL, NULL, NULL, 0, NULL) == 1


def test_fused_index_topk_rejects_bad_arguments_on_host(lib):
    P = ctypes.c_void_p
    f = lib.csa2_index_topk
    f.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, I64, P, ctypes.c_int, P, P, ctypes.c_int, P, P,
                  ctypes.c_int, ctypes.c_int, P, P, ctypes.c_int, P, P]
    fake, FP8, BF16 = P(0x1000), 1, 0
    assert f(2, 1, 1, 10, NULL, FP8, NULL, NULL, FP8, NULL, NULL, 0, 512, NULL, NULL, 0, NULL, NULL) == 0   # REUSE
    assert f(5, 1, 1, 10, fake, FP8, fake, fake, FP8, fake, NULL, 0, 512, fake, NULL, 0, NULL, NULL) == 1   # bad mode
    assert f(0, 1, 1, 10, fake, BF16, fake, fake, BF16, fake, NULL, 0, 512, fake, NULL, 0, NULL, NULL) == 1  # bf16
    assert f(0, 1, 1, 10, fake, FP8, fake, fake, FP8, fake, NULL, 0, 0, fake, NULL, 0, NULL, NULL) == 1     # K = 0
    assert f(0, 1, 1, 10, fake, FP8, fake, fake, FP8, fake, fake, 8, 512, fake, NULL, 0, NULL, NULL) == 1   # FULL + pool
    assert f(0, 1, 1, 10, fake, FP8, fake, fake, FP8, fake, NULL, 0, 512, fake, fake, 4096, NULL, NULL) == 1  # P_out
    assert f(1, 1, 1, 10, fake, FP8, fake, fake, FP8, fake, NULL, 8, 512, fake, NULL, 0, NULL, NULL) == 1   # no pool
    assert f(1, 1, 1, 10, fake, FP8, fake, fake, FP8, fake, fake, 8, 512, fake, fake, 8, NULL, NULL) == 1   # pool_out
    assert f(0, 1, 1, 10, P(0x1008), FP8, fake, fake, FP8, fake, NULL, 0, 512, fake, NULL, 0, NULL, NULL) == 1  # align
    assert f(0, 1, 1, 10, fake, FP8, fake, fake, FP8, NULL, NULL, 0, 512, fake, NULL, 0, NULL, NULL) == 1   # kv_len
    assert "kv_len" in _last_error(lib) or "null" in _last_error(lib)


def test_swa_and_noalloc_attention_reject_bad_arguments_on_host(lib):
    P = ctypes.c_void_p
    f = lib.csa2_swa_attn_fp8
    f.argtypes = [ctypes.c_int] * 5 + [P, P, ctypes.c_int, P, ctypes.c_float, P, P, P, P, P, P]
    fake = P(0x1000)
    assert f(1, 1, 64, 576, 512, fake, fake, 0, fake, 0.1, NULL, NULL, fake, NULL, NULL, NULL) == 1     # W = 0
    assert f(1, 1, 64, 576, 512, fake, fake, 1024, fake, 0.1, NULL, NULL, fake, NULL, NULL, NULL) == 1  # W > 512
    assert f(1, 1, 64, 128, 64, fake, fake, 128, fake, 0.1, NULL, NULL, fake, NULL, NULL, NULL) == 2    # D = 128
    assert f(1, 1, 32, 576, 512, fake, fake, 128, fake, 0.1, NULL, NULL, fake, NULL, NULL, NULL) == 2   # H % 64
    assert f(1, 1, 64, 576, 512, fake, fake, 128, fake, 0.1, fake, NULL, fake, NULL, NULL, NULL) == 1   # o without lse
    assert f(1, 1, 64, 576, 512, P(0x1004), fake, 128, fake, 0.1, NULL, NULL, fake, NULL, NULL, NULL) == 1  # align
    assert f(0, 1, 64, 576, 512, NULL, NULL, 128, NULL, 0.1, NULL, NULL, NULL, NULL, NULL, NULL) == 0    # empty
    g = lib.csa2_sparse_attn_fp4_noalloc
    g.argtypes = [ctypes.c_int] * 6 + [P, P, P, I64, P, ctypes.c_int, P, ctypes.c_float, P, ctypes.c_int, P, P, P]
    assert g(0, 1, 1, 64, 256, 192, fake, fake, fake, 10, fake, 512, NULL, 0.1, fake, 2, NULL, NULL, NULL) == 2
    assert g(0, 1, 1, 64, 576, 512, fake, fake, fake, 10, fake, 0, NULL, 0.1, fake, 2, NULL, NULL, NULL) == 1
    assert g(7, 1, 1, 64, 576, 512, fake, fake, fake, 10, fake, 512, NULL, 0.1, fake, 2, NULL, NULL, NULL) == 1
