"""The Python binding's own checks (CPU only): the C calls see plain pointers,
so the binding refuses tensors whose element size does not match what the
call reads or writes, and buffers smaller than the call touches, before any
call is made.  The library is replaced by a recorder here, so no kernel runs
and CPU tensors stand in for device ones."""
from __future__ import annotations

import pytest
import torch

import sparse_attention_fp4_quantize_gb300 as csa2


class _FakeLib:
    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def call(*a):
            self.calls.append(name)
            return 0
        return call


@pytest.fixture()
def fake(monkeypatch):
    lib = _FakeLib()
    monkeypatch.setattr(csa2, "_lib", lib)
    monkeypatch.setattr(csa2, "_on_device", lambda t: True)   # the binding's own device check only
    monkeypatch.setattr(csa2, "_stream", lambda s: None)
    return lib


def _z(*shape, dtype=torch.float32):
    return torch.zeros(*shape, dtype=dtype)


def test_valid_arguments_reach_the_library(fake):
    B, T, N, H, D, dv, K = 2, 1, 100, 64, 576, 512, 16
    i32, u8, i16 = torch.int32, torch.uint8, torch.int16
    csa2.csa2_quantize_kv_fp4(_z(5, D, dtype=i16), _z(8, D // 2, dtype=u8), _z(8, D // 16, dtype=u8),
                              dst_slot=_z(5, dtype=torch.int64), err_flag=_z(1, dtype=i32))
    csa2.csa2_index_score(0, _z(B, T, 4, 64, dtype=u8), _z(B, T, 4), _z(B, N, 64, dtype=u8), _z(B * T, dtype=i32),
                          _z(B, T, N))
    csa2.csa2_topk(0, _z(B, T, N), _z(B, T, K, dtype=i32), kv_len=_z(B * T, dtype=i32))
    csa2.csa2_build_pool(_z(B, T, N), _z(B * T, dtype=i32), _z(B, T, 2048, dtype=i32))
    csa2.csa2_index_topk(0, _z(B, T, 4, 64, dtype=u8), _z(B, T, 4), _z(B, N, 64, dtype=u8), _z(B * T, dtype=i32),
                         _z(B, T, K, dtype=i32), pool_out=_z(B, T, 2048, dtype=i32))
    csa2.csa2_sparse_attn_fp4(0, _z(B, T, H, D, dtype=i16), _z(B * N, D // 2, dtype=u8),
                              _z(B * N, D // 16, dtype=u8), N, _z(B, T, K, dtype=i32), _z(B, T, H, dv), 0.1,
                              kv_len=_z(B * T, dtype=i32), lse=_z(B, T, H))
    csa2.csa2_swa_attn_fp8(_z(B, T, H, D, dtype=i16), _z(B, 128, D, dtype=u8), _z(B * T, dtype=i32),
                           _z(B, T, H, dv), 0.1, o_sparse=_z(B, T, H, dv), lse_sparse=_z(B, T, H))
    assert fake.calls == ["csa2_quantize_kv_fp4", "csa2_index_score", "csa2_topk", "csa2_build_pool",
                          "csa2_index_topk", "csa2_sparse_attn_fp4", "csa2_swa_attn_fp8"]


def test_wrong_element_sizes_are_refused(fake):
    B, T, N, H, D, dv, K = 2, 1, 100, 64, 576, 512, 16
    i32, u8, i16 = torch.int32, torch.uint8, torch.int16
    q, codes, scales = _z(B, T, H, D, dtype=i16), _z(B * N, D // 2, dtype=u8), _z(B * N, D // 16, dtype=u8)
    idx, out = _z(B, T, K, dtype=i32), _z(B, T, H, dv)
    with pytest.raises(TypeError):                                       # fp16 output: half the bytes
        csa2.csa2_sparse_attn_fp4(0, q, codes, scales, N, idx, out.half(), 0.1)
    with pytest.raises(TypeError):                                       # int64 indices
        csa2.csa2_sparse_attn_fp4(0, q, codes, scales, N, idx.long(), out, 0.1)
    with pytest.raises(TypeError):                                       # fp32 query
        csa2.csa2_sparse_attn_fp4(0, q.float(), codes, scales, N, idx, out, 0.1)
    with pytest.raises(TypeError):                                       # fp16 query: bf16's size, other values
        csa2.csa2_sparse_attn_fp4(0, q.half(), codes, scales, N, idx, out, 0.1)
    with pytest.raises(TypeError):                                       # fp16 query in the window branch
        csa2.csa2_swa_attn_fp8(q.half(), _z(B, 128, D, dtype=u8), _z(B * T, dtype=i32), out, 0.1)
    with pytest.raises(TypeError):                                       # fp16 kv rows
        csa2.csa2_quantize_kv_fp4(_z(5, D, dtype=torch.float16), _z(5, D // 2, dtype=u8), _z(5, D // 16, dtype=u8))
    with pytest.raises(TypeError):                                       # fp16 kv rows before RoPE
        csa2.csa2_rope_quantize_kv_fp4(_z(5, D, dtype=torch.float16), _z(5, dtype=i32), _z(8, 32, 2),
                                       _z(5, D // 2, dtype=u8), _z(5, D // 16, dtype=u8))
    with pytest.raises(TypeError):                                       # int64 kv_len
        csa2.csa2_topk(0, _z(B, T, N), idx, kv_len=_z(B * T, dtype=torch.int64))
    with pytest.raises(TypeError):                                       # fp32 kv rows
        csa2.csa2_quantize_kv_fp4(_z(5, D), _z(5, D // 2, dtype=u8), _z(5, D // 16, dtype=u8))
    with pytest.raises(TypeError):                                       # float err_flag
        csa2.csa2_index_score(0, _z(B, T, 4, 64, dtype=u8), _z(B, T, 4), _z(B, N, 64, dtype=u8),
                              _z(B * T, dtype=i32), _z(B, T, N), err_flag=_z(1))
    assert fake.calls == []


def test_buffers_smaller_than_the_call_touches_are_refused(fake):
    B, T, N, H, D, dv, K = 2, 1, 100, 64, 576, 512, 16
    i32, u8, i16 = torch.int32, torch.uint8, torch.int16
    q, idx, out = _z(B, T, H, D, dtype=i16), _z(B, T, K, dtype=i32), _z(B, T, H, dv)
    with pytest.raises(ValueError):                                      # planes of one sequence for two
        csa2.csa2_sparse_attn_fp4(0, q, _z(N, D // 2, dtype=u8), _z(N, D // 16, dtype=u8), N, idx, out, 0.1)
    with pytest.raises(ValueError):                                      # lse of one head row
        csa2.csa2_sparse_attn_fp4(0, q, _z(B * N, D // 2, dtype=u8), _z(B * N, D // 16, dtype=u8), N, idx, out,
                                  0.1, lse=_z(B, T, 1))
    with pytest.raises(ValueError):                                      # scores of a shorter row
        csa2.csa2_index_score(0, _z(B, T, 4, 64, dtype=u8), _z(B, T, 4), _z(B, N, 64, dtype=u8),
                              _z(B * T, dtype=i32), _z(B, T, N - 1))
    with pytest.raises(ValueError):                                      # kv_len for one query of two
        csa2.csa2_topk(0, _z(B, T, N), idx, kv_len=_z(1, dtype=i32))
    with pytest.raises(ValueError):                                      # codes rows of the wrong width
        csa2.csa2_quantize_kv_fp4(_z(5, D, dtype=i16), _z(5, D // 4, dtype=u8), _z(5, D // 16, dtype=u8))
    with pytest.raises(ValueError):                                      # dst_slot shorter than the rows
        csa2.csa2_quantize_kv_fp4(_z(5, D, dtype=i16), _z(8, D // 2, dtype=u8), _z(8, D // 16, dtype=u8),
                                  dst_slot=_z(4, dtype=torch.int64))
    with pytest.raises(ValueError):                                      # pool_out of one row of two
        csa2.csa2_index_topk(0, _z(B, T, 4, 64, dtype=u8), _z(B, T, 4), _z(B, N, 64, dtype=u8),
                             _z(B * T, dtype=i32), idx, pool_out=_z(1, T, 2048, dtype=i32))
    assert fake.calls == []


def test_prefetch_planes_are_checked(fake):
    B, T, N, H, D, dv, K = 2, 1, 100, 64, 576, 512, 16
    i32, u8, i16 = torch.int32, torch.uint8, torch.int16
    q, idx, out = _z(B, T, H, D, dtype=i16), _z(B, T, K, dtype=i32), _z(B, T, H, dv)
    codes, scales = _z(B * N, D // 2, dtype=u8), _z(B * N, D // 16, dtype=u8)
    with pytest.raises(ValueError):                                      # next codes without next scales
        csa2.csa2_sparse_attn_fp4_prefetch(0, q, codes, scales, N, idx, out, 0.1, next_codes=codes)
    with pytest.raises(ValueError):                                      # next planes of one sequence for two
        csa2.csa2_sparse_attn_fp4_prefetch(0, q, codes, scales, N, idx, out, 0.1, next_codes=codes[:N],
                                           next_scales=scales[:N])
    assert fake.calls == []
    csa2.csa2_sparse_attn_fp4_prefetch(0, q, codes, scales, N, idx, out, 0.1, next_codes=codes, next_scales=scales)
    csa2.csa2_sparse_attn_fp4_prefetch(0, q, codes, scales, N, idx, out, 0.1)
    assert fake.calls == ["csa2_sparse_attn_fp4_prefetch"] * 2


def test_reuse_calls_and_rejected_dtypes_pass_through_to_the_library(fake):
    # Reuse mode does no work, so its buffers are not checked; bf16 indexer tensors on the FP8-only
    # fused calls are the library's to reject (it returns a status)
    csa2.csa2_topk(csa2.MODE_REUSE, _z(1, 1, 4), _z(1, 1, 16, dtype=torch.int32))
    csa2.csa2_index_topk(0, _z(1, 1, 4, 32, dtype=torch.int16), _z(1, 1, 4), _z(1, 100, 64, dtype=torch.int16),
                         _z(1, dtype=torch.int32), _z(1, 1, 16, dtype=torch.int32))
    assert fake.calls == ["csa2_topk", "csa2_index_topk"]
