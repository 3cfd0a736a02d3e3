"""The no-allocation attention entry point (csa2_sparse_attn_fp4_noalloc).

Some callers may not allocate device memory at all (an engine that plans all
of its device memory before serving, or code that must avoid cudaMalloc /
cudaFree because they can synchronise the device).  For them the library
offers a variant of the sparse attention whose split-KV scratch is an array
built into the library.  This file checks, through the C ABI, that the variant
gives the same output as the regular entry point (within the attention
tolerance of the other tests) on two calls in a row with different inputs, and
that the array covers every supported shape on this GPU.

It is collected last on purpose, and it needs no other test to have run.
Marked gpu.
"""
import ctypes

import numpy as np
import pytest
import torch

import gen

pytestmark = pytest.mark.gpu
DEV = "cuda"
ATTN_RTOL = 2e-3


def _inputs(seed, B, N, K=512, H=64, D=576):
    w = gen.scaled(gen.FULL_BATCHED_DECODE, B=B, N=N, K=K, H=H, seed=seed)
    codes, scales = gen.fp4_planes(seed, 1, B * N, D, device=DEV)
    kl = torch.full((B,), N, dtype=torch.int32)
    idx = gen.random_indices(w, kl, frac_pad=0.05)
    q = gen.normal_bf16(seed, 2, (B, 1, H, D), device=DEV)
    return q, codes, scales, idx.to(DEV), kl.to(DEV)


def _rel_err(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    den = np.abs(b).max(-1)
    num = np.abs(a - b).max(-1)
    den[den == 0] = 1.0
    return float((num / den).max())


def test_noalloc_matches_workspace_entry_point_twice():
    import sparse_attention_fp4_quantize_gb300 as csa2
    lib = csa2._lib
    sm = 1.0 / 576 ** 0.5
    for call, seed in enumerate((11, 12)):
        B, N = (8, 3000) if call == 0 else (32, 5000)
        q, codes, scales, idx, kl = _inputs(seed, B, N)
        need = csa2.csa2_sparse_attn_workspace_bytes(B, 1, 64, 576, 512, 512)
        assert 0 < need <= csa2.noalloc_max_scratch_bytes()
        ref = torch.empty(B, 1, 64, 512, device=DEV)
        ref_lse = torch.empty(B, 1, 64, device=DEV)
        ws = torch.empty(need, dtype=torch.uint8, device=DEV)
        csa2.csa2_sparse_attn_fp4(0, q, codes, scales, N, idx, ref, sm, kv_len=kl, lse=ref_lse, workspace=ws)
        out = torch.full((B, 1, 64, 512), 9.0, device=DEV)
        lse = torch.full((B, 1, 64), 9.0, device=DEV)
        stream = torch.cuda.current_stream().cuda_stream
        P = ctypes.c_void_p
        rc = lib.csa2_sparse_attn_fp4_noalloc(0, B, 1, 64, 576, 512, P(q.data_ptr()), P(codes.data_ptr()),
                                              P(scales.data_ptr()), N, P(idx.data_ptr()), 512, P(kl.data_ptr()),
                                              sm, P(out.data_ptr()), 2, P(lse.data_ptr()), None, P(stream))
        assert rc == 0, lib.csa2_last_error().decode()
        torch.cuda.synchronize()
        assert _rel_err(out, ref) <= ATTN_RTOL
        assert torch.allclose(lse, ref_lse, rtol=1e-5, atol=1e-5)


def test_noalloc_scratch_covers_every_shape_on_this_gpu():
    """The split policy keeps splits x tokens x head blocks <= the SM count, so
    no supported shape needs more than SMs x 64 x 513 x 4 bytes (+256)."""
    import sparse_attention_fp4_quantize_gb300 as csa2
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    worst = sms * 64 * 513 * 4 + 256
    if worst > csa2.noalloc_max_scratch_bytes():
        pytest.skip("larger GPU: some shapes are rejected by design")
    for B, H in [(1, 64), (2, 128), (32, 64), (152, 64), (5, 64 * 30)]:
        assert csa2.csa2_sparse_attn_workspace_bytes(B, 1, H, 576, 512, 512) <= csa2.noalloc_max_scratch_bytes()
