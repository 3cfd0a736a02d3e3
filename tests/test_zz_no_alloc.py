"""The no-allocation attention entry point (csa2_sparse_attn_fp4_noalloc).

Some callers may not allocate device memory at all (an engine that plans all
of its device memory before serving, or code that must avoid cudaMalloc /
cudaFree because they can synchronise the device).  For them the library
offers a variant of the sparse attention whose split-KV scratch is an array
built into the library.  This file checks, through the C ABI, that the variant
gives bitwise the same output as the regular entry point on calls in a row
with different inputs, and
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


def _inputs(seed, B, N, K, H, D):
    w = gen.scaled(gen.FULL_BATCHED_DECODE, B=B, N=N, K=K, H=H, D=D, dv=D - 64, seed=seed)
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


# shapes that take the split-KV path (and so need scratch): 128-channel
# entries, and 576-channel entries with more than 1024 selected
CASES = [(11, 8, 3000, 512, 16, 128), (12, 3, 5000, 512, 32, 128), (13, 2, 4000, 1536, 64, 576)]


def test_noalloc_matches_workspace_entry_point_twice():
    import sparse_attention_fp4_quantize_gb300 as csa2
    lib = csa2._lib
    for seed, B, N, K, H, D in CASES:
        dv = D - 64
        sm = 1.0 / D ** 0.5
        q, codes, scales, idx, kl = _inputs(seed, B, N, K, H, D)
        need = csa2.csa2_sparse_attn_workspace_bytes(B, 1, H, D, dv, K)
        assert 0 < need <= csa2.noalloc_max_scratch_bytes()
        ref = torch.empty(B, 1, H, dv, device=DEV)
        ref_lse = torch.empty(B, 1, H, device=DEV)
        ws = torch.empty(need, dtype=torch.uint8, device=DEV)
        csa2.csa2_sparse_attn_fp4(0, q, codes, scales, N, idx, ref, sm, kv_len=kl, lse=ref_lse, workspace=ws)
        out = torch.full((B, 1, H, dv), 9.0, device=DEV)
        lse = torch.full((B, 1, H), 9.0, device=DEV)
        stream = torch.cuda.current_stream().cuda_stream
        P = ctypes.c_void_p
        rc = lib.csa2_sparse_attn_fp4_noalloc(0, B, 1, H, D, dv, P(q.data_ptr()), P(codes.data_ptr()),
                                              P(scales.data_ptr()), N, P(idx.data_ptr()), K, P(kl.data_ptr()),
                                              sm, P(out.data_ptr()), 2, P(lse.data_ptr()), None, P(stream))
        assert rc == 0, lib.csa2_last_error().decode()
        torch.cuda.synchronize()
        # the same kernels on the same inputs: bitwise the workspace entry point's result
        assert torch.equal(out, ref), "max rel err %g" % _rel_err(out, ref)
        assert torch.equal(lse, ref_lse)


def test_noalloc_scratch_covers_every_shape_on_this_gpu():
    """The split policy keeps splits x tokens x head blocks <= the SM count, so
    no supported shape needs more than SMs x 64 x 513 x 4 bytes (+256)."""
    import sparse_attention_fp4_quantize_gb300 as csa2
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    worst = sms * 64 * 513 * 4 + 256
    if worst > csa2.noalloc_max_scratch_bytes():
        pytest.skip("larger GPU: some shapes are rejected by design")
    for B, H, D, K in [(1, 64, 576, 2048), (2, 128, 576, 1100), (1, 16, 128, 512), (9, 64 * 16, 576, 2048),
                       (1, 16 * 150, 128, 2048)]:
        assert csa2.csa2_sparse_attn_workspace_bytes(B, 1, H, D, D - 64, K) <= csa2.noalloc_max_scratch_bytes()
