"""csa2_swa_attn_fp8 (sliding-window branch over FP8 window KV, merged with
the sparse branch by log-sum-exp) against the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gen
import oracle
from helpers import check_attn, check_lse

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def csa2():
    import sparse_attention_fp4_quantize_gb300 as lib
    return lib


def _inputs(seed, B, T, H, W):
    q = gen.normal_bf16(seed, 1, (B, T, H, 576))
    kv = gen.e4m3_bytes(torch.randn(B, W, 576, generator=torch.Generator().manual_seed(seed)))
    return q, kv


@pytest.mark.parametrize("B,T,H,W,lens", [(4, 1, 64, 128, [128, 100, 1, 0]), (2, 1, 64, 512, [512, 300]),
                                          (3, 1, 128, 200, [200, 129, 57]), (2, 2, 64, 64, [64, 10, 0, 33])])
def test_swa_alone_matches_oracle(csa2, B, T, H, W, lens):
    q, kv = _inputs(B * 7 + W, B, T, H, W)
    sl = torch.tensor(lens, dtype=torch.int32)
    out = torch.full((B, T, H, 512), 7.0, device=DEV)
    lse = torch.full((B, T, H), 7.0, device=DEV)
    csa2.csa2_swa_attn_fp8(q.to(DEV), kv.to(DEV), sl.to(DEV), out, 1 / 24.0, lse=lse)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.swa_attn_merge(gen.as_numpy(q).view(np.uint16), gen.as_numpy(kv), sl.numpy(), 1 / 24.0, 512)
    check_attn(out.cpu().numpy(), ref_o, "swa")
    check_lse(lse.cpu().numpy(), ref_l, "swa lse")


@pytest.mark.parametrize("in_place", [True, False])
def test_swa_merged_with_sparse_branch_matches_oracle(csa2, in_place):
    B, T, H, N, K, W = 4, 1, 64, 3000, 512, 128
    q, kv = _inputs(5, B, T, H, W)
    codes, scales = gen.fp4_planes(6, 1, B * N, 576)
    kl = torch.tensor([3000, 2500, 2000, 700], dtype=torch.int32)
    idx = torch.stack([torch.randperm(int(kl[b]), generator=torch.Generator().manual_seed(b))[:K]
                       for b in range(B)]).to(torch.int32).reshape(B, T, K)
    sl = torch.tensor([128, 64, 0, 17], dtype=torch.int32)
    o_sp = torch.empty(B, T, H, 512, device=DEV)
    l_sp = torch.empty(B, T, H, device=DEV)
    csa2.csa2_sparse_attn_fp4(0, q.to(DEV), codes.to(DEV), scales.to(DEV), N, idx.to(DEV), o_sp, 1 / 24.0,
                              kv_len=kl.to(DEV), lse=l_sp)
    out = o_sp if in_place else torch.empty_like(o_sp)
    lse = torch.empty(B, T, H, device=DEV)
    csa2.csa2_swa_attn_fp8(q.to(DEV), kv.to(DEV), sl.to(DEV), out, 1 / 24.0, o_sparse=o_sp, lse_sparse=l_sp, lse=lse)
    torch.cuda.synchronize()
    qn = gen.as_numpy(q).view(np.uint16)
    ro, rl, bad = oracle.sparse_attn(qn, gen.as_numpy(codes), gen.as_numpy(scales), N, gen.as_numpy(idx),
                                     kl.numpy(), 1 / 24.0, 512)
    assert bad == 0
    ref_o, ref_l = oracle.swa_attn_merge(qn, gen.as_numpy(kv), sl.numpy(), 1 / 24.0, 512, ro, rl)
    check_attn(out.cpu().numpy(), ref_o, "merged")
    check_lse(lse.cpu().numpy(), ref_l, "merged lse")


def test_swa_empty_window_keeps_sparse_and_empty_both_is_zero(csa2):
    B, T, H, W = 2, 1, 64, 128
    q, kv = _inputs(9, B, T, H, W)
    o_sp = torch.randn(B, T, H, 512, device=DEV)
    l_sp = torch.randn(B, T, H, device=DEV)
    l_sp[1, 0, :5] = -float("inf")
    out = torch.empty_like(o_sp)
    lse = torch.empty(B, T, H, device=DEV)
    csa2.csa2_swa_attn_fp8(q.to(DEV), kv.to(DEV), torch.zeros(B, dtype=torch.int32, device=DEV), out, 0.05,
                           o_sparse=o_sp, lse_sparse=l_sp, lse=lse)
    torch.cuda.synchronize()
    fin = torch.isfinite(l_sp)
    assert torch.allclose(out[fin], o_sp[fin], rtol=1e-6, atol=1e-6)
    assert torch.allclose(lse[fin], l_sp[fin], rtol=1e-6, atol=1e-6)
    assert (out[~fin] == 0).all() and torch.isneginf(lse[~fin]).all()
