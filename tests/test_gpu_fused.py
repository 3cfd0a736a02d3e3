"""csa2_index_topk (fused decode indexer: score -> [pool ->] Top-K, FP8) against
the oracle's unfused chain index_score -> build_pool -> topk on the same
seeded inputs.  Selections must agree outside the tie band of the oracle's
fp64 scores (the GPU selects on its fp32 scores)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gen
import oracle
from helpers import check_selection

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def csa2():
    import sparse_attention_fp4_quantize_gb300 as lib
    return lib


def _ref_scores(mode, q, w, k, kl, pool=None):
    return oracle.index_score(mode, gen.as_numpy(q), oracle.FP8_E4M3, gen.as_numpy(w), gen.as_numpy(k),
                              oracle.FP8_E4M3, gen.as_numpy(kl), pool=None if pool is None else gen.as_numpy(pool))


def _block_max(ref, kl, G=8):
    """fp64 block maxima over each row's valid positions (-inf where none)."""
    B, T, N = ref.shape
    nb = (N + G - 1) // G
    out = np.full((B, T, nb), -np.inf)
    for b in range(B):
        for t in range(T):
            n = min(int(kl[b * T + t]), N)
            r = ref[b, t, :n]
            pad = np.full(nb * G - n, -np.inf)
            out[b, t] = np.concatenate([r, pad]).reshape(nb, G).max(1)
    return out


def _fused(csa2, mode, q, w, k, kl, K, pool=None, P_out=0, flag=None):
    B, T = q.shape[0], q.shape[1]
    idx = torch.full((B, T, K), -99, dtype=torch.int32, device=DEV)
    pool_out = torch.full((B, T, P_out), -99, dtype=torch.int32, device=DEV) if P_out else None
    csa2.csa2_index_topk(mode, q.to(DEV), w.to(DEV), k.to(DEV), kl.to(DEV), idx,
                         pool_blocks=None if pool is None else pool.to(DEV), pool_out=pool_out, err_flag=flag)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), (pool_out.cpu().numpy() if P_out else None)


def _check_rows(got, want, ref_of_row, K, what):
    B, T, _ = got.shape
    for b in range(B):
        for t in range(T):
            check_selection(got[b, t], want[b, t], lambda ids: ref_of_row(b, t)[ids], K, what)


@pytest.mark.parametrize("B,T,N,K,P_out", [(2, 1, 3000, 512, 256), (3, 1, 1000, 64, 0), (1, 3, 5000, 512, 2048),
                                           (4, 1, 777, 512, 64), (2, 1, 130, 16, 8)])
def test_fused_full_matches_oracle_chain(csa2, B, T, N, K, P_out):
    q = gen.normal_e4m3(21, 1, (B, T, 4, 64))
    k = gen.normal_e4m3(21, 2, (B, N, 64))
    w = gen.uniform01(21, 3, (B, T, 4))
    kl = torch.tensor([max(1, (N * (i + 2)) // (B * T + 1)) for i in range(B * T)], dtype=torch.int32)
    kl[0] = N
    ref = _ref_scores(0, q, w, k, kl)
    s32 = ref.astype(np.float32)
    got_idx, got_pool = _fused(csa2, 0, q, w, k, kl, K, P_out=P_out)
    want_idx = oracle.topk(oracle.FULL, s32, gen.as_numpy(kl), K=K)
    _check_rows(got_idx, want_idx, lambda b, t: ref[b, t], K, "fused topk")
    if P_out:
        want_pool = oracle.build_pool(s32, gen.as_numpy(kl), P=P_out)
        bm = _block_max(ref, gen.as_numpy(kl))
        _check_rows(got_pool, want_pool, lambda b, t: bm[b, t], P_out, "fused pool")


def test_fused_full_short_and_empty_rows(csa2):
    """Rows with no visible entry (all -1), fewer visible entries than K or
    than the pool's blocks, a partial last block, and kv_len beyond N
    (clamped), with the pool written."""
    B, T, N, K, P_out = 1, 8, 4000, 512, 2048
    q = gen.normal_e4m3(23, 1, (B, T, 4, 64))
    k = gen.normal_e4m3(23, 2, (B, N, 64))
    w = gen.uniform01(23, 3, (B, T, 4))
    kl = torch.tensor([0, 1, 7, 9, 511, 513, 4000, 10 ** 6], dtype=torch.int32)
    ref = _ref_scores(0, q, w, k, kl)
    s32 = ref.astype(np.float32)
    got_idx, got_pool = _fused(csa2, 0, q, w, k, kl, K, P_out=P_out)
    want_idx = oracle.topk(oracle.FULL, s32, gen.as_numpy(kl), K=K)
    _check_rows(got_idx, want_idx, lambda b, t: ref[b, t], K, "fused topk (short rows)")
    want_pool = oracle.build_pool(s32, gen.as_numpy(kl), P=P_out)
    bm = _block_max(ref, gen.as_numpy(kl))
    _check_rows(got_pool, want_pool, lambda b, t: bm[b, t], P_out, "fused pool (short rows)")
    assert (got_idx[0, 0] == -1).all() and (got_pool[0, 0] == -1).all()
    assert sorted(got_idx[0, 2][got_idx[0, 2] >= 0].tolist()) == list(range(7))


def test_fused_full_batched_decode_full_size(csa2):
    """B=32 sequences x n_b in [8192,16384] entries, Top-512 and the 2048-block pool."""
    w = gen.FULL_BATCHED_DECODE
    q, wt, k = gen.indexer_inputs(w)
    kl = gen.kv_lengths(w)
    ref = _ref_scores(0, q, wt, k, kl)
    s32 = ref.astype(np.float32)
    got_idx, got_pool = _fused(csa2, 0, q, wt, k, kl, 512, P_out=2048)
    _check_rows(got_idx, oracle.topk(oracle.FULL, s32, gen.as_numpy(kl), K=512), lambda b, t: ref[b, t], 512,
                "fused topk")
    bm = _block_max(ref, gen.as_numpy(kl))
    _check_rows(got_pool, oracle.build_pool(s32, gen.as_numpy(kl), P=2048), lambda b, t: bm[b, t], 2048,
                "fused pool")


def test_fused_reindex_matches_oracle_chain_and_flags_bad_pool(csa2):
    B, N, P, K = 3, 20000, 512, 512
    q = gen.normal_e4m3(22, 1, (B, 1, 4, 64))
    k = gen.normal_e4m3(22, 2, (B, N, 64))
    w = gen.uniform01(22, 3, (B, 1, 4))
    kl = torch.tensor([20000, 15001, 9000], dtype=torch.int32)
    g = torch.Generator().manual_seed(5)
    pool = torch.stack([torch.randperm((N + 7) // 8, generator=g)[:P] for _ in range(B)]).to(torch.int32)
    pool = pool.reshape(B, 1, P)
    pool[0, 0, :40] = -1
    ref = _ref_scores(1, q, w, k, kl, pool)
    want = oracle.topk(oracle.REINDEX, ref.astype(np.float32), None, pool=gen.as_numpy(pool), K=K)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    got, _ = _fused(csa2, 1, q, w, k, kl, K, pool=pool, flag=flag)
    assert int(flag.item()) == 0
    pos_score = [{int(8 * pool[b, 0, p] + i): ref[b, 0, 8 * p + i] for p in range(P) for i in range(8)
                  if pool[b, 0, p] >= 0} for b in range(B)]
    for b in range(B):
        check_selection(got[b, 0], want[b, 0], lambda ids: np.array([pos_score[b][int(j)] for j in ids]), K,
                        "fused reindex")
    bad = pool.clone()
    bad[1, 0, 3] = (N + 7) // 8
    got_bad, _ = _fused(csa2, 1, q, w, k, kl, K, pool=bad, flag=flag)
    assert int(flag.item()) & csa2.FLAG_BAD_POOL
    assert all(j < 0 or j < N for j in got_bad[1, 0])


def test_fused_long_rows_use_wider_clusters(csa2):
    """1M-token context (262144 entries per row): rows span a cluster of 8 CTAs."""
    B, N, K = 2, 262144, 512
    q = gen.normal_e4m3(23, 1, (B, 1, 4, 64))
    k = gen.normal_e4m3(23, 2, (B, N, 64))
    w = gen.uniform01(23, 3, (B, 1, 4))
    kl = torch.tensor([N, 200001], dtype=torch.int32)
    ref = _ref_scores(0, q, w, k, kl)
    s32 = ref.astype(np.float32)
    got_idx, got_pool = _fused(csa2, 0, q, w, k, kl, K, P_out=2048)
    _check_rows(got_idx, oracle.topk(oracle.FULL, s32, gen.as_numpy(kl), K=K), lambda b, t: ref[b, t], K,
                "fused topk")
    bm = _block_max(ref, gen.as_numpy(kl))
    _check_rows(got_pool, oracle.build_pool(s32, gen.as_numpy(kl), P=2048), lambda b, t: bm[b, t], 2048,
                "fused pool")


def test_fused_equals_unfused_gpu_chain(csa2):
    """Same scores on both paths: the fused selection is the unfused one, id for id (as sets)."""
    w = gen.scaled(gen.FULL_BATCHED_DECODE, B=8)
    q, wt, k = gen.indexer_inputs(w)
    kl = gen.kv_lengths(w)
    scores = torch.empty(w.B, 1, w.N, device=DEV)
    csa2.csa2_index_score(0, q.to(DEV), wt.to(DEV), k.to(DEV), kl.to(DEV), scores)
    idx_u = torch.empty(w.B, 1, 512, dtype=torch.int32, device=DEV)
    pool_u = torch.empty(w.B, 1, 2048, dtype=torch.int32, device=DEV)
    csa2.csa2_topk(0, scores, idx_u, kv_len=kl.to(DEV))
    csa2.csa2_build_pool(scores, kl.to(DEV), pool_u)
    got_idx, got_pool = _fused(csa2, 0, q, wt, k, kl, 512, P_out=2048)
    for b in range(w.B):
        assert sorted(got_idx[b, 0].tolist()) == sorted(idx_u[b, 0].cpu().tolist())
        assert sorted(got_pool[b, 0].tolist()) == sorted(pool_u[b, 0].cpu().tolist())


def test_fused_rejects_bf16_and_reuse_is_noop(csa2):
    q = torch.zeros(1, 1, 4, 64, dtype=torch.int16, device=DEV)
    k = torch.zeros(1, 100, 64, dtype=torch.int16, device=DEV)
    w = torch.ones(1, 1, 4, device=DEV)
    kl = torch.tensor([100], dtype=torch.int32, device=DEV)
    idx = torch.full((1, 1, 16), 7, dtype=torch.int32, device=DEV)
    with pytest.raises(csa2.Csa2Error):
        csa2.csa2_index_topk(0, q, w, k, kl, idx)
    q8 = torch.zeros(1, 1, 4, 64, dtype=torch.uint8, device=DEV)
    k8 = torch.zeros(1, 100, 64, dtype=torch.uint8, device=DEV)
    csa2.csa2_index_topk(2, q8, w, k8, kl, idx)
    torch.cuda.synchronize()
    assert (idx == 7).all()
