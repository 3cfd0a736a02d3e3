"""csa2_index_topk_dense (fused indexer for many query tokens: block maxima ->
the K best blocks -> their 8K candidates rescored -> Top-K, FP8) against the oracle's unfused
chain index_score -> topk on the same seeded inputs.  Selections must agree
outside the tie band of the oracle's fp64 scores (the GPU selects on its
fp32 scores)."""
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


def _ref_scores(q, w, k, kl):
    return oracle.index_score(0, gen.as_numpy(q), oracle.FP8_E4M3, gen.as_numpy(w), gen.as_numpy(k),
                              oracle.FP8_E4M3, gen.as_numpy(kl))


def _dense(csa2, q, w, k, kl, K):
    B, T = q.shape[0], q.shape[1]
    idx = torch.full((B, T, K), -99, dtype=torch.int32, device=DEV)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    csa2.csa2_index_topk_dense(q.to(DEV), w.to(DEV), k.to(DEV), kl.to(DEV), idx, err_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    return idx.cpu().numpy()


def _check_rows(got, want, ref, K, what):
    B, T, _ = got.shape
    for b in range(B):
        for t in range(T):
            check_selection(got[b, t], want[b, t], lambda ids: ref[b, t][ids], K, what)


def _causal_lengths(T, N, first_pos):
    """Entry j covers tokens [4j, 4j+4): the query at token p sees j < (p+1)//4."""
    return torch.tensor([min(N, (first_pos + t + 1) // 4) for t in range(T)], dtype=torch.int32)


@pytest.mark.parametrize("B,T,N,K,first_pos", [(1, 100, 3000, 512, 11000), (2, 64, 777, 64, 3000),
                                               (1, 130, 5000, 2048, 12000), (1, 70, 20000, 1, 79000),
                                               (3, 65, 1029, 16, 2500)])
def test_dense_matches_oracle_chain(csa2, B, T, N, K, first_pos):
    q = gen.normal_e4m3(31, 1, (B, T, 4, 64))
    k = gen.normal_e4m3(31, 2, (B, N, 64))
    w = gen.uniform01(31, 3, (B, T, 4))
    kl = _causal_lengths(T, N, first_pos).repeat(B)
    ref = _ref_scores(q, w, k, kl)
    want = oracle.topk(oracle.FULL, ref.astype(np.float32), gen.as_numpy(kl), K=K)
    got = _dense(csa2, q, w, k, kl, K)
    _check_rows(got, want, ref, K, "dense topk")


def test_dense_long_context_and_single_query_rows(csa2):
    """1M-token context (262144 entries: the block maxima of a row take 128 KB
    of shared memory) with 16 queries, and B=3 sequences of one query each."""
    q = gen.normal_e4m3(34, 1, (1, 16, 4, 64))
    k = gen.normal_e4m3(34, 2, (1, 262144, 64))
    w = gen.uniform01(34, 3, (1, 16, 4))
    kl = _causal_lengths(16, 262144, 1048576 - 16)
    ref = _ref_scores(q, w, k, kl)
    want = oracle.topk(oracle.FULL, ref.astype(np.float32), gen.as_numpy(kl), K=512)
    _check_rows(_dense(csa2, q, w, k, kl, 512), want, ref, 512, "dense topk (1M context)")
    q1 = gen.normal_e4m3(35, 1, (3, 1, 4, 64))
    k1 = gen.normal_e4m3(35, 2, (3, 9000, 64))
    w1 = gen.uniform01(35, 3, (3, 1, 4))
    kl1 = torch.tensor([9000, 4321, 600], dtype=torch.int32)
    ref1 = _ref_scores(q1, w1, k1, kl1)
    want1 = oracle.topk(oracle.FULL, ref1.astype(np.float32), gen.as_numpy(kl1), K=512)
    _check_rows(_dense(csa2, q1, w1, k1, kl1, 512), want1, ref1, 512, "dense topk (T=1)")


def test_dense_short_and_empty_rows(csa2):
    """Rows with no visible entry (all -1), fewer than K visible entries (all
    of them, then -1), fewer than K blocks but more than K entries, and
    kv_len beyond N (clamped)."""
    B, T, N, K = 1, 64, 4000, 512
    q = gen.normal_e4m3(32, 1, (B, T, 4, 64))
    k = gen.normal_e4m3(32, 2, (B, N, 64))
    w = gen.uniform01(32, 3, (B, T, 4))
    lens = [0, 1, 7, 8, 9, 300, 511, 512, 513, 1000, 4095, 4096, 5000, 10 ** 6] + [(37 * t) % 4100 for t in range(50)]
    kl = torch.tensor(lens[:T], dtype=torch.int32)
    ref = _ref_scores(q, w, k, kl)
    want = oracle.topk(oracle.FULL, ref.astype(np.float32), gen.as_numpy(kl), K=K)
    got = _dense(csa2, q, w, k, kl, K)
    _check_rows(got, want, ref, K, "dense topk (short rows)")
    assert (got[0, 0] == -1).all()
    assert sorted(got[0, 2][got[0, 2] >= 0].tolist()) == list(range(7))


@pytest.mark.parametrize("first_pos", [16000, 40000])
def test_dense_all_ties(csa2, first_pos):
    """w = 0 makes every visible score 0.  Ties go to the lowest positions, as
    in the oracle's Top-K, so each row takes positions 0 .. K-1 (every visible
    one when there are fewer): with about 500 blocks per row every block is a
    candidate; with 625 blocks the K tied block maxima are the lowest K blocks."""
    B, T, N, K = 1, 64, 5000, 512
    q = gen.normal_e4m3(33, 1, (B, T, 4, 64))
    k = gen.normal_e4m3(33, 2, (B, N, 64))
    w = torch.zeros(B, T, 4)
    kl = _causal_lengths(T, N, first_pos).repeat(B)
    got = _dense(csa2, q, w, k, kl, K)
    for t in range(T):
        ids = got[0, t]
        n = min(K, int(kl[t]))
        sel = ids[ids >= 0]
        assert sorted(sel.tolist()) == list(range(n))
        assert (ids[n:] == -1).all()


def test_dense_prefill_chunk_full_size(csa2):
    """4096 causal queries x 32768 entries, Top-512: id-for-id against the
    unfused GPU chain (same fp32 scores), and 24 sampled queries against the
    oracle."""
    w4 = gen.PREFILL_CHUNK
    q, wt, k = gen.indexer_inputs(w4, device=DEV)
    kl = gen.kv_lengths(w4).to(DEV)
    T, N = w4.T, w4.N
    idx = torch.empty(1, T, 512, dtype=torch.int32, device=DEV)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    csa2.csa2_index_topk_dense(q, wt, k, kl, idx, err_flag=flag)
    scores = torch.empty(1, T, N, device=DEV)
    csa2.csa2_index_score(0, q, wt, k, kl, scores)
    idx_u = torch.empty(1, T, 512, dtype=torch.int32, device=DEV)
    csa2.csa2_topk(0, scores, idx_u, kv_len=kl)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    a = torch.sort(idx[0], dim=1).values
    b = torch.sort(idx_u[0], dim=1).values
    same = (a == b).all(1)
    # rows that differ may only differ at the 512th fp32 score (the rescoring
    # may round a score differently in the last bits)
    for t in torch.nonzero(~same).flatten().tolist():
        s = scores[0, t]
        kth = float(torch.topk(s, 512).values[-1])
        d = set(idx[0, t].tolist()) ^ set(idx_u[0, t].tolist())
        assert all(abs(float(s[j]) - kth) <= 1e-5 * abs(kth) for j in d), "row %d differs off the tie" % t
    rows = torch.linspace(0, T - 1, 24).long()
    qs, ws, kls = q[:, rows].cpu(), wt[:, rows].cpu(), kl[rows].cpu()
    ref = _ref_scores(qs, ws, k.cpu(), kls)
    want = oracle.topk(oracle.FULL, ref.astype(np.float32), gen.as_numpy(kls), K=512)
    got = idx[:, rows].cpu().numpy()
    _check_rows(got, want, ref, 512, "dense topk (prefill sample)")


def test_dense_rejects_bad_arguments(csa2):
    q = torch.zeros(1, 64, 4, 64, dtype=torch.uint8, device=DEV)
    k = torch.zeros(1, 100, 64, dtype=torch.uint8, device=DEV)
    w = torch.ones(1, 64, 4, device=DEV)
    kl = torch.full((64,), 100, dtype=torch.int32, device=DEV)
    idx = torch.empty(1, 64, 16, dtype=torch.int32, device=DEV)
    small = torch.empty(64, dtype=torch.uint8, device=DEV)
    with pytest.raises(csa2.Csa2Error) as e:
        csa2.csa2_index_topk_dense(q, w, k, kl, idx, workspace=small)
    assert e.value.status == 3   # CSA2_ERR_WORKSPACE
    with pytest.raises(csa2.Csa2Error):
        csa2.csa2_index_topk_dense(q.view(torch.int16)[..., :32].contiguous(), w, k, kl, idx)   # bf16
    big = torch.zeros(1, 262145, 64, dtype=torch.uint8, device=DEV)
    with pytest.raises(csa2.Csa2Error) as e:
        csa2.csa2_index_topk_dense(q, w, big, kl, idx)
    assert e.value.status == 2   # CSA2_ERR_UNSUPPORTED
