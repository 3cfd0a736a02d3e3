"""Pins of the oracle's indexer, pool, Top-K and attention (CPU only).

Special cases with closed forms, library routines (torch fp64 einsum,
softmax, topk) and brute-force sorts on tiny inputs; invariants that follow
from the mode definitions (Reindex selects only inside the pool, Reindex
with the Full layer's own query reproduces the Full selection, Reuse leaves
the source's indices untouched).
"""
import math

import numpy as np
import pytest
import torch

import gen

FULL, REINDEX, REUSE = 0, 1, 2
BF16, FP8 = 0, 1


def _bf16(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bf16_val(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


def _e4m3_val(b):
    return torch.from_numpy(np.ascontiguousarray(b)).view(torch.float8_e4m3fn).double().numpy()


# ------------------------------------------------------------ index score
def test_index_score_one_hot_gives_relu_of_key(orc):
    B, N = 2, 40
    k = gen.normal_bf16(1, 1, (B, N, 64)).numpy().view(np.uint16)
    kv = _bf16_val(k)
    for h, d in [(0, 0), (3, 63), (2, 17)]:
        q = np.zeros((B, 1, 4, 64), np.float32)
        q[:, :, h, d] = 1.0
        w = np.zeros((B, 1, 4), np.float32)
        w[:, :, h] = 1.0
        s = orc.index_score(FULL, _bf16(q), BF16, w, k, BF16, np.full(B, N, np.int32))
        assert (s[:, 0, :] == np.maximum(kv[:, :, d], 0)).all()


def test_index_score_zero_query_and_mask(orc):
    B, N = 2, 33
    k = gen.normal_e4m3(2, 1, (B, N, 64)).numpy()
    q = np.zeros((B, 1, 4, 64), np.uint8)
    w = np.ones((B, 1, 4), np.float32)
    kl = np.array([33, 5], np.int32)
    s = orc.index_score(FULL, q, FP8, w, k, FP8, kl)
    assert (s[0, 0] == 0).all()
    assert (s[1, 0, :5] == 0).all() and np.isneginf(s[1, 0, 5:]).all()


@pytest.mark.parametrize("dt", [BF16, FP8])
def test_index_score_matches_torch_einsum(orc, dt):
    B, T, N = 3, 2, 100
    if dt == BF16:
        q = gen.normal_bf16(3, 1, (B, T, 4, 64)).numpy().view(np.uint16)
        k = gen.normal_bf16(3, 2, (B, N, 64)).numpy().view(np.uint16)
        qv, kv = _bf16_val(q), _bf16_val(k)
    else:
        q = gen.normal_e4m3(3, 1, (B, T, 4, 64)).numpy()
        k = gen.normal_e4m3(3, 2, (B, N, 64)).numpy()
        qv, kv = _e4m3_val(q), _e4m3_val(k)
    w = gen.uniform01(3, 3, (B, T, 4)).numpy()
    kl = np.array([100, 64, 99, 1, 50, 100], np.int32)
    s, mag = orc.index_score(FULL, q, dt, w, k, dt, kl, with_mag=True)
    dots = torch.einsum("bthd,bnd->bthn", torch.from_numpy(qv), torch.from_numpy(kv))
    ref = (torch.from_numpy(w.astype(np.float64))[..., None] * dots.clamp(min=0)).sum(2).numpy()
    amag = (torch.from_numpy(w.astype(np.float64))[..., None] *
            torch.einsum("bthd,bnd->bthn", torch.from_numpy(np.abs(qv)), torch.from_numpy(np.abs(kv)))).sum(2).numpy()
    mask = np.arange(N)[None, None, :] < kl.reshape(B, T)[..., None]
    assert np.allclose(s[mask], ref[mask], rtol=1e-12, atol=1e-12)
    assert np.isneginf(s[~mask]).all()
    assert np.allclose(mag[mask], amag[mask], rtol=1e-12)


def test_index_score_reindex_is_full_at_pool_positions(orc):
    B, N, P = 2, 200, 6
    q = gen.normal_e4m3(4, 1, (B, 1, 4, 64)).numpy()
    k = gen.normal_e4m3(4, 2, (B, N, 64)).numpy()
    w = gen.uniform01(4, 3, (B, 1, 4)).numpy()
    kl = np.array([200, 61], np.int32)
    full = orc.index_score(FULL, q, FP8, w, k, FP8, kl)
    pool = np.array([[[3, 0, 24, -1, 7, 1]], [[7, 0, -1, -1, 2, 5]]], np.int32)
    re = orc.index_score(REINDEX, q, FP8, w, k, FP8, kl, pool=pool)
    assert re.shape == (B, 1, 8 * P)
    for b in range(B):
        for p in range(P):
            for i in range(8):
                blk = pool[b, 0, p]
                j = 8 * blk + i
                v = re[b, 0, 8 * p + i]
                if blk < 0 or j >= kl[b]:
                    assert np.isneginf(v)
                else:
                    assert v == full[b, 0, j]


# ------------------------------------------------------------ top-k
def _brute_topk(v, K):
    cand = [(x, i) for i, x in enumerate(v) if x > -math.inf]
    cand = sorted(cand, key=lambda t: (-t[0], t[1]))[:K]
    return [i for _, i in cand] + [-1] * (K - len(cand))


def test_topk_brute_force_tiny(orc):
    rng = np.random.default_rng(8)
    for trial in range(200):
        n = int(rng.integers(1, 65))
        K = int(rng.integers(1, 17))
        kind = trial % 4
        if kind == 0:
            v = rng.standard_normal(n)
        elif kind == 1:
            v = rng.integers(0, 3, n).astype(np.float64)            # heavy ties
        elif kind == 2:
            v = np.zeros(n)                                          # all ties
        else:
            v = rng.standard_normal(n)
            v[rng.random(n) < 0.7] = -np.inf                         # < K valid
        v32 = v.astype(np.float32)
        kl = np.array([n], np.int32)
        got = orc.topk(FULL, v32.reshape(1, 1, n), kl, K=K)[0, 0]
        assert list(got) == _brute_topk(list(v32.astype(np.float64)), K)


def test_topk_respects_kv_len_and_matches_torch(orc):
    s = gen.uniform01(9, 1, (4, 1, 3000)).numpy()
    kl = np.array([3000, 2999, 600, 512], np.int32)
    got = orc.topk(FULL, s, kl, K=512)
    for b in range(4):
        ref = torch.topk(torch.from_numpy(s[b, 0, :kl[b]]), 512).indices.numpy()
        assert set(got[b, 0]) == set(ref)
    assert (got[3, 0] >= 0).all()


def test_topk_reuse_is_noop(orc):
    s = gen.uniform01(9, 2, (1, 1, 100)).numpy()
    idx = orc.topk(REUSE, s, None, K=16)
    assert (idx == -7).all()       # the sentinel the wrapper pre-fills: untouched


# ------------------------------------------------------------ pool
def test_pool_brute_force(orc):
    rng = np.random.default_rng(10)
    for trial in range(50):
        N = int(rng.integers(1, 200))
        P = int(rng.integers(1, 12))
        s = rng.standard_normal((1, 1, N)).astype(np.float32)
        if trial % 3 == 0:
            s = np.round(s).astype(np.float32)                          # ties
        kl = np.array([int(rng.integers(0, N + 1))], np.int32)
        got = orc.build_pool(s, kl, P=P)[0, 0]
        nb = (N + 7) // 8
        bs = []
        for beta in range(nb):
            vals = [float(s[0, 0, j]) for j in range(8 * beta, min(8 * beta + 8, int(kl[0])))]
            bs.append(max(vals) if vals else -math.inf)
        assert list(got) == _brute_topk(bs, P)


def test_pool_invariants_and_coverage(orc):
    N = 16384
    s = gen.uniform01(11, 1, (2, 1, N)).numpy()
    kl = np.array([16384, 9001], np.int32)
    pool = orc.build_pool(s, kl, P=2048)
    for b in range(2):
        blocks = pool[b, 0]
        valid = blocks[blocks >= 0]
        assert len(valid) * 8 <= 16384
        # n <= 16384 entries -> the pool covers every valid entry
        assert set(valid) == set(range((kl[b] + 7) // 8))
    # a long row: chosen block maxima dominate unchosen ones
    N2 = 64 * 1024
    s2 = gen.uniform01(11, 2, (1, 1, N2)).numpy()
    pool2 = orc.build_pool(s2, np.array([N2], np.int32), P=2048)[0, 0]
    bmax = s2[0, 0].reshape(-1, 8).max(1)
    chosen = np.zeros(len(bmax), bool)
    chosen[pool2] = True
    assert chosen.sum() == 2048
    assert bmax[chosen].min() >= bmax[~chosen].max()


# ------------------------------------------------------------ Reindex invariants
def test_reindex_same_query_reproduces_full_topk(orc):
    """With the Reindex layer's q, w equal to the Full layer's and the pool
    built from those scores, Reindex Top-512 equals Full Top-512: a block
    holding a top-512 entry has block max >= the 512th score, there are at
    most 512 such blocks, and 512 <= 2048."""
    B, N = 2, 40000
    q = gen.normal_e4m3(12, 1, (B, 1, 4, 64)).numpy()
    k = gen.normal_e4m3(12, 2, (B, N, 64)).numpy()
    w = gen.uniform01(12, 3, (B, 1, 4)).numpy()
    kl = np.array([40000, 31000], np.int32)
    full = orc.index_score(FULL, q, FP8, w, k, FP8, kl).astype(np.float32)
    pool = orc.build_pool(full, kl, P=2048)
    top_full = orc.topk(FULL, full, kl, K=512)
    re = orc.index_score(REINDEX, q, FP8, w, k, FP8, kl, pool=pool).astype(np.float32)
    top_re = orc.topk(REINDEX, re, kl, pool=pool, K=512)
    for b in range(B):
        assert set(top_re[b, 0]) == set(top_full[b, 0])
        in_pool = set()
        for blk in pool[b, 0]:
            if blk >= 0:
                in_pool.update(range(8 * blk, 8 * blk + 8))
        assert set(top_re[b, 0]) <= in_pool


def test_reindex_new_query_selects_inside_pool(orc):
    B, N = 1, 30000
    q1 = gen.normal_e4m3(13, 1, (B, 1, 4, 64)).numpy()
    q2 = gen.normal_e4m3(13, 4, (B, 1, 4, 64)).numpy()
    k = gen.normal_e4m3(13, 2, (B, N, 64)).numpy()
    w1 = gen.uniform01(13, 3, (B, 1, 4)).numpy()
    w2 = gen.uniform01(13, 5, (B, 1, 4)).numpy()
    kl = np.array([N], np.int32)
    full = orc.index_score(FULL, q1, FP8, w1, k, FP8, kl).astype(np.float32)
    pool = orc.build_pool(full, kl, P=2048)
    re = orc.index_score(REINDEX, q2, FP8, w2, k, FP8, kl, pool=pool).astype(np.float32)
    top_re = orc.topk(REINDEX, re, kl, pool=pool, K=512)
    blocks = set(pool[0, 0][pool[0, 0] >= 0])
    assert all(j // 8 in blocks for j in top_re[0, 0])
    assert len(set(top_re[0, 0])) == 512


# ------------------------------------------------------------ attention
def _kv(orc, seed, R, D):
    bits = gen.kv_rows(seed, 1, R, D, rms=True).numpy().view(np.uint16)
    return orc.quantize_kv_fp4(bits)


def test_attn_single_index_returns_value_row(orc):
    D, dv, N = 128, 64, 50
    codes, scales = _kv(orc, 14, N, D)
    vhat = orc.dequant_fp4(codes, scales)
    q = gen.normal_bf16(14, 2, (1, 1, 4, D)).numpy().view(np.uint16)
    idx = np.full((1, 1, 8), -1, np.int32)
    idx[0, 0, 5] = 17
    out, lse, bad = orc.sparse_attn(q, codes, scales, N, idx, np.array([N], np.int32), 0.1, dv)
    assert bad == 0
    for h in range(4):
        assert (out[0, 0, h] == vhat[17, :dv]).all()
        z = 0.1 * (_bf16_val(q[0, 0, h]) * vhat[17]).sum()
        assert abs(lse[0, 0, h] - z) <= 1e-12 * max(1, abs(z))


def test_attn_zero_query_is_mean_of_values(orc):
    D, dv, N = 576, 512, 300
    codes, scales = _kv(orc, 15, N, D)
    vhat = orc.dequant_fp4(codes, scales)
    q = np.zeros((1, 1, 2, D), np.uint16)
    sel = np.array([3, 99, 250, 7, 0, 299], np.int32)
    idx = np.concatenate([sel, [-1, -1]]).astype(np.int32).reshape(1, 1, 8)
    out, lse, _ = orc.sparse_attn(q, codes, scales, N, idx, np.array([N], np.int32), 0.05, dv)
    assert np.allclose(out[0, 0, 0], vhat[sel, :dv].mean(0), rtol=1e-12, atol=1e-14)
    assert abs(lse[0, 0, 1] - math.log(6)) < 1e-12


def test_attn_select_all_is_dense_softmax_attention(orc):
    D, dv, N, H = 128, 64, 40, 3
    codes, scales = _kv(orc, 16, 2 * N, D)
    q = gen.normal_bf16(16, 2, (2, 1, H, D)).numpy().view(np.uint16)
    idx = np.stack([np.random.default_rng(b).permutation(N) for b in range(2)]).astype(np.int32).reshape(2, 1, N)
    sm = 1 / math.sqrt(D)
    out, lse, _ = orc.sparse_attn(q, codes, scales, N, idx, np.array([N, N], np.int32), sm, dv)
    kh = torch.from_numpy(orc.dequant_fp4(codes, scales)).reshape(2, N, D)
    qt = torch.from_numpy(_bf16_val(q))[:, 0]                            # [2, H, D]
    z = sm * torch.einsum("bhd,bnd->bhn", qt, kh)
    ref = torch.einsum("bhn,bnc->bhc", torch.softmax(z, -1), kh[..., :dv])
    assert np.allclose(out[:, 0], ref.numpy(), rtol=1e-10, atol=1e-12)
    assert np.allclose(lse[:, 0], torch.logsumexp(z, -1).numpy(), rtol=1e-12)


def test_attn_empty_and_bad_indices(orc):
    D, dv, N = 128, 64, 20
    codes, scales = _kv(orc, 17, N, D)
    q = gen.normal_bf16(17, 2, (1, 2, 2, D)).numpy().view(np.uint16)
    idx = np.array([[[-1, -1, -1, -1], [3, 25, -5, 19]]], np.int32)
    out, lse, bad = orc.sparse_attn(q, codes, scales, N, idx, np.array([20, 20], np.int32), 0.1, dv)
    assert (out[0, 0] == 0).all() and np.isneginf(lse[0, 0]).all()
    assert bad == 2                                                      # 25 >= kv_len and -5
    ref, _, _ = orc.sparse_attn(q[:, 1:], codes, scales, N, np.array([[[3, 19]]], np.int32),
                                np.array([20], np.int32), 0.1, dv)
    assert np.allclose(out[0, 1], ref[0, 0], rtol=1e-13)


def test_reuse_layer_consumes_source_indices_unchanged(orc):
    """A Reuse layer runs no indexer and no selection: its attention uses the
    source layer's index buffer as is."""
    D, dv, N = 128, 64, 300
    codes, scales = _kv(orc, 18, N, D)
    s = gen.uniform01(18, 1, (1, 1, N)).numpy()
    idx_src = orc.topk(FULL, s, np.array([N], np.int32), K=64)
    idx_copy = idx_src.copy()
    s_reuse = gen.uniform01(18, 2, (1, 1, N)).numpy()
    _ = orc.topk(REUSE, s_reuse, None, K=64)
    assert (idx_src == idx_copy).all()
    q_layer = gen.normal_bf16(18, 3, (1, 1, 2, D)).numpy().view(np.uint16)
    a, _, _ = orc.sparse_attn(q_layer, codes, scales, N, idx_src, np.array([N], np.int32), 0.1, dv)
    b, _, _ = orc.sparse_attn(q_layer, codes, scales, N, idx_copy, np.array([N], np.int32), 0.1, dv)
    assert (a == b).all()
