"""The counting argument behind csa2_index_topk_dense, checked on the CPU.

For each row, split the visible positions into aligned blocks of 8 and let
tau be the K-th largest block maximum (no threshold when fewer than K blocks
exist).  Then (i) at least K scores are >= tau, (ii) at most 8(K-1) scores are
> tau, and (iii) the oracle's Top-K equals every score > tau plus the lowest
positions among those equal to tau.  Rows come from the oracle's indexer
scores and from adversarial value sets (many ties, one hot block, sorted
runs)."""
from __future__ import annotations

import numpy as np
import pytest

import gen
import oracle


def _tau(row, K):
    n = row.size
    nb = (n + 7) // 8
    if nb < K:
        return -np.inf
    pad = np.full(nb * 8 - n, -np.inf)
    bm = np.concatenate([row, pad]).reshape(nb, 8).max(1)
    return np.sort(bm)[::-1][K - 1]


def _check(row, K):
    tau = _tau(row, K)
    n_ge = int((row >= tau).sum())
    n_gt = int((row > tau).sum())
    assert n_ge >= min(K, row.size)
    assert n_gt <= 8 * (K - 1)
    # (iii): the oracle's selection is reproduced from the two candidate sets
    want = oracle.topk(oracle.FULL, row.astype(np.float32)[None, None, :], None, K=K)[0, 0]
    want = sorted(int(j) for j in want if j >= 0)
    gt = np.nonzero(row > tau)[0]
    eq = np.nonzero(row == tau)[0]
    if gt.size >= K:
        got = np.argsort(-row[gt], kind="stable")[:K]
        got = gt[got]
    else:
        got = np.concatenate([gt, eq[: K - gt.size]])
    assert sorted(got.tolist()) == want


@pytest.mark.parametrize("K", [1, 16, 512])
def test_bound_on_indexer_scores(K):
    B, T, N = 1, 6, 6000
    q = gen.normal_e4m3(41, 1, (B, T, 4, 64))
    k = gen.normal_e4m3(41, 2, (B, N, 64))
    w = gen.uniform01(41, 3, (B, T, 4))
    kl = np.array([6000, 5999, 4097, 4096, 300, 9], np.int32)
    s = oracle.index_score(0, gen.as_numpy(q), oracle.FP8_E4M3, gen.as_numpy(w), gen.as_numpy(k),
                           oracle.FP8_E4M3, kl)
    for t in range(T):
        row = s[0, t, : kl[t]].astype(np.float32).astype(np.float64)
        _check(row, K)


def test_bound_on_adversarial_rows():
    rng = np.random.default_rng(7)
    K = 64
    rows = [
        np.zeros(3000),                                    # all ties
        np.repeat(rng.integers(0, 5, 400), 8).astype(float),  # whole blocks equal, few values
        np.sort(rng.standard_normal(2000)),               # ascending: the top sits in the last blocks
        np.sort(rng.standard_normal(2000))[::-1].copy(),   # descending
        np.where(np.arange(4000) < 8, 100.0, rng.standard_normal(4000)),   # one hot block
        rng.integers(0, 3, 5000).astype(float),            # three values, ties everywhere
    ]
    for row in rows:
        _check(row, K)
