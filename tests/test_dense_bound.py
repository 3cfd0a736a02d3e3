"""The argument behind csa2_index_topk_dense, checked on the CPU.

For each row, split the visible positions into aligned blocks of 8 and let
tau be the K-th largest block maximum.  Take the K blocks whose maximum is
largest (ties at tau broken by block id here; the kernel breaks them in any
order).  Then (i) at least K scores are >= tau, (ii) every score outside the
K blocks is <= tau, and (iii) the Top-K of the scores inside them equals the
oracle's Top-K up to ties at the K-th value.  Rows come from the oracle's
indexer scores and from adversarial value sets (many ties, one hot block,
sorted runs)."""
from __future__ import annotations

import numpy as np
import pytest

import gen
import oracle


def _blocks(row, K):
    n = row.size
    nb = (n + 7) // 8
    pad = np.full(nb * 8 - n, -np.inf)
    bm = np.concatenate([row, pad]).reshape(nb, 8).max(1)
    if nb <= K:
        return -np.inf, np.arange(nb)
    tau = np.sort(bm)[::-1][K - 1]
    above = np.nonzero(bm > tau)[0]
    ties = np.nonzero(bm == tau)[0][: K - above.size]
    return tau, np.concatenate([above, ties])


def _check(row, K):
    tau, blocks = _blocks(row, K)
    cand = np.concatenate([np.arange(8 * b, min(8 * b + 8, row.size)) for b in blocks]) if blocks.size else np.array([], int)
    assert int((row >= tau).sum()) >= min(K, row.size)
    outside = np.setdiff1d(np.arange(row.size), cand)
    assert (row[outside] <= tau).all()
    want = oracle.topk(oracle.FULL, row.astype(np.float32)[None, None, :], None, K=K)[0, 0]
    want = set(int(j) for j in want if j >= 0)
    order = np.argsort(-row[cand], kind="stable")[: min(K, cand.size)]
    got = set(int(j) for j in cand[order])
    assert len(got) == len(want)
    kth = min(row[j] for j in want) if want else None
    assert all(row[j] == kth for j in got ^ want)   # they may differ only by ties at the K-th value


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


def test_bound_with_interval_block_maxima():
    """With only an interval L_b <= max_b <= U_b per block (e.g. from packed
    low-precision arithmetic), let tau_L be the K-th largest L_b: at least K
    scores reach tau_L, so the blocks with U_b >= tau_L hold a Top-K of the
    row (every score elsewhere is < tau_L)."""
    rng = np.random.default_rng(11)
    K = 64
    for trial in range(40):
        n = int(rng.integers(600, 4000))
        row = rng.standard_normal(n) if trial % 2 else rng.integers(0, 6, n).astype(float)
        row = row.astype(np.float32).astype(np.float64)      # the values the selection sees
        nb = (n + 7) // 8
        bm = np.concatenate([row, np.full(nb * 8 - n, -np.inf)]).reshape(nb, 8).max(1)
        err = 10.0 ** rng.uniform(-6, -2)
        lo = bm - err * (np.abs(bm) + 1) * rng.random(nb)
        hi = bm + err * (np.abs(bm) + 1) * rng.random(nb)
        tau_l = np.sort(lo)[::-1][K - 1]
        keep = np.nonzero(hi >= tau_l)[0]
        assert keep.size >= K
        cand = np.concatenate([np.arange(8 * b, min(8 * b + 8, n)) for b in keep])
        outside = np.setdiff1d(np.arange(n), cand)
        assert (row[outside] < tau_l).all()
        want = oracle.topk(oracle.FULL, row.astype(np.float32)[None, None, :], None, K=K)[0, 0]
        kth = min(row[j] for j in want)
        got = cand[np.argsort(-row[cand], kind="stable")[:K]]
        assert all(row[j] == kth for j in set(got.tolist()) ^ set(want.tolist()))
