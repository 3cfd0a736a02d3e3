"""Shared comparison helpers for the GPU parity tests.

Tolerances (applied to the CUDA library against the fp64 CPU oracle on the
same inputs):
  * FP4 codes and scale bytes: bit-exact.
  * indexer scores: |s_gpu - s_ref| <= 1e-4 * max(|s_ref|, sum_h |w_h| sum_d |q_hd k_d|)
    (the magnitude sum is the dot product's conditioning; a score near 0 after
    ReLU has no meaningful pure relative error).  This widens the plain
    "1e-4 relative" of the specification where q.k cancels; the plain relative
    error |s_gpu - s_ref| / |s_ref| <= 1e-4 is also required of every score
    whose magnitude sum is at most COND_MAX times the score (no heavy
    cancellation), and its worst value is returned.
  * Top-K / pool sets: equal, except members whose oracle score lies within
    1e-5 relative of the oracle's K-th score (the tie band).
  * attention: per (b, t, h) row, max_c |o_gpu - o_ref| / max_c |o_ref| <= 2e-3.
"""
from __future__ import annotations

import numpy as np

SCORE_RTOL = 1e-4
COND_MAX = 10.0
TIE_RTOL = 1e-5
ATTN_RTOL = 2e-3


def check_scores(got, ref, mag, what="scores"):
    got = np.asarray(got, np.float64)
    fin = np.isfinite(ref)
    assert (np.isneginf(got) == ~fin).all(), "%s: -inf pattern differs (%d mismatches)" % (
        what, int((np.isneginf(got) != ~fin).sum()))
    err = np.abs(got[fin] - ref[fin])
    tol = SCORE_RTOL * np.maximum(np.abs(ref[fin]), mag[fin])
    bad = err > tol
    assert not bad.any(), "%s: %d of %d outside tolerance, worst err/tol %.3g" % (
        what, int(bad.sum()), bad.size, float((err / np.maximum(tol, 1e-300)).max()))
    r, m = np.abs(ref[fin]), mag[fin]
    wc = (r > 0) & (m <= COND_MAX * r)          # well-conditioned scores: the plain relative error
    plain = float((err[wc] / r[wc]).max()) if wc.any() else 0.0
    assert plain <= SCORE_RTOL, "%s: plain relative error %.3g on well-conditioned scores" % (what, plain)
    return plain


def kth_score(ref_row, K):
    v = ref_row[np.isfinite(ref_row)]
    if v.size < K:
        return None
    return np.partition(v, v.size - K)[v.size - K]


def check_selection(got_row, want_row, ref_scores_of, K, what="topk"):
    """got_row/want_row: selected ids (-1 padded).  ref_scores_of(ids) -> the
    oracle's fp64 score of each id.  Sets must agree outside the tie band."""
    got = [int(x) for x in got_row if x != -1]
    want = [int(x) for x in want_row if x != -1]
    assert len(got) == len(set(got)), "%s: duplicate ids" % what
    assert len(got) == len(want), "%s: %d selected, oracle %d" % (what, len(got), len(want))
    gs, ws = set(got), set(want)
    diff = sorted(gs ^ ws)
    if not diff:
        return 0
    ws_scores = ref_scores_of(np.array(sorted(ws)))
    kth = float(np.min(ws_scores))            # the oracle's K-th (smallest selected) score
    d_scores = ref_scores_of(np.array(diff))
    band = np.abs(d_scores - kth) <= TIE_RTOL * abs(kth)
    assert band.all(), "%s: %d ids differ outside the tie band (kth=%r, worst |ds|=%r)" % (
        what, int((~band).sum()), kth, float(np.abs(d_scores - kth).max()))
    return len(diff)


def check_attn(got, ref, what="attention"):
    got = np.asarray(got, np.float64)
    den = np.abs(ref).max(-1)
    num = np.abs(got - ref).max(-1)
    zero = den == 0
    assert (num[zero] == 0).all(), "%s: nonzero output where the oracle is 0" % what
    rel = num[~zero] / den[~zero]
    worst = float(rel.max()) if rel.size else 0.0
    assert worst <= ATTN_RTOL, "%s: max row rel err %.3g > %g" % (what, worst, ATTN_RTOL)
    return worst


def check_lse(got, ref, what="lse"):
    got = np.asarray(got, np.float64)
    fin = np.isfinite(ref)
    assert (np.isneginf(got) == ~fin).all(), "%s: -inf pattern differs" % what
    err = np.abs(got[fin] - ref[fin])
    assert (err <= 1e-4 * np.maximum(1.0, np.abs(ref[fin]))).all(), "%s: max err %.3g" % (what, err.max())
