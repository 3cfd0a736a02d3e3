"""Pins of the oracle's sliding-window branch (FP8 window KV) and its
log-sum-exp merge with the sparse branch: the merged result must be the
softmax attention over the union of both branches' entries, computed here
directly (dense numpy fp64 over the concatenated dequantised rows)."""
import numpy as np
import torch

import gen
import oracle


def _e4m3_values(b):
    return torch.from_numpy(np.ascontiguousarray(b)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _bf16_values(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _dense(q, K, V, scale):
    """q [H, D], K [n, D], V [n, dv] -> out [H, dv], lse [H] (softmax attention)."""
    z = scale * q @ K.T
    m = z.max(1, keepdims=True)
    e = np.exp(z - m)
    return (e @ V) / e.sum(1, keepdims=True), (m[:, 0] + np.log(e.sum(1)))


def _case(seed, B=2, T=1, H=4, D=64, dv=48, N=300, K=40, W=24):
    rng = np.random.default_rng(seed)
    q = gen.bf16_bits(torch.from_numpy(rng.standard_normal((B, T, H, D)).astype(np.float32))).numpy().view(np.uint16)
    codes, scales = oracle.quantize_kv_fp4(
        gen.bf16_bits(torch.from_numpy(rng.standard_normal((B * N, D)).astype(np.float32))).numpy().view(np.uint16))
    idx = np.stack([rng.permutation(N)[:K] for _ in range(B * T)]).astype(np.int32).reshape(B, T, K)
    kvw = gen.e4m3_bytes(torch.from_numpy(rng.standard_normal((B, W, D)).astype(np.float32))).numpy()
    return q, codes, scales, idx, kvw, N


def test_merge_is_attention_over_the_union_of_both_branches():
    B, T, H, D, dv, N, K, W = 2, 1, 4, 64, 48, 300, 40, 24
    q, codes, scales, idx, kvw, N = _case(1)
    kl = np.full(B * T, N, np.int32)
    sl = np.array([W, 17], np.int32)
    scale = 0.125
    o_s, l_s, bad = oracle.sparse_attn(q, codes, scales, N, idx, kl, scale, dv)
    assert bad == 0
    out, lse = oracle.swa_attn_merge(q, kvw, sl, scale, dv, o_s, l_s)
    deq = oracle.dequant_fp4(codes, scales)
    for b in range(B):
        Ks = deq[b * N + idx[b, 0]]
        Kw = _e4m3_values(kvw[b, :sl[b]])
        Ku = np.concatenate([Ks, Kw])
        ref_o, ref_l = _dense(_bf16_values(q[b, 0]), Ku, Ku[:, :dv], scale)
        assert np.allclose(out[b, 0], ref_o, rtol=1e-12, atol=1e-12)
        assert np.allclose(lse[b, 0], ref_l, rtol=1e-12, atol=1e-12)


def test_window_alone_and_single_row_window():
    q, codes, scales, idx, kvw, N = _case(2)
    B, W = 2, 24
    out, lse = oracle.swa_attn_merge(q, kvw, np.array([W, 1], np.int32), 0.2, 48)
    for b, n in ((0, W), (1, 1)):
        Kw = _e4m3_values(kvw[b, :n])
        ref_o, ref_l = _dense(_bf16_values(q[b, 0]), Kw, Kw[:, :48], 0.2)
        assert np.allclose(out[b, 0], ref_o, rtol=1e-12, atol=1e-12) and np.allclose(lse[b, 0], ref_l)
    # one row: the output is that row's first dv channels for every head
    assert np.array_equal(out[1, 0], np.tile(_e4m3_values(kvw[1, 0])[:48], (4, 1)))


def test_empty_window_returns_the_sparse_branch_and_empty_both_gives_zero():
    q, codes, scales, idx, kvw, N = _case(3)
    o_s = np.random.default_rng(0).standard_normal((2, 1, 4, 48))
    l_s = np.array([[[0.5, -1.0, np.inf * -1, 2.0]], [[1.0, 1.0, 1.0, 1.0]]])
    out, lse = oracle.swa_attn_merge(q, kvw, np.array([0, 0], np.int32), 0.1, 48, o_s, l_s)
    fin = np.isfinite(l_s)
    assert np.array_equal(out[fin], o_s[fin]) and np.array_equal(lse[fin], l_s[fin])
    assert (out[~fin] == 0).all() and np.isneginf(lse[~fin]).all()


def test_sparse_lse_minus_inf_leaves_the_window_branch():
    q, codes, scales, idx, kvw, N = _case(4)
    o_s = np.full((2, 1, 4, 48), 123.0)
    l_s = np.full((2, 1, 4), -np.inf)
    a, la = oracle.swa_attn_merge(q, kvw, np.array([24, 24], np.int32), 0.1, 48, o_s, l_s)
    b, lb = oracle.swa_attn_merge(q, kvw, np.array([24, 24], np.int32), 0.1, 48)
    assert np.array_equal(a, b) and np.array_equal(la, lb)
