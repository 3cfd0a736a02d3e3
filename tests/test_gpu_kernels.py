"""GPU parity of each libcsa2 call against the CPU oracle on identical inputs
(through the C ABI via the Python binding).  Marked gpu."""
import numpy as np
import pytest
import torch

import gen
import oracle
from helpers import check_attn, check_lse, check_scores

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def csa2():
    import sparse_attention_fp4_quantize_gb300 as m
    return m


def _bits_to_float(bits_u16):
    return torch.from_numpy(np.ascontiguousarray(bits_u16).view(np.int16)).view(torch.bfloat16).double().numpy()


def _gpu_quant(csa2, bits_u16, dst_slot=None, n_slots=None, stride=None, flag=None):
    R, D = bits_u16.shape
    src = torch.from_numpy(np.ascontiguousarray(bits_u16).view(np.int16))
    if stride is not None:
        wide = torch.zeros(R, stride, dtype=torch.int16)
        wide[:, :D] = src
        kv = wide.to(DEV)[:, :D]
    else:
        kv = src.to(DEV)
    S = R if n_slots is None else n_slots
    codes = torch.zeros(S, D // 2, dtype=torch.uint8, device=DEV)
    scales = torch.zeros(S, D // 16, dtype=torch.uint8, device=DEV)
    ds = None if dst_slot is None else torch.from_numpy(np.asarray(dst_slot, np.int64)).to(DEV)
    csa2.csa2_quantize_kv_fp4(kv, codes, scales, dst_slot=ds, err_flag=flag)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


def _assert_bitexact(got, want, what):
    gc, gs = got
    wc, ws = want
    bad_s = np.nonzero(gs != ws)
    assert bad_s[0].size == 0, "%s: %d scale bytes differ, first at %s: gpu %02x oracle %02x" % (
        what, bad_s[0].size, (bad_s[0][0], bad_s[1][0]), gs[bad_s][0], ws[bad_s][0])
    bad_c = np.nonzero(gc != wc)
    assert bad_c[0].size == 0, "%s: %d code bytes differ, first at %s: gpu %02x oracle %02x" % (
        what, bad_c[0].size, (bad_c[0][0], bad_c[1][0]), gc[bad_c][0], wc[bad_c][0])


# ---------------------------------------------------------------------------- quantise
def _finite_bf16_patterns():
    p = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    return p[((p >> 7) & 0xFF) != 0xFF]


def test_quantize_exhaustive_amax_sweep(csa2):
    """Every finite bf16 value as the amax of a group (at every position)."""
    v = _finite_bf16_patterns()
    rows = np.zeros((v.size, 16), np.uint16)
    rows[np.arange(v.size), np.arange(v.size) % 16] = v
    _assert_bitexact(_gpu_quant(csa2, rows), oracle.quantize_kv_fp4(rows), "amax sweep")


def test_quantize_exhaustive_codes_per_scale(csa2):
    """For every positive finite scale byte s: every finite bf16 x with
    |x| <= 6s, quantised in groups whose amax is exactly 6s (so the group scale
    is s and |x|/s covers [0, 6] including every tie)."""
    pats = _finite_bf16_patterns()
    vals = _bits_to_float(pats)
    setter_bits = torch.tensor([6.0 * oracle.e4m3_value(sb) for sb in range(1, 0x7F)],
                               dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    groups = []
    for i, sb in enumerate(range(1, 0x7F)):
        A = 6.0 * oracle.e4m3_value(sb)
        xs = pats[np.abs(vals) <= A]
        n = -(-xs.size // 15)
        g = np.zeros((n, 16), np.uint16)
        flat = np.zeros(n * 15, np.uint16)
        flat[: xs.size] = xs
        g[:, 1:] = flat.reshape(n, 15)
        g[:, 0] = setter_bits[i] | (0x8000 if i % 2 else 0)      # +-6s
        groups.append(g)
    rows = np.concatenate(groups)
    assert rows.shape[0] > 100_000
    got = _gpu_quant(csa2, rows)
    want = oracle.quantize_kv_fp4(rows)
    _assert_bitexact(got, want, "code sweep")
    assert (want[1][:, 0] >= 1).all()


def test_quantize_golden_groups(csa2):
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "fp4_groups.txt")
    for ln in open(path):
        ln = ln.strip()
        if not ln or ln.startswith("#"):
            continue
        name, xs, sb, cs = [p.strip() for p in ln.split(";")]
        bits = torch.tensor([float(x) for x in xs.split()]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        codes, scales = _gpu_quant(csa2, bits.reshape(1, 16))
        want = [int(c, 16) for c in cs.split()]
        assert scales[0, 0] == int(sb, 16), name
        assert list(codes[0]) == [want[2 * i] | (want[2 * i + 1] << 4) for i in range(8)], name


@pytest.mark.parametrize("D,rms", [(128, True), (576, True), (576, False), (64, True), (1024, False)])
def test_quantize_random_rows(csa2, D, rms):
    R = 3001
    rows = gen.as_numpy(gen.kv_rows(7, D, R, D, rms=rms, rope_pos=torch.arange(R) * 4 if rms else None))
    _assert_bitexact(_gpu_quant(csa2, rows), oracle.quantize_kv_fp4(rows), "random D=%d" % D)


def test_quantize_scatter_strided_and_bad_slots(csa2):
    R, D, S = 257, 576, 1000
    rows = gen.as_numpy(gen.kv_rows(8, 1, R, D))
    slots = np.random.default_rng(0).permutation(S)[:R].astype(np.int64)
    want = oracle.quantize_kv_fp4(rows, dst_slot=slots, n_slots=S)
    got = _gpu_quant(csa2, rows, dst_slot=slots, n_slots=S, stride=D + 64)
    _assert_bitexact(got, want, "scatter+stride")
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    bad = slots.copy()
    bad[3] = S          # out of range
    bad[5] = -2
    got = _gpu_quant(csa2, rows, dst_slot=bad, n_slots=S, flag=flag)
    assert int(flag.item()) & csa2.FLAG_BAD_SLOT
    keep = np.ones(R, bool)
    keep[[3, 5]] = False
    assert (got[0][bad[keep]] == want[0][slots[keep]]).all()


def test_quantize_full_append_size_sampled(csa2):
    """1,048,576 x 576 rows (the append workload) on the GPU; sampled rows vs the oracle."""
    w = gen.APPEND_POOL
    R, D = w.B * w.N, w.D
    rows = gen.kv_cache_rows(w, device=DEV)
    codes = torch.empty(R, D // 2, dtype=torch.uint8, device=DEV)
    scales = torch.empty(R, D // 16, dtype=torch.uint8, device=DEV)
    csa2.csa2_quantize_kv_fp4(rows, codes, scales)
    torch.cuda.synchronize()
    pick = np.unique(np.concatenate([np.random.default_rng(1).integers(0, R, 6000), [0, R - 1]]))
    sel = torch.from_numpy(pick).to(DEV)
    want = oracle.quantize_kv_fp4(gen.as_numpy(rows[sel]))
    _assert_bitexact((codes[sel].cpu().numpy(), scales[sel].cpu().numpy()), want, "append sample")


# ---------------------------------------------------------------------------- index score
def _score_gpu(csa2, mode, q, w, k, kv_len, pool=None, M=None, flag=None):
    B, T = q.shape[0], q.shape[1]
    N = k.shape[1]
    M = N if mode == csa2.MODE_FULL else 8 * pool.shape[-1]
    out = torch.full((B, T, M), 12345.0, device=DEV)
    csa2.csa2_index_score(mode, q.to(DEV), w.to(DEV), k.to(DEV), kv_len.to(DEV), out,
                          pool_blocks=None if pool is None else pool.to(DEV), err_flag=flag)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _score_ref(mode, q, w, k, kv_len, pool=None):
    dt = oracle.BF16 if q.dtype == torch.int16 else oracle.FP8_E4M3
    return oracle.index_score(mode, gen.as_numpy(q), dt, gen.as_numpy(w), gen.as_numpy(k), dt,
                              gen.as_numpy(kv_len), pool=None if pool is None else gen.as_numpy(pool),
                              with_mag=True)


def test_index_score_tiny_bf16(csa2):
    w = gen.TINY_FULL_DECODE
    q, wt, k = gen.indexer_inputs(w)
    kl = gen.kv_lengths(w)
    ref, mag = _score_ref(0, q, wt, k, kl)
    check_scores(_score_gpu(csa2, 0, q, wt, k, kl), ref, mag)


@pytest.mark.parametrize("B,T,N", [(3, 1, 1000), (2, 5, 777), (1, 2, 16), (4, 1, 1),
                                   (2, 100, 1000), (1, 64, 130), (3, 200, 4100)])   # T >= 64: tensor-core path
def test_index_score_full_ragged_fp8(csa2, B, T, N):
    q = gen.normal_e4m3(9, 1, (B, T, 4, 64))
    k = gen.normal_e4m3(9, 2, (B, N, 64))
    wt = gen.uniform01(9, 3, (B, T, 4))
    kl = torch.tensor([(N * (i + 1)) // (B * T) + (i % 3) for i in range(B * T)], dtype=torch.int32)
    kl[0] = 0
    if B * T > 2:
        kl[1] = N + 50
    ref, mag = _score_ref(0, q, wt, k, kl)
    check_scores(_score_gpu(csa2, 0, q, wt, k, kl), ref, mag)


def test_index_score_full_batched_decode_full_size(csa2):
    w = gen.FULL_BATCHED_DECODE
    q, wt, k = gen.indexer_inputs(w)
    kl = gen.kv_lengths(w)
    ref, mag = _score_ref(0, q, wt, k, kl)
    check_scores(_score_gpu(csa2, 0, q, wt, k, kl), ref, mag)


def test_index_score_reindex_with_bad_pool_ids(csa2):
    B, N, P = 2, 4000, 64
    q = gen.normal_e4m3(10, 1, (B, 1, 4, 64))
    k = gen.normal_e4m3(10, 2, (B, N, 64))
    wt = gen.uniform01(10, 3, (B, 1, 4))
    kl = torch.tensor([4000, 3001], dtype=torch.int32)
    g = torch.Generator().manual_seed(3)
    pool = torch.randint(0, (N + 7) // 8, (B, 1, P), generator=g, dtype=torch.int32)
    pool[0, 0, 5] = -1
    pool[1, 0, 7] = 390          # partially beyond kv_len 3001 (block 375 holds j 3000)
    ref, mag = _score_ref(1, q, wt, k, kl, pool)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    check_scores(_score_gpu(csa2, 1, q, wt, k, kl, pool, flag=flag), ref, mag)
    assert int(flag.item()) == 0
    bad = pool.clone()
    bad[0, 0, 9] = (N + 7) // 8       # out of range -> -inf, flagged
    bad[1, 0, 2] = -5
    got = _score_gpu(csa2, 1, q, wt, k, kl, bad, flag=flag)
    assert int(flag.item()) & csa2.FLAG_BAD_POOL
    assert np.isneginf(got[0, 0, 72:80]).all() and np.isneginf(got[1, 0, 16:24]).all()


def test_index_score_prefill_sampled(csa2):
    """4096 causal queries x 32768 keys on the GPU; 6 sampled queries vs the oracle."""
    w = gen.PREFILL_CHUNK
    q, wt, k = gen.indexer_inputs(w)
    kl = gen.kv_lengths(w)
    got = _score_gpu(csa2, 0, q, wt, k, kl)
    pick = [0, 1, 1000, 2047, 4094, 4095]
    ref, mag = _score_ref(0, q[:, pick], wt[:, pick], k, kl[pick])
    check_scores(got[:, pick], ref, mag)


# ---------------------------------------------------------------------------- top-k / pool
def _topk_gpu(csa2, mode, scores, K, kv_len=None, pool=None):
    B, T, M = scores.shape
    idx = torch.full((B, T, K), -99, dtype=torch.int32, device=DEV)
    csa2.csa2_topk(mode, torch.from_numpy(scores).to(DEV), idx,
                   kv_len=None if kv_len is None else torch.from_numpy(kv_len).to(DEV),
                   pool_blocks=None if pool is None else torch.from_numpy(pool).to(DEV))
    torch.cuda.synchronize()
    return idx.cpu().numpy()


def _same_sets(got, want):
    B, T, K = got.shape
    for b in range(B):
        for t in range(T):
            g = got[b, t]
            assert len(set(g[g != -1])) == (g != -1).sum(), "duplicates"
            assert sorted(g.tolist()) == sorted(want[b, t].tolist()), (b, t)


@pytest.mark.parametrize("B,M,K,kind", [(1, 1024, 512, "rand"), (32, 16384, 512, "rand"), (8, 16384, 512, "ties"),
                                        (100, 4096, 512, "rand"), (3, 32768, 2048, "rand"), (5, 700, 512, "few"),
                                        (7, 5000, 1, "rand"), (2, 64, 16, "allsame"), (4, 262144, 512, "rand"),
                                        (16, 8192, 512, "ties")])
def test_topk_full_matches_oracle_exactly(csa2, B, M, K, kind):
    rng = np.random.default_rng(B * 7 + M)
    if kind == "ties":
        s = rng.integers(0, 5, (B, 1, M)).astype(np.float32)
    elif kind == "allsame":
        s = np.full((B, 1, M), 0.25, np.float32)
    else:
        s = rng.random((B, 1, M), dtype=np.float32)
    if kind == "few":
        s[rng.random(s.shape) < 0.6] = -np.inf
    kl = rng.integers(max(1, M // 2), M + 1, B).astype(np.int32)
    kl[0] = M
    want = oracle.topk(oracle.FULL, s, kl, K=K)
    got = _topk_gpu(csa2, 0, s, K, kv_len=kl)
    _same_sets(got, want)


def test_topk_reindex_maps_to_global_positions(csa2):
    B, P, K = 8, 2048, 512
    rng = np.random.default_rng(4)
    pool = np.stack([rng.permutation(32768)[:P] for _ in range(B)]).astype(np.int32).reshape(B, 1, P)
    pool[0, 0, :100] = -1
    s = rng.random((B, 1, 8 * P), dtype=np.float32)
    s[0, 0, :800] = -np.inf
    s[1, 0, ::3] = 0.5                      # ties
    want = oracle.topk(oracle.REINDEX, s, None, pool=pool, K=K)
    got = _topk_gpu(csa2, 1, s, K, pool=pool)
    _same_sets(got, want)


def test_topk_reuse_leaves_idx_untouched(csa2):
    s = torch.rand(2, 1, 1000, device=DEV)
    idx = torch.arange(2 * 512, dtype=torch.int32, device=DEV).reshape(2, 1, 512)
    before = idx.clone()
    csa2.csa2_topk(csa2.MODE_REUSE, s, idx)
    torch.cuda.synchronize()
    assert torch.equal(idx, before)


@pytest.mark.parametrize("B,N,kind", [(8, 262144, "rand"), (16, 65536, "rand"), (2, 16384, "rand"),
                                      (3, 1003, "rand"), (4, 100000, "ties")])
def test_build_pool_matches_oracle_exactly(csa2, B, N, kind):
    rng = np.random.default_rng(N)
    if kind == "ties":
        s = rng.integers(0, 20, (B, 1, N)).astype(np.float32)
    else:
        s = rng.random((B, 1, N), dtype=np.float32)
    kl = rng.integers(N // 2, N + 1, B).astype(np.int32)
    kl[0] = N
    want = oracle.build_pool(s, kl, P=2048)
    pool = torch.full((B, 1, 2048), -99, dtype=torch.int32, device=DEV)
    csa2.csa2_build_pool(torch.from_numpy(s).to(DEV), torch.from_numpy(kl).to(DEV), pool)
    torch.cuda.synchronize()
    _same_sets(pool.cpu().numpy(), want)


# ---------------------------------------------------------------------------- attention
def _kv_planes(w, B, N, seed_stream=10):
    rows = gen.as_numpy(gen.kv_cache_rows(gen.scaled(w, B=B, N=N), stream=seed_stream))
    return oracle.quantize_kv_fp4(rows)


def _attn_gpu(csa2, q, codes, scales, N, idx, kv_len, sm, dv, flag=None):
    B, T, H, D = q.shape
    K = idx.shape[-1]
    out = torch.full((B, T, H, dv), 7.0, device=DEV)
    lse = torch.full((B, T, H), 7.0, device=DEV)
    ws = csa2.workspace_for_attn(B, T, H, D, dv, K, device=DEV)
    csa2.csa2_sparse_attn_fp4(csa2.MODE_FULL, q.to(DEV), torch.from_numpy(codes).to(DEV),
                              torch.from_numpy(scales).to(DEV), N, torch.from_numpy(idx).to(DEV), out, sm,
                              kv_len=None if kv_len is None else torch.from_numpy(kv_len).to(DEV), lse=lse,
                              err_flag=flag, workspace=ws)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("base,B,T,N,K,H,pad", [
    ("tiny", 1, 1, 1024, 512, 16, 0.0),
    ("tiny", 3, 2, 700, 100, 32, 0.2),
    ("full", 4, 1, 16384, 512, 64, 0.0),
    ("full", 2, 3, 5000, 512, 128, 0.1),
    ("full", 40, 1, 3000, 512, 64, 0.0),      # many rows: no split-KV
    ("full", 1, 1, 600, 33, 64, 0.0),
    ("full", 2, 1, 2000, 1, 64, 0.0),
    ("full", 3, 1, 4000, 1024, 64, 0.1),      # K > 512: the mma.sync kernel
    ("full", 2, 2, 3000, 700, 64, 0.0),       # K > 512, not a multiple of the entry tile
    ("full", 1, 1, 3000, 1500, 64, 0.0),      # one row, K = 1500: split-KV partials + combine
    # enough (token, 64-head) items for the one-CTA-per-item kernel (more than a quarter of the SMs)
    ("full", 48, 1, 3000, 512, 64, 0.1),      # four tiles, padded rows
    ("full", 24, 2, 2000, 300, 64, 0.0),      # three tiles, the last one ragged, two tokens per row
    ("full", 40, 1, 900, 100, 128, 0.2),      # one tile, two head blocks
    ("full", 20, 1, 5000, 257, 128, 0.0),     # three tiles, one entry in the last
    # more items than SMs: each persistent CTA takes several in turn
    ("full", 320, 1, 3000, 300, 64, 0.1),
    ("full", 160, 1, 2000, 200, 128, 0.0),
])
def test_sparse_attn_matches_oracle(csa2, base, B, T, N, K, H, pad):
    w0 = gen.TINY_FULL_DECODE if base == "tiny" else gen.FULL_BATCHED_DECODE
    w = gen.scaled(w0, B=B, T=T, N=N, K=K, H=H)
    codes, scales = _kv_planes(w0, B, N)
    kl = np.full(B * T, N, np.int32)
    kl[-1] = max(K, N - 7)
    idx = gen.as_numpy(gen.random_indices(w, torch.from_numpy(kl), frac_pad=pad))
    q = gen.attn_query(w)
    sm = gen.softmax_scale(w.D)
    got, glse = _attn_gpu(csa2, q, codes, scales, N, idx, kl, sm, w.dv)
    ref, rlse, bad = oracle.sparse_attn(gen.as_numpy(q), codes, scales, N, idx, kl, sm, w.dv)
    assert bad == 0
    check_attn(got, ref)
    check_lse(glse, rlse)


def test_sparse_attn_many_tokens_running_max_moves(csa2):
    """Launches with many (token, 64-head) items take one CTA per item and an
    online softmax over its 128-entry tiles, whose running maximum moves only
    when a tile's maximum exceeds it by a wide margin.  Entries 2000.. of every
    sequence get scale bytes 16x larger (four more exponent steps), so their
    logits are about 16x wider: tokens whose large entries sit in the last two
    tiles raise the maximum after two tiles (the partial output is rescaled),
    the others meet them in the first two tiles (later tiles add almost
    nothing), and one token alternates them.  Against the oracle."""
    B, N, K = 48, 3000, 512
    w = gen.scaled(gen.FULL_BATCHED_DECODE, B=B, T=1, N=N, K=K, H=64)
    codes, scales = _kv_planes(gen.FULL_BATCHED_DECODE, B, N)
    scales = scales.copy()
    big = np.zeros(B * N, bool)
    for bb in range(B):
        big[bb * N + 2000:(bb + 1) * N] = True
    sc = scales[big].astype(np.int32)
    scales[big] = np.where(sc == 0, 0, np.minimum(sc + 0x20, 0x7E)).astype(np.uint8)
    rng = np.random.default_rng(7)
    idx = np.empty((B, 1, K), np.int32)
    for bb in range(B):
        small = rng.choice(2000, 256, replace=False)
        large = 2000 + rng.choice(N - 2000, 256, replace=False)
        if bb % 2 == 0:
            row = np.concatenate([small, large])
        else:
            row = np.concatenate([large, small])
        if bb == 1:
            row = np.stack([small, large], 1).reshape(-1)
        idx[bb, 0] = row
    q = gen.attn_query(w)
    sm = gen.softmax_scale(w.D)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    got, glse = _attn_gpu(csa2, q, codes, scales, N, idx, None, sm, w.dv, flag=flag)
    ref, rlse, bad = oracle.sparse_attn(gen.as_numpy(q), codes, scales, N, idx, None, sm, w.dv)
    assert bad == 0 and int(flag.item()) == 0
    check_attn(got, ref)
    check_lse(glse, rlse)


def test_sparse_attn_cluster_slices_empty_and_repeated_entries(csa2):
    """K = 512 on the tensor-core path splits a row over 4 CTAs of 128
    entries.  Rows whose last, first or first three slices hold only -1, a
    row selecting one entry 512 times, one selecting every entry twice (in
    different slices) and one with every other slot -1, against the oracle;
    kv_len NULL stands for N."""
    N, K = 3000, 512
    w = gen.scaled(gen.FULL_BATCHED_DECODE, B=6, T=1, N=N, K=K, H=64)
    codes, scales = _kv_planes(gen.FULL_BATCHED_DECODE, 6, N)
    idx = gen.as_numpy(gen.random_indices(w, torch.full((6,), N, dtype=torch.int32))).copy()
    idx[0, 0, 384:] = -1
    idx[1, 0, :128] = -1
    idx[2, 0, :384] = -1
    idx[3, 0, :] = 1234
    idx[4, 0, 256:] = idx[4, 0, :256]
    idx[5, 0, 1::2] = -1
    q = gen.attn_query(w)
    sm = gen.softmax_scale(w.D)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    got, glse = _attn_gpu(csa2, q, codes, scales, N, idx, None, sm, w.dv, flag=flag)
    ref, rlse, bad = oracle.sparse_attn(gen.as_numpy(q), codes, scales, N, idx, None, sm, w.dv)
    assert bad == 0 and int(flag.item()) == 0
    check_attn(got, ref)
    check_lse(glse, rlse)


def test_sparse_attn_empty_rows_and_bad_indices(csa2):
    w = gen.scaled(gen.FULL_BATCHED_DECODE, B=2, T=2, N=1000, K=64)
    codes, scales = _kv_planes(gen.FULL_BATCHED_DECODE, 2, 1000)
    kl = np.array([1000, 1000, 500, 1000], np.int32)
    idx = gen.as_numpy(gen.random_indices(w, torch.from_numpy(kl)))
    idx[0, 0, :] = -1                    # empty row
    idx[0, 1, 3] = 1000                  # >= kv_len
    idx[1, 0, 4] = 700                   # >= kv_len (500)
    idx[1, 1, 5] = -3
    q = gen.attn_query(w)
    sm = gen.softmax_scale(w.D)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    got, glse = _attn_gpu(csa2, q, codes, scales, 1000, idx, kl, sm, w.dv, flag=flag)
    ref, rlse, bad = oracle.sparse_attn(gen.as_numpy(q), codes, scales, 1000, idx, kl, sm, w.dv)
    assert bad == 3 and int(flag.item()) & csa2.FLAG_BAD_INDEX
    assert (got[0, 0] == 0).all() and np.isneginf(glse[0, 0]).all()
    check_attn(got, ref)
    check_lse(glse, rlse)


def test_sparse_attn_workspace_is_required_when_split(csa2):
    q = torch.zeros(1, 1, 64, 576, dtype=torch.int16, device=DEV)
    codes = torch.zeros(100, 288, dtype=torch.uint8, device=DEV)
    scales = torch.zeros(100, 36, dtype=torch.uint8, device=DEV)
    idx = torch.zeros(1, 1, 1536, dtype=torch.int32, device=DEV)     # K > 512 on one row: split-KV partials
    out = torch.zeros(1, 1, 64, 512, device=DEV)
    assert csa2.csa2_sparse_attn_workspace_bytes(1, 1, 64, 576, 512, 512) == 0   # tcgen05 path: no scratch
    assert csa2.csa2_sparse_attn_workspace_bytes(1, 1, 64, 576, 512, 1536) > 0
    with pytest.raises(csa2.Csa2Error) as e:
        csa2.csa2_sparse_attn_fp4(0, q, codes, scales, 100, idx, out, 0.1)
    assert e.value.status == 3


def test_bounded_wait_times_out_and_the_context_stays_usable():
    """A wait that nothing completes gives up, flags CSA2_FLAG_TIMEOUT, and the
    next launch on the same context runs normally."""
    import sparse_attention_fp4_quantize_gb300 as csa2
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    csa2.csa2_selftest_bounded_wait(flag, max_polls=2048)
    torch.cuda.synchronize()
    assert int(flag.item()) & csa2.FLAG_TIMEOUT
    rows = gen.kv_rows(0, 1, 64, 128, device="cuda")
    codes = torch.empty(64, 64, dtype=torch.uint8, device="cuda")
    scales = torch.empty(64, 8, dtype=torch.uint8, device="cuda")
    csa2.csa2_quantize_kv_fp4(rows, codes, scales)
    torch.cuda.synchronize()
    want_c, want_s = oracle.quantize_kv_fp4(gen.as_numpy(rows).reshape(64, 128))
    assert (codes.cpu().numpy() == want_c).all() and (scales.cpu().numpy() == want_s).all()


@pytest.mark.parametrize("B,N,K,H", [(4, 16384, 512, 64), (3, 3000, 300, 128), (2, 5000, 1024, 64)])
def test_sparse_attn_prefetch_variant_is_the_same_attention(csa2, B, N, K, H):
    """csa2_sparse_attn_fp4_prefetch only adds an L2 hint for another pair of
    planes: its output and lse are bitwise those of csa2_sparse_attn_fp4, the
    hinted planes are left untouched, and on the split-KV path (K > 512) the
    hint is simply not issued."""
    w = gen.scaled(gen.FULL_BATCHED_DECODE, B=B, N=N, K=K, H=H)
    kv_len = gen.kv_lengths(w).clamp(max=N)
    codes, scales = gen.fp4_planes(5, 1, B * N, 576, device=DEV)
    nc, ns = gen.fp4_planes(5, 2, B * N, 576, device=DEV)
    nc0, ns0 = nc.clone(), ns.clone()
    idx = gen.random_indices(w, kv_len, frac_pad=0.05).to(DEV)
    q = gen.normal_bf16(5, 3, (B, 1, H, 576), device=DEV)
    kl = kv_len.to(DEV)
    ws = csa2.workspace_for_attn(B, 1, H, 576, 512, K, device=DEV)
    outs = []
    for pf in (False, True):
        out = torch.full((B, 1, H, 512), 7.0, device=DEV)
        lse = torch.full((B, 1, H), 7.0, device=DEV)
        flag = torch.zeros(1, dtype=torch.int32, device=DEV)
        if pf:
            csa2.csa2_sparse_attn_fp4_prefetch(csa2.MODE_REUSE, q, codes, scales, N, idx, out, 1 / 24.0,
                                               next_codes=nc, next_scales=ns, kv_len=kl, lse=lse, err_flag=flag,
                                               workspace=ws)
        else:
            csa2.csa2_sparse_attn_fp4(csa2.MODE_REUSE, q, codes, scales, N, idx, out, 1 / 24.0, kv_len=kl, lse=lse,
                                      err_flag=flag, workspace=ws)
        torch.cuda.synchronize()
        assert int(flag.item()) == 0
        outs.append((out, lse))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    assert torch.equal(nc, nc0) and torch.equal(ns, ns0)
