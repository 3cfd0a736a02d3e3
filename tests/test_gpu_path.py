"""End-to-end parity of the hot path on the five synthetic workloads: the GPU
chain (quantise -> score -> pool -> Top-512 -> attention, with Reindex and
Reuse layers) against the oracle chain on the same seeded inputs.  At sizes
the oracle cannot finish in seconds, sampled outputs are checked.  Marked gpu.

Where a stage's output feeds the next, the GPU chain uses its own results and
the oracle chain its own; selections are compared modulo the tie band, and the
attention is additionally checked on the oracle's own index set."""
import numpy as np
import pytest
import torch

import gen
import oracle
from helpers import check_attn, check_lse, check_scores, check_selection

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def csa2():
    import sparse_attention_fp4_quantize_gb300 as m
    return m


def _np(t):
    return gen.as_numpy(t)


def _idx_dt(w):
    return oracle.BF16 if w.idx_dtype == "bf16" else oracle.FP8_E4M3


def _gpu_quant_all(csa2, rows_dev, D):
    R = rows_dev.shape[0]
    codes = torch.empty(R, D // 2, dtype=torch.uint8, device=DEV)
    scales = torch.empty(R, D // 16, dtype=torch.uint8, device=DEV)
    csa2.csa2_quantize_kv_fp4(rows_dev, codes, scales)
    return codes, scales


def _oracle_attn_on_selection(q_np, rows_dev, codes_dev, scales_dev, N, idx_np, kv_len_np, sm, dv):
    """Oracle attention on the entries named by idx_np only: their bf16 rows are
    copied back, quantised by the ORACLE, compared bit-exactly with the GPU
    planes of the same rows, and relabelled to a compact table."""
    B, T, K = idx_np.shape
    D = rows_dev.shape[1]
    sel_rows, remap = [], np.full_like(idx_np, -1)
    base = 0
    for b in range(B):
        ids = np.unique(idx_np[b][idx_np[b] >= 0])
        sel_rows.append(b * N + ids)
        lut = {int(j): base + i for i, j in enumerate(ids)}
        for t in range(T):
            remap[b, t] = [lut.get(int(j), -1) if j >= 0 else -1 for j in idx_np[b, t]]
        base += ids.size
    flat = np.concatenate(sel_rows).astype(np.int64)
    sel = torch.from_numpy(flat).to(DEV)
    oc, os_ = oracle.quantize_kv_fp4(_np(rows_dev[sel]))
    assert (codes_dev[sel].cpu().numpy() == oc).all() and (scales_dev[sel].cpu().numpy() == os_).all()
    # one flat "sequence" holding every selected row; remapped indices are global
    qf = q_np.reshape(1, B * T, *q_np.shape[2:])
    kl = np.full(B * T, oc.shape[0], np.int32)
    out, lse, bad = oracle.sparse_attn(qf, oc, os_, oc.shape[0], remap.reshape(1, B * T, K), kl, sm, dv)
    assert bad == 0
    return out.reshape(B, T, *out.shape[2:]), lse.reshape(B, T, -1)


def _check_topk_rows(got, want, ref_scores, K, what):
    B, T, _ = got.shape
    n = 0
    for b in range(B):
        for t in range(T):
            n += check_selection(got[b, t], want[b, t], lambda ids: ref_scores[b, t][ids], K, what)
    return n


def _run_attn(csa2, q, codes, scales, N, idx, kv_len, sm, dv, mode=0):
    B, T, H, D = q.shape
    K = idx.shape[-1]
    out = torch.empty(B, T, H, dv, device=DEV)
    lse = torch.empty(B, T, H, device=DEV)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = csa2.workspace_for_attn(B, T, H, D, dv, K, device=DEV)
    csa2.csa2_sparse_attn_fp4(mode, q, codes, scales, N, idx, out, sm, kv_len=kv_len, lse=lse, err_flag=flag,
                              workspace=ws)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    return out, lse


@pytest.mark.parametrize("wl", [gen.TINY_FULL_DECODE, gen.FULL_BATCHED_DECODE], ids=["tiny", "batched"])
def test_full_group_decode_chain(csa2, wl):
    """A Full layer (score -> pool -> Top-512 -> attention) followed by 3 Reuse
    layers attending with the same indices over the same KV."""
    w = wl
    B, N, D, dv, H, K = w.B, w.N, w.D, w.dv, w.H, w.K
    kv_len = gen.kv_lengths(w)
    rows = gen.kv_cache_rows(w, device=DEV)
    codes, scales = _gpu_quant_all(csa2, rows, D)
    q_idx, wt, k_idx = gen.indexer_inputs(w)
    kl = kv_len.to(DEV)
    scores = torch.empty(B, 1, N, device=DEV)
    csa2.csa2_index_score(0, q_idx.to(DEV), wt.to(DEV), k_idx.to(DEV), kl, scores)
    pool = torch.empty(B, 1, 2048, dtype=torch.int32, device=DEV)
    csa2.csa2_build_pool(scores, kl, pool)
    idx = torch.empty(B, 1, K, dtype=torch.int32, device=DEV)
    csa2.csa2_topk(0, scores, idx, kv_len=kl)
    torch.cuda.synchronize()

    ref, mag = oracle.index_score(0, _np(q_idx), _idx_dt(w), _np(wt), _np(k_idx), _idx_dt(w), _np(kv_len),
                                  with_mag=True)
    check_scores(scores.cpu().numpy(), ref, mag)
    ref_pool = oracle.build_pool(ref.astype(np.float32), _np(kv_len))
    # n <= 16384 here: the pool covers every valid block, exactly
    for b in range(B):
        assert set(pool[b, 0].cpu().numpy()) - {-1} == set(range((int(kv_len[b]) + 7) // 8))
        assert set(ref_pool[b, 0]) - {-1} == set(range((int(kv_len[b]) + 7) // 8))
    ref_idx = oracle.topk(0, ref.astype(np.float32), _np(kv_len), K=K)
    _check_topk_rows(idx.cpu().numpy(), ref_idx, ref, K, "top-512")

    sm = gen.softmax_scale(D)
    for layer in range(4):                       # Full + 3 Reuse, each with its own Q
        q = gen.attn_query(w, layer=layer)
        mode = 0 if layer == 0 else 2
        if mode == 2:
            before = idx.clone()
            csa2.csa2_topk(2, scores, idx)           # Reuse: no selection
            assert torch.equal(idx, before)
        out, lse = _run_attn(csa2, q.to(DEV), codes, scales, N, idx, kl, sm, dv, mode=mode)
        # parity on the oracle's own selection
        out_o, lse_o = _run_attn(csa2, q.to(DEV), codes, scales, N, torch.from_numpy(ref_idx).to(DEV), kl, sm,
                                 dv, mode=mode)
        r_out, r_lse = _oracle_attn_on_selection(_np(q), rows, codes, scales, N, ref_idx, _np(kv_len), sm, dv)
        check_attn(out_o.cpu().numpy(), r_out)
        check_lse(lse_o.cpu().numpy(), r_lse)
        # the GPU chain's own output where its selection equals the oracle's
        g_idx = idx.cpu().numpy()
        same = np.array([sorted(g_idx[b, 0]) == sorted(ref_idx[b, 0]) for b in range(B)])
        if same.any():
            check_attn(out.cpu().numpy()[same], r_out[same])


def test_reindex_reuse_group_at_1m(csa2):
    """B=8 sequences of 262144 entries: pool from a Full layer's scores, one
    Reindex layer (own q, w) -> Top-512 inside the pool (the unfused chain
    against the oracle, the fused indexer against the chain), then the
    Reindex layer and 3 Reuse layers attend with those indices, each over its
    own FP4 KV."""
    w = gen.REINDEX_REUSE_1M
    B, N, D, dv, H, K, P = w.B, w.N, w.D, w.dv, w.H, w.K, w.P
    kv_len = gen.kv_lengths(w)
    kl = kv_len.to(DEV)
    q0, w0, k_idx = gen.indexer_inputs(w, layer=0, device=DEV)
    q1, w1, _ = gen.indexer_inputs(w, layer=1, device=DEV)
    full = torch.empty(B, 1, N, device=DEV)
    csa2.csa2_index_score(0, q0, w0, k_idx, kl, full)
    pool = torch.empty(B, 1, P, dtype=torch.int32, device=DEV)
    csa2.csa2_build_pool(full, kl, pool)
    rs = torch.empty(B, 1, 8 * P, device=DEV)
    csa2.csa2_index_score(1, q1, w1, k_idx, kl, rs, pool_blocks=pool)
    idx = torch.empty(B, 1, K, dtype=torch.int32, device=DEV)
    csa2.csa2_topk(1, rs, idx, pool_blocks=pool)
    torch.cuda.synchronize()

    # oracle: Full scores, pool (tie band on block maxima), Reindex, Top-512
    ref_full, mag = oracle.index_score(0, _np(q0), 1, _np(w0), _np(k_idx), 1, _np(kv_len), with_mag=True)
    check_scores(full.cpu().numpy(), ref_full, mag, "full scores")
    ref_pool = oracle.build_pool(ref_full.astype(np.float32), _np(kv_len))
    bmax = ref_full.reshape(B, 1, N // 8, 8).max(-1)
    g_pool = pool.cpu().numpy()
    _check_topk_rows(g_pool, ref_pool, bmax, P, "pool")
    # Reindex parity on the ORACLE's pool (so both sides score the same candidates)
    rs_o = torch.empty(B, 1, 8 * P, device=DEV)
    csa2.csa2_index_score(1, q1, w1, k_idx, kl, rs_o, pool_blocks=torch.from_numpy(ref_pool).to(DEV))
    torch.cuda.synchronize()
    ref_rs, rmag = oracle.index_score(1, _np(q1), 1, _np(w1), _np(k_idx), 1, _np(kv_len), pool=ref_pool,
                                      with_mag=True)
    check_scores(rs_o.cpu().numpy(), ref_rs, rmag, "reindex scores")
    ref_idx = oracle.topk(1, ref_rs.astype(np.float32), None, pool=ref_pool, K=K)
    # GPU chain selection: inside its own pool, and equal to the oracle's where the pools agree
    g_idx = idx.cpu().numpy()
    for b in range(B):
        blocks = set(g_pool[b, 0][g_pool[b, 0] >= 0])
        assert all(int(j) // 8 in blocks for j in g_idx[b, 0] if j >= 0)
        assert (g_idx[b, 0] >= 0).all() and len(set(g_idx[b, 0])) == K
    pools_same = np.array([sorted(g_pool[b, 0]) == sorted(ref_pool[b, 0]) for b in range(B)])
    ref_pos_score = {}
    for b in range(B):
        for p in range(P):
            blk = ref_pool[b, 0, p]
            for i in range(8):
                ref_pos_score[(b, 8 * int(blk) + i)] = ref_rs[b, 0, 8 * p + i]
    for b in np.nonzero(pools_same)[0]:
        check_selection(g_idx[b, 0], ref_idx[b, 0], lambda ids: np.array([ref_pos_score[(b, int(j))] for j in ids]),
                        K, "reindex top-512")
    # the fused indexer (the decode step's call; one launch, rows over 8-CTA clusters at this
    # length) scores with the same tiling, so it selects the chain's set row for row
    idx_f = torch.full((B, 1, K), -7, dtype=torch.int32, device=DEV)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    csa2.csa2_index_topk(1, q1, w1, k_idx, kl, idx_f, pool_blocks=pool, err_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    g_f = idx_f.cpu().numpy()
    for b in range(B):
        assert sorted(g_f[b, 0].tolist()) == sorted(g_idx[b, 0].tolist())

    # 4 attention layers over their own KV, all with the Reindex layer's indices
    sm = gen.softmax_scale(D)
    ridx_dev = torch.from_numpy(ref_idx).to(DEV)
    for layer in range(4):
        rows = gen.kv_cache_rows(w, stream=40 + layer, device=DEV)
        codes, scales = _gpu_quant_all(csa2, rows, D)
        q = gen.attn_query(w, layer=layer)
        mode = 1 if layer == 0 else 2
        out, lse = _run_attn(csa2, q.to(DEV), codes, scales, N, ridx_dev, kl, sm, dv, mode=mode)
        r_out, r_lse = _oracle_attn_on_selection(_np(q), rows, codes, scales, N, ref_idx, _np(kv_len), sm, dv)
        check_attn(out.cpu().numpy(), r_out, "layer %d" % layer)
        check_lse(lse.cpu().numpy(), r_lse)
        del rows, codes, scales
        torch.cuda.empty_cache()


def test_prefill_chunk_sampled(csa2):
    """4096 causal queries at 128K context: scores, per-query Top-512 and
    attention for all queries on the GPU; sampled queries vs the oracle."""
    w = gen.PREFILL_CHUNK
    T, N, D, dv, H, K = w.T, w.N, w.D, w.dv, w.H, w.K
    kv_len = gen.kv_lengths(w)
    kl = kv_len.to(DEV)
    rows = gen.kv_cache_rows(w, device=DEV)
    codes, scales = _gpu_quant_all(csa2, rows, D)
    q_idx, wt, k_idx = gen.indexer_inputs(w, device=DEV)
    scores = torch.empty(1, T, N, device=DEV)
    csa2.csa2_index_score(0, q_idx, wt, k_idx, kl, scores)
    idx = torch.empty(1, T, K, dtype=torch.int32, device=DEV)
    csa2.csa2_topk(0, scores, idx, kv_len=kl)
    q = gen.attn_query(w, device=DEV)
    out, lse = _run_attn(csa2, q, codes, scales, N, idx, kl, gen.softmax_scale(D), dv)
    pick = [0, 1, 777, 2048, 4095]
    ref, mag = oracle.index_score(0, _np(q_idx[:, pick]), 1, _np(wt[:, pick]), _np(k_idx), 1, _np(kv_len[pick]),
                                  with_mag=True)
    check_scores(scores[:, pick].cpu().numpy(), ref, mag)
    ref_idx = oracle.topk(0, ref.astype(np.float32), _np(kv_len[pick]), K=K)
    g_idx = idx[:, pick].cpu().numpy()
    _check_topk_rows(g_idx, ref_idx, ref, K, "prefill top-512")
    # attention of the sampled queries on the oracle's selection
    qs = q[:, pick].contiguous()
    out_o, lse_o = _run_attn(csa2, qs, codes, scales, N, torch.from_numpy(ref_idx).to(DEV),
                             kl[pick].contiguous(), gen.softmax_scale(D), dv)
    r_out, r_lse = _oracle_attn_on_selection(_np(qs), rows, codes, scales, N, ref_idx, _np(kv_len[pick]),
                                             gen.softmax_scale(D), dv)
    check_attn(out_o.cpu().numpy(), r_out)
    check_lse(lse_o.cpu().numpy(), r_lse)
    # the full-run outputs of the sampled queries equal the 5-query run where selections agree
    same = [i for i in range(len(pick)) if sorted(g_idx[0, i]) == sorted(ref_idx[0, i])]
    if same:
        check_attn(out[:, pick].cpu().numpy()[:, same], r_out[:, same])


def test_append_and_pool_b16(csa2):
    """Pool for 16 sequences of 65536 entries from GPU Full scores vs the oracle."""
    w = gen.APPEND_POOL
    B, N, P = w.B, w.N, w.P
    kv_len = gen.kv_lengths(w)
    kl = kv_len.to(DEV)
    q_idx, wt, k_idx = gen.indexer_inputs(w, device=DEV)
    scores = torch.empty(B, 1, N, device=DEV)
    csa2.csa2_index_score(0, q_idx, wt, k_idx, kl, scores)
    pool = torch.empty(B, 1, P, dtype=torch.int32, device=DEV)
    csa2.csa2_build_pool(scores, kl, pool)
    torch.cuda.synchronize()
    ref, mag = oracle.index_score(0, _np(q_idx), 1, _np(wt), _np(k_idx), 1, _np(kv_len), with_mag=True)
    check_scores(scores.cpu().numpy(), ref, mag)
    ref_pool = oracle.build_pool(ref.astype(np.float32), _np(kv_len))
    bmax = ref.reshape(B, 1, N // 8, 8).max(-1)
    _check_topk_rows(pool.cpu().numpy(), ref_pool, bmax, P, "pool")
    # invariants: <= 16384 candidates, chosen block maxima dominate (outside the band)
    for b in range(B):
        blk = pool[b, 0].cpu().numpy()
        assert (blk >= 0).sum() * 8 <= 16384


@pytest.mark.parametrize("fused", [True, False])
def test_decoder_step_schedule_runs_and_reuses_indices(csa2, fused):
    """The 20-layer decoder step driver (fused indexer calls, or score + pool
    + Top-K): every Reuse layer's output equals a direct attention call with
    its group's indices, and Reindex selections lie inside the pool."""
    from sparse_attention_fp4_quantize_gb300.decode import DecoderStep, StepShape
    st = DecoderStep(StepShape(B=4, N=3000, fused_indexer=fused), device=DEV)
    w = gen.scaled(gen.FULL_BATCHED_DECODE, B=4, N=3000)
    st.kv_len.copy_(gen.kv_lengths(w).clamp(max=3000).to(DEV))
    for kv in range(st.n_kv):
        rows = gen.kv_cache_rows(w, stream=60 + kv, device=DEV)
        c, s = st.kv_planes(kv)
        csa2.csa2_quantize_kv_fp4(rows, c, s)
    _, _, k_idx = gen.indexer_inputs(w, device=DEV)
    st.k_idx.copy_(k_idx)
    for gi in range(len(st.groups)):
        qi, wi, _ = gen.indexer_inputs(w, layer=gi, device=DEV)
        st.inputs["q_idx"][gi].copy_(qi)
        st.inputs["w_idx"][gi].copy_(wi)
    for layer in range(st.L):
        st.inputs["q"][layer].copy_(gen.attn_query(w, layer=layer, device=DEV))
    st.inputs["new_rows"].copy_(gen.kv_rows(5, 70, st.n_kv * 4, 576, device=DEV))
    st.set_append_slots()
    st.run()
    torch.cuda.synchronize()
    assert int(st.err.item()) == 0
    pool = st.pool.cpu().numpy()
    for gi, layer in enumerate(st.groups):
        idx = st.idx[gi].cpu().numpy()
        assert (idx >= 0).all()
        if gi > 0:
            for b in range(4):
                blocks = set(pool[b, 0][pool[b, 0] >= 0])
                assert all(int(j) // 8 in blocks for j in idx[b, 0])
    for layer in range(st.L):
        gi = max(i for i, l0 in enumerate(st.groups) if l0 <= layer)
        c, s = st.kv_planes(layer)
        out, _ = _run_attn(csa2, st.inputs["q"][layer], c, s, 3000, st.idx[gi], st.kv_len, st.sm_scale, 512,
                           mode=2)
        assert torch.equal(out, st.out[layer])
