"""The benchmarked decode step as a whole against the oracle.

The step is built exactly as the benchmark builds it (32 sequences of 8192 to
16384 entries, capacity 16384, 576-channel FP4 KV per layer, FP8 indexer,
fused score -> pool -> Top-512 calls, 20 layers in the decoder's schedule:
1 Full + 3 Reuse, then 4 x (1 Reindex + 3 Reuse), the step's new KV row of
every layer appended into its slot) and run once.  For sampled sequences the
oracle then runs the same chain on its own: quantise every layer's KV rows
(the appended row in its slot), Full scores, the 2048-block pool, Top-512,
the four Reindex groups inside the pool, and the 20 attentions with each
group's selection.  Compared: the FP4 planes bit for bit, every group's
selection within the tie band, and every layer's output and log-sum-exp
within the attention tolerance on the oracle's selection.  Marked gpu."""
import numpy as np
import pytest
import torch

import gen
import oracle
from helpers import check_attn, check_lse, check_selection

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def step():
    import bench
    import sparse_attention_fp4_quantize_gb300  # noqa: F401  (fails loudly without libcsa2.so)
    from sparse_attention_fp4_quantize_gb300.decode import DecoderStep, StepShape
    st = DecoderStep(StepShape(B=bench.B, N=bench.NCAP, D=bench.D, dv=bench.DV, H=bench.H, K=bench.K, P=bench.P),
                     device=DEV)
    bench._fill_instance(st, seed=1)
    st.run()
    torch.cuda.synchronize()
    yield st
    del st
    torch.cuda.empty_cache()


def _samples(st):
    kl = st.kv_len.cpu().numpy()
    return sorted({0, int(np.argmax(kl)), int(np.argmin(kl)), st.shape.B - 1})


def test_step_matches_oracle_chain(step):
    import bench
    import sparse_attention_fp4_quantize_gb300 as csa2
    st = step
    s = st.shape
    B, N, D, dv, K, P = s.B, s.N, s.D, s.dv, s.K, s.P
    seed = 1
    assert int(st.err.item()) == 0
    sm = st.sm_scale
    kv_len = st.kv_len.cpu().numpy().astype(np.int32)
    k_all = st.k_idx.cpu().numpy()
    new_rows = st.inputs["new_rows"].cpu().numpy().view(np.uint16)
    groups = st.groups                                   # first layer of each group
    for b in _samples(st):
        n = int(kv_len[b])
        kvl = np.array([n], np.int32)
        kb = k_all[b:b + 1]
        # ---- the indexer chain: Full scores -> pool -> Top-512, then Reindex groups in the pool
        ref_idx, score_of = [], []
        pool = None
        for gi, layer in enumerate(groups):
            qi = st.inputs["q_idx"][gi][b:b + 1].cpu().numpy()
            wi = st.inputs["w_idx"][gi][b:b + 1].cpu().numpy()
            full = oracle.index_score(oracle.FULL, qi, oracle.FP8_E4M3, wi, kb, oracle.FP8_E4M3, kvl)
            f32 = full.astype(np.float32)
            if s.schedule[layer] == "full":
                if layer == 0:
                    pool = oracle.build_pool(f32, kvl, P=P)
                    assert set(pool[0, 0][pool[0, 0] >= 0].tolist()) == set(range((n + 7) // 8))
                idx_r = oracle.topk(oracle.FULL, f32, kvl, K=K)
            else:
                rs = oracle.index_score(oracle.REINDEX, qi, oracle.FP8_E4M3, wi, kb, oracle.FP8_E4M3, kvl, pool=pool)
                idx_r = oracle.topk(oracle.REINDEX, rs.astype(np.float32), None, pool=pool, K=K)
            ref_idx.append(idx_r)
            score_of.append(full[0, 0])
            got = st.idx[gi][b, 0].cpu().numpy()
            check_selection(got, idx_r[0, 0], lambda ids, f=full[0, 0]: f[ids], K, "group %d seq %d" % (gi, b))
        # ---- every layer's FP4 planes (with the appended row) and attention
        gi = -1
        for layer, mode in enumerate(s.schedule):
            if mode != "reuse":
                gi += 1
            rows = gen.kv_rows(seed, 100 + layer, B * N, D, rms=True, device=DEV)[b * N:(b + 1) * N].cpu().numpy()
            rows = rows.view(np.uint16).copy()
            rows[n - 1] = new_rows[layer * B + b]        # the step's append: slot kv_len - 1
            oc, os_ = oracle.quantize_kv_fp4(rows)
            c, sc = st.kv_planes(layer)
            assert np.array_equal(c[b * N:(b + 1) * N].cpu().numpy(), oc), "layer %d seq %d codes" % (layer, b)
            assert np.array_equal(sc[b * N:(b + 1) * N].cpu().numpy(), os_), "layer %d seq %d scales" % (layer, b)
            q = st.inputs["q"][layer][b:b + 1].cpu().numpy().view(np.uint16)
            o_ref, lse_ref, bad = oracle.sparse_attn(q, oc, os_, N, ref_idx[gi], kvl, sm, dv)
            assert bad == 0
            got_idx = st.idx[gi][b, 0].cpu().numpy()
            if set(got_idx.tolist()) == set(ref_idx[gi][0, 0].tolist()):
                o_gpu = st.out[layer][b:b + 1].cpu().numpy()
                l_gpu = st.lse[layer][b:b + 1].cpu().numpy()
            else:   # the selections differ inside the tie band: the same kernel on the oracle's set
                o_t = torch.empty(1, 1, s.H, dv, device=DEV)
                l_t = torch.empty(1, 1, s.H, device=DEV)
                csa2.csa2_sparse_attn_fp4(csa2.MODE_REUSE, st.inputs["q"][layer][b:b + 1].contiguous(),
                                          c[b * N:(b + 1) * N], sc[b * N:(b + 1) * N], N,
                                          torch.from_numpy(ref_idx[gi]).to(DEV), o_t, sm,
                                          kv_len=st.kv_len[b:b + 1].contiguous(), lse=l_t)
                torch.cuda.synchronize()
                o_gpu, l_gpu = o_t.cpu().numpy(), l_t.cpu().numpy()
            check_attn(o_gpu, o_ref, "layer %d seq %d" % (layer, b))
            check_lse(l_gpu, lse_ref, "layer %d seq %d lse" % (layer, b))
    assert bench.LAYERS == len(s.schedule)
