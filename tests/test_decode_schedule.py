"""Host logic of the decode step (CPU only): the layer schedule is the pages'
grouping ("DeepSeek-V4.1-Flash：把 KV Cache 压缩到极限的百万上下文 MoE", CSA2
section: 20 layers in groups of 4, the first 1 Full + 3 Reuse, the others
1 Reindex + 3 Reuse), and one step issues the library calls in model order,
with Reuse layers consuming their group's index buffer and every layer its
own FP4 KV.  The library calls are replaced by recorders, so no kernel runs;
the recorded launches must equal the count the benchmark reports."""
from __future__ import annotations

import pytest

import sparse_attention_fp4_quantize_gb300 as csa2
import sparse_attention_fp4_quantize_gb300.decode as dec

CALLS = ["csa2_quantize_kv_fp4", "csa2_index_topk", "csa2_index_score", "csa2_build_pool", "csa2_topk",
         "csa2_sparse_attn_fp4", "csa2_sparse_attn_fp4_prefetch"]
ATTN = ("csa2_sparse_attn_fp4", "csa2_sparse_attn_fp4_prefetch")


def test_schedule_is_the_pages_grouping():
    s = dec.DECODER_SCHEDULE
    assert len(s) == 20
    groups = [s[i:i + 4] for i in range(0, 20, 4)]
    assert groups[0] == ("full", "reuse", "reuse", "reuse")
    assert groups[1:] == [("reindex", "reuse", "reuse", "reuse")] * 4


def _record(monkeypatch):
    calls = []
    for name in CALLS:
        monkeypatch.setattr(dec, name, lambda *a, _n=name, **kw: calls.append((_n, a, kw)))
    return calls


def _launches(calls):
    """Calls that launch a kernel: every call except the Reuse-mode no-ops."""
    return [c for c in calls if not (c[0] in ("csa2_topk", "csa2_index_topk", "csa2_index_score")
                                     and c[1][0] == csa2.MODE_REUSE)]


@pytest.mark.parametrize("fused", [True, False])
def test_one_step_issues_the_calls_in_model_order(monkeypatch, fused):
    calls = _record(monkeypatch)
    st = dec.DecoderStep(dec.StepShape(B=2, N=64, fused_indexer=fused), device="cpu")
    st.run()
    assert calls[0][0] == "csa2_quantize_kv_fp4"
    attn = [c for c in calls if c[0] in ATTN]
    assert [c[1][0] for c in attn] == [{"full": csa2.MODE_FULL, "reindex": csa2.MODE_REINDEX,
                                         "reuse": csa2.MODE_REUSE}[m] for m in dec.DECODER_SCHEDULE]
    # every layer attends over its own KV planes; Reuse layers use their group's indices
    code_ptrs = [c[1][2].data_ptr() for c in attn]
    assert len(set(code_ptrs)) == 20
    idx_ptrs = [c[1][5].data_ptr() for c in attn]
    for layer in range(20):
        assert idx_ptrs[layer] == idx_ptrs[layer - layer % 4]
    assert len(set(idx_ptrs)) == 5
    # a layer followed by a Reuse layer hints that layer's planes into L2; the group's last does not
    for layer in range(20):
        nxt_reuse = layer + 1 < 20 and dec.DECODER_SCHEDULE[layer + 1] == "reuse"
        assert attn[layer][0] == ("csa2_sparse_attn_fp4_prefetch" if nxt_reuse else "csa2_sparse_attn_fp4")
        if nxt_reuse:
            assert attn[layer][2]["next_codes"].data_ptr() == code_ptrs[layer + 1]
            assert attn[layer][2]["next_scales"].data_ptr() == attn[layer + 1][1][3].data_ptr()
    # each group's indexer runs before the group's first attention and after the previous layer's
    order = [c[0] for c in calls]
    first_attn = [i for i, c in enumerate(calls) if c[0] in ATTN]
    sel = "csa2_index_topk" if fused else "csa2_topk"
    for g in range(5):
        i_attn = first_attn[4 * g]
        prev = first_attn[4 * g - 1] if g else 0
        assert sel in order[prev:i_attn]
    # the pool: written by the Full layer only, read by the Reindex layers
    if fused:
        idx_calls = [c for c in calls if c[0] == "csa2_index_topk"]
        assert [c[1][0] for c in idx_calls] == [csa2.MODE_FULL] + [csa2.MODE_REINDEX] * 4
        assert idx_calls[0][2]["pool_out"] is st.pool
        assert all(c[2]["pool_blocks"] is st.pool for c in idx_calls[1:])
    else:
        assert order.count("csa2_build_pool") == 1
    assert len(_launches(calls)) == st.launches_per_step() == (26 if fused else 32)
