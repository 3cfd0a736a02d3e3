"""csa2_rope_quantize_kv_fp4 (RoPE fused ahead of the FP4 quantiser) against
the oracle's RoPE + quantiser: codes and scale bytes bit-exact."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gen
import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def csa2():
    import sparse_attention_fp4_quantize_gb300 as lib
    return lib


def _run(csa2, x_bits, pos, tab, dst_slot=None, n_slots=None, flag=None):
    R, D = x_bits.shape
    S = R if n_slots is None else n_slots
    codes = torch.full((S, D // 2), 0xAB, dtype=torch.uint8, device=DEV)
    scales = torch.full((S, D // 16), 0xCD, dtype=torch.uint8, device=DEV)
    csa2.csa2_rope_quantize_kv_fp4(x_bits.to(DEV), pos.to(DEV), tab.to(DEV), codes, scales,
                                   dst_slot=None if dst_slot is None else dst_slot.to(DEV), err_flag=flag)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


@pytest.mark.parametrize("R,D,n_pos", [(5000, 576, 65536), (33, 128, 100), (1, 576, 1), (4097, 576, 300)])
def test_rope_quantize_bit_exact(csa2, R, D, n_pos):
    x = gen.kv_rows(31, R % 97, R, D, rms=(D == 576))
    pos = torch.randint(0, n_pos, (R,), generator=torch.Generator().manual_seed(R), dtype=torch.int32)
    tab = gen.rope_table(n_pos)
    got_c, got_s = _run(csa2, x, pos, tab)
    want_c, want_s = oracle.rope_quantize_kv_fp4(gen.as_numpy(x).view(np.uint16), pos.numpy(), tab.numpy())
    assert (got_c == want_c).all(), "codes differ in %d bytes" % int((got_c != want_c).sum())
    assert (got_s == want_s).all(), "scales differ in %d bytes" % int((got_s != want_s).sum())


def test_rope_quantize_equals_quantize_of_oracle_rope_rows(csa2):
    R = 2048
    x = gen.kv_rows(32, 1, R, 576)
    pos = torch.randint(0, 131072, (R,), generator=torch.Generator().manual_seed(9), dtype=torch.int32)
    tab = gen.rope_table(131072)
    got = _run(csa2, x, pos, tab)
    rot = torch.from_numpy(oracle.rope_bf16(gen.as_numpy(x).view(np.uint16), pos.numpy(), tab.numpy()).view(np.int16))
    codes = torch.empty(R, 288, dtype=torch.uint8, device=DEV)
    scales = torch.empty(R, 36, dtype=torch.uint8, device=DEV)
    csa2.csa2_quantize_kv_fp4(rot.to(DEV), codes, scales)
    torch.cuda.synchronize()
    assert (got[0] == codes.cpu().numpy()).all() and (got[1] == scales.cpu().numpy()).all()


def test_rope_quantize_scatter_and_bad_positions(csa2):
    R, S = 64, 200
    x = gen.kv_rows(33, 2, R, 576)
    tab = gen.rope_table(50)
    pos = torch.randint(0, 50, (R,), generator=torch.Generator().manual_seed(2), dtype=torch.int32)
    slot = torch.randperm(S, generator=torch.Generator().manual_seed(3))[:R].to(torch.int64)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    got_c, got_s = _run(csa2, x, pos, tab, dst_slot=slot, n_slots=S, flag=flag)
    assert int(flag.item()) == 0
    want_c, want_s = oracle.rope_quantize_kv_fp4(gen.as_numpy(x).view(np.uint16), pos.numpy(), tab.numpy(),
                                                 dst_slot=slot.numpy(), n_slots=S)
    sel = slot.numpy()
    assert (got_c[sel] == want_c[sel]).all() and (got_s[sel] == want_s[sel]).all()
    untouched = np.setdiff1d(np.arange(S), sel)
    assert (got_c[untouched] == 0xAB).all() and (got_s[untouched] == 0xCD).all()
    bad = pos.clone()
    bad[5] = 50
    bad[9] = -1
    got_c, got_s = _run(csa2, x, bad, tab, flag=flag)
    assert int(flag.item()) & csa2.FLAG_BAD_INDEX
    want_c, want_s = oracle.quantize_kv_fp4(gen.as_numpy(x).view(np.uint16))
    for r in (5, 9):   # latent groups still written, the rotated groups left untouched
        assert (got_c[r, :256] == want_c[r, :256]).all() and (got_s[r, :32] == want_s[r, :32]).all()
        assert (got_c[r, 256:] == 0xAB).all() and (got_s[r, 32:] == 0xCD).all()
