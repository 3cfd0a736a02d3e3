"""Pins of the oracle's RoPE (the fused append path: RoPE, bf16, then the FP4
quantiser).  READING (the pages fix no layout): interleaved pairs (2i, 2i+1)
of the last rope_dim channels, a caller-supplied fp32 (cos, sin) table, fp32
products and sums without fused multiply-add, bf16 round to nearest even."""
import numpy as np
import torch

import gen
import oracle


def _bits(x):
    return gen.bf16_bits(torch.as_tensor(x, dtype=torch.float32)).numpy().view(np.uint16)


def _vals(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _table(cs_pairs):
    return np.asarray(cs_pairs, np.float32).reshape(1, -1, 2)


def test_identity_rotation_is_exact():
    rng = np.random.default_rng(1)
    x = _bits(rng.standard_normal((50, 96)) * 10)
    out = oracle.rope_bf16(x, np.zeros(50, np.int32), _table([[1.0, 0.0]] * 32), rope_dim=64)
    assert (out == x).all()


def test_quarter_turn_maps_a_b_to_minus_b_a():
    rng = np.random.default_rng(2)
    x = _bits(rng.standard_normal((20, 64)) * 3)
    out = oracle.rope_bf16(x, np.zeros(20, np.int32), _table([[0.0, 1.0]] * 32), rope_dim=64)
    a, b = _vals(x[:, 0::2]), _vals(x[:, 1::2])
    ra, rb = _vals(out[:, 0::2]), _vals(out[:, 1::2])
    assert (ra == -b).all() and (rb == a).all()


def test_unit_vectors_give_the_table_rounded_to_bf16():
    """(1, 0) -> (c, s) and (0, 1) -> (-s, c), each rounded once to bf16: fixes
    which product carries the sine and its sign."""
    ang = np.linspace(0.1, 3.0, 32)
    tab = _table(np.stack([np.cos(ang), np.sin(ang)], -1))
    one, zero = _bits(1.0)[()], _bits(0.0)[()]
    x = np.array([[one, zero] * 32, [zero, one] * 32], np.uint16)
    out = oracle.rope_bf16(x, np.zeros(2, np.int32), tab, rope_dim=64)
    c, s = tab[0, :, 0], tab[0, :, 1]
    assert (out[0, 0::2] == _bits(c)).all() and (out[0, 1::2] == _bits(s)).all()
    assert (out[1, 0::2] == _bits(-s)).all() and (out[1, 1::2] == _bits(c)).all()


def test_equal_cos_and_sin_cancel_exactly_without_fma():
    """With cos = sin (the same fp32 value) and a pair (a, a), the two products
    of the first output are the same rounded fp32 number, so it is exactly +0;
    the second is twice that product.  A fused multiply-add would leave the
    product's rounding error in the first output instead of 0."""
    rng = np.random.default_rng(8)
    a = _bits(rng.standard_normal(4 * 32) * 5).reshape(4, 32)
    x = np.stack([a, a], -1).reshape(4, 64)
    c = np.float32(np.sqrt(0.5))
    out = oracle.rope_bf16(x, np.zeros(4, np.int32), _table([[c, c]] * 32), rope_dim=64)
    prod = _vals(a) * c                                   # fp32 product, rounded once
    assert (out[:, 0::2] == 0).all()                      # +0 bits
    assert (out[:, 1::2] == _bits(prod + prod)).all()
    assert (_vals(a).astype(np.float64) * float(c) != prod).any()   # the products are inexact


def test_channels_before_the_rope_range_pass_through_and_positions_select_rows():
    rng = np.random.default_rng(3)
    x = _bits(rng.standard_normal((6, 576)))
    tab = gen.rope_table(10).numpy()
    pos = np.array([0, 9, 3, 3, 7, 1], np.int32)
    out = oracle.rope_bf16(x, pos, tab)
    assert (out[:, :512] == x[:, :512]).all()
    assert (out[0] == x[0]).all()                      # position 0: cos 1, sin 0
    assert (out[2] == out[3]).all() == (x[2] == x[3]).all()
    for r in range(6):   # each row equals its own single-row rotation
        assert (oracle.rope_bf16(x[r:r + 1], pos[r:r + 1], tab) == out[r]).all()


def test_rotation_preserves_pair_norms_within_bf16_rounding():
    rng = np.random.default_rng(4)
    x = _bits(rng.standard_normal((200, 64)) * 5)
    tab = gen.rope_table(4096).numpy()
    pos = rng.integers(0, 4096, 200).astype(np.int32)
    out = oracle.rope_bf16(x, pos, tab)
    n0 = np.hypot(_vals(x[:, 0::2]).astype(np.float64), _vals(x[:, 1::2]))
    n1 = np.hypot(_vals(out[:, 0::2]).astype(np.float64), _vals(out[:, 1::2]))
    assert (np.abs(n1 - n0) <= 2 ** -7 * n0 + 1e-30).all()


def test_composition_of_rotations_matches_the_summed_angle():
    rng = np.random.default_rng(5)
    x = _bits(rng.standard_normal((100, 64)))
    tab = gen.rope_table(200).numpy()
    once = oracle.rope_bf16(x, np.full(100, 150, np.int32), tab)
    twice = oracle.rope_bf16(oracle.rope_bf16(x, np.full(100, 100, np.int32), tab), np.full(100, 50, np.int32), tab)
    d = np.abs(_vals(once).astype(np.float64) - _vals(twice))
    assert (d <= 2 ** -6 * (np.abs(_vals(once)) + 1.0)).all()


def test_matches_the_torch_input_generator_bit_for_bit():
    """gen.rope_interleaved (torch, separate fp32 tensor ops, no FMA) with the
    same fp32 table is an independent implementation of the same arithmetic."""
    rng = np.random.default_rng(6)
    xf = torch.from_numpy(rng.standard_normal((64, 576)).astype(np.float32))
    xb = gen.bf16_bits(xf)
    pos = torch.from_numpy(rng.integers(0, 5000, 64).astype(np.int32))
    tab = gen.rope_table(5000)
    out = oracle.rope_bf16(xb.numpy().view(np.uint16), pos.numpy(), tab.numpy())
    xv = xb.view(torch.bfloat16).to(torch.float32)
    r = xv[:, 512:].reshape(64, 32, 2)
    c, s = tab[pos.long(), :, 0], tab[pos.long(), :, 1]
    a, b = r[..., 0], r[..., 1]
    rot = torch.stack((a * c - b * s, a * s + b * c), -1).reshape(64, 64)
    ref = torch.cat((xv[:, :512], rot), -1).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (out == ref).all()


def test_rope_then_quantise_is_the_quantiser_of_the_rotated_rows():
    rng = np.random.default_rng(7)
    x = _bits(rng.standard_normal((32, 576)))
    tab = gen.rope_table(64).numpy()
    pos = rng.integers(0, 64, 32).astype(np.int32)
    c1, s1 = oracle.rope_quantize_kv_fp4(x, pos, tab)
    c2, s2 = oracle.quantize_kv_fp4(oracle.rope_bf16(x, pos, tab))
    assert (c1 == c2).all() and (s1 == s2).all()
    # RoPE leaves the 512 latent channels' codes unchanged
    c0, s0 = oracle.quantize_kv_fp4(x)
    assert (c1[:, :256] == c0[:, :256]).all() and (s1[:, :32] == s0[:, :32]).all()
