"""The tensor-core attention's f16 operands, checked on the CPU.

The attention feeds its MMAs with f16 operands:
  * each dequantised cache value is an E2M1 magnitude (at most 2 significant
    bits) times an E4M3 scale (at most 4), so it has at most 6 significant
    bits and lies in [2^-10, 2688]: every one is an exact f16 number;
  * each query row is multiplied by 2^sh, sh = 14 - floor(log2 max|q|)
    (clamped to [-60, 60]), so its largest magnitude lands in [2^14, 2^15),
    then rounded to f16.  A bf16 value has 8 significant bits, so the
    conversion is exact down to 2^-31 of the row's largest value; below
    that, f16 subnormals round it with an error under 2^-39 of the largest.
    The clamp bounds the supported range: the row's largest |q| must be
    below 2^76 (from there on the scaled value overflows f16); for rows
    whose largest |q| is below 2^-46 the scale stops at 2^60, and values
    below 2^-77 round (absolute error at most 2^-85).
This restates that arithmetic in NumPy; the CUDA code is not used."""
from __future__ import annotations

import numpy as np

import oracle


def test_every_dequantised_value_is_an_exact_f16():
    vals = np.array([oracle.e2m1_value(c) * oracle.e4m3_value(s) for c in range(16) for s in range(0x7F)]
                    + [oracle.e2m1_value(c) * oracle.e4m3_value(s | 0x80) for c in range(16) for s in range(0x7F)])
    assert (vals.astype(np.float16).astype(np.float64) == vals).all()
    nz = np.abs(vals[vals != 0])
    assert nz.min() == 2.0 ** -10 and nz.max() == 2688.0


def test_every_e4m3_window_value_is_an_exact_f16():
    vals = np.array([oracle.e4m3_value(b) for b in range(256) if (b & 0x7F) != 0x7F])
    assert (vals.astype(np.float16).astype(np.float64) == vals).all()


def _bf16_positive():
    bits = np.arange(1, 0x7F80, dtype=np.uint32)
    return (bits << 16).view(np.float32).astype(np.float64)


def _scaled_f16(v, mx):
    e2 = int(np.floor(np.log2(mx)))
    sh = min(60, max(-60, 14 - e2))
    s = v * 2.0 ** sh
    with np.errstate(over="ignore"):
        return s, s.astype(np.float16).astype(np.float64), sh


def test_query_scaling_is_exact_within_2_31_of_the_row_maximum():
    v_all = _bf16_positive()
    # row maxima: both ends of every binade the clamp leaves unaffected
    maxima = [2.0 ** e * m for e in range(-46, 75) for m in (1.0, 1.9921875)]
    for mx in maxima:
        v = v_all[v_all <= mx]
        s, f, sh = _scaled_f16(v, mx)
        assert 2.0 ** 14 <= mx * 2.0 ** sh < 2.0 ** 15
        exact = v >= mx * 2.0 ** -31
        assert (f[exact] == s[exact]).all(), mx
        assert (np.abs(f - s) / 2.0 ** sh <= mx * 2.0 ** -39).all(), mx


def test_query_rows_at_the_clamp():
    for mx in (2.0 ** 75, 2.0 ** 75 * 1.9921875):             # the largest bf16 values below 2^76
        v = _bf16_positive()
        v = v[v <= mx]
        s, f, _ = _scaled_f16(v, mx)
        assert np.isfinite(f).all()
        exact = v >= mx * 2.0 ** -31
        assert (f[exact] == s[exact]).all()
    _, f, _ = _scaled_f16(np.array([2.0 ** 76]), 2.0 ** 76)
    assert np.isinf(f).all()                                    # the documented upper limit


def test_tiny_rows_round_only_below_2_77():
    v = _bf16_positive()
    v = v[v <= 2.0 ** -50]
    s, f, sh = _scaled_f16(v, 2.0 ** -50)
    assert sh == 60
    assert (f[v >= 2.0 ** -77] == s[v >= 2.0 ** -77]).all()
    assert (np.abs(f - s) * 2.0 ** -60 <= 2.0 ** -85).all()

