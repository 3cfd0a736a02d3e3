"""The quantiser's divide-free rounding, checked exhaustively on the CPU.

The FP4 quantiser forms |x| / s as |x| times an approximate reciprocal of the
group scale s, rounds that product to 12 significant bits (adding half of the
dropped range to the bit pattern, then truncating), and lets a round-to-
nearest-even conversion pick the E2M1 code.  The group scale itself is
amax * fp32(1/6), rounded to 12 bits, then converted to E4M3 with
round-to-nearest-even and saturation.  The claim is that both decisions
equal those of the exact quotients for every bf16 input and every scale, as
long as the reciprocal is within 2^-21 (relative) of 1/s.

The path from the reciprocal to the code is monotone (an fp32 product, the
12-bit rounding, the nearest-code choice), so checking the two ends of the
reciprocal's error interval covers every reciprocal inside it.  This test
restates that arithmetic in NumPy (the CUDA code is not used); the expected
codes and scales come from the oracle's encoders and from the exact rule."""
from __future__ import annotations

import numpy as np
import torch

import oracle


def _round12(v):
    """fp32 -> 12 significant bits: add half of the dropped 12-bit range to
    the bit pattern, then clear it (the quantiser's rounding step)."""
    u = np.asarray(v, np.float32).view(np.uint32)
    return ((u + np.uint32(0x800)) & np.uint32(0xFFFFF000)).view(np.float32)


def _e2m1_code(r):
    """Nearest E2M1 magnitude code of r >= 0, ties to the even code,
    saturating at 6: thresholds are the midpoints of the grid
    {0, .5, 1, 1.5, 2, 3, 4, 6}; at a midpoint the even code wins."""
    r = np.asarray(r, np.float64)
    return ((r > 0.25).astype(int) + (r >= 0.75) + (r > 1.25) + (r >= 1.75) + (r > 2.5) + (r >= 3.5)
            + (r > 5.0))


def _bf16_magnitudes():
    bits = np.arange(0, 0x7F80, dtype=np.uint32)           # +0 .. largest finite bf16
    return (bits << 16).view(np.float32)


def test_code_rule_matches_the_oracle_encoder():
    r = np.concatenate([np.arange(0, 6.5, 0.125), [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, 100.0]])
    assert all(int(_e2m1_code(x)) == oracle.e2m1_encode_mag(float(x)) for x in r)


def test_scale_byte_is_exact_for_every_bf16_amax():
    amax = _bf16_magnitudes()
    sixth = np.float32(1.0) / np.float32(6.0)                # fp32(1/6), rounded once
    v = _round12(amax * sixth)                               # fp32 product, rounded once
    got = torch.from_numpy(np.minimum(v, np.float32(448.0))).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    want = np.array([oracle.e4m3_encode_pos(float(a) / 6.0) for a in amax.astype(np.float64)], np.uint8)
    assert (got == want).all(), "scale differs for %d amax values" % int((got != want).sum())


def test_codes_are_exact_for_every_scale_and_bf16_value_within_the_reciprocal_bound():
    x = _bf16_magnitudes()
    x64 = x.astype(np.float64)
    checked = 0
    for sb in range(1, 0x7F):                                 # every positive finite E4M3 scale
        s = oracle.e4m3_value(sb)
        want = _e2m1_code(x64 / s)
        lo = np.float32(np.nextafter(np.float32((1.0 / s) * (1.0 - 2.0 ** -21)), np.float32(0)))
        hi = np.float32(np.nextafter(np.float32((1.0 / s) * (1.0 + 2.0 ** -21)), np.float32(np.inf)))
        assert lo < np.float32(1.0 / s) < hi
        for inv in (lo, np.float32(1.0 / s), hi):
            with np.errstate(over="ignore"):                  # huge x / tiny s: inf, code 7 both ways
                q = _round12(x * inv)                         # fp32 product, 12-bit rounding
            got = _e2m1_code(q.astype(np.float64))
            bad = np.nonzero(got != want)[0]
            assert bad.size == 0, "scale 0x%02X, reciprocal %r: x=%r gives code %d, exact %d" % (
                sb, float(inv), float(x[bad[0]]), int(got[bad[0]]), int(want[bad[0]]))
            checked += x.size
    assert checked == 126 * 3 * 0x7F80


def test_the_12_bit_rounding_is_what_restores_the_ties():
    """Without the 12-bit step (or with truncation instead of rounding) a
    reciprocal 2^-21 off moves exact midpoints and their codes: the check
    above is not vacuous."""
    x = _bf16_magnitudes()
    x64 = x.astype(np.float64)

    def wrong_codes(step):
        n = 0
        for sb in range(1, 0x7F):
            s = oracle.e4m3_value(sb)
            want = _e2m1_code(x64 / s)
            for inv in (np.float32((1.0 / s) * (1 - 2.0 ** -21)), np.float32((1.0 / s) * (1 + 2.0 ** -21))):
                with np.errstate(over="ignore"):
                    n += int((_e2m1_code(step(x * inv).astype(np.float64)) != want).sum())
        return n

    def truncate12(v):
        return (np.asarray(v, np.float32).view(np.uint32) & np.uint32(0xFFFFF000)).view(np.float32)

    assert wrong_codes(lambda v: np.asarray(v, np.float32)) > 0
    assert wrong_codes(truncate12) > 0
    assert wrong_codes(_round12) == 0

