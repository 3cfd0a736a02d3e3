"""Pins of the oracle's element formats and FP4 quantisation (CPU only).

Each check ties the oracle to something other than itself: the golden
closed-form values derived by hand from the format definitions, torch's
float8_e4m3fn cast and decode (a library routine), or brute-force nearest
search over the value grids.
"""
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

E2M1_MAG = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for ln in f:
            ln = ln.strip()
            if ln and not ln.startswith("#"):
                yield ln


def _bf16_bits(vals):
    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------- formats
def test_golden_format_values(orc):
    seen = set()
    for ln in _golden_lines("formats.txt"):
        f = ln.split()
        if f[0] == "e4m3":
            v = orc.e4m3_value(int(f[1], 16))
            assert v == float(f[2]) and math.copysign(1, v) == math.copysign(1, float(f[2]))
        elif f[0] == "e2m1":
            v = orc.e2m1_value(int(f[1], 16))
            assert v == float(f[2]) and math.copysign(1, v) == math.copysign(1, float(f[2]))
        elif f[0] == "entry_bytes":
            D = int(f[1])
            codes, scales = orc.quantize_kv_fp4(np.zeros((1, D), np.uint16))
            assert codes.nbytes + scales.nbytes == int(f[2])
        elif f[0] == "pool":
            assert int(f[1]) * int(f[2]) == int(f[3])
        seen.add(f[0])
    assert {"e4m3", "e2m1", "entry_bytes", "pool"} <= seen


def test_e4m3_decode_matches_torch_all_256(orc):
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([orc.e4m3_value(b) for b in range(256)])
    nan_ref, nan_got = np.isnan(ref), np.isnan(got)
    assert (nan_ref == nan_got).all() and nan_ref.sum() == 2      # 0x7F, 0xFF
    assert (got[~nan_got] == ref[~nan_ref]).all()
    assert (np.signbit(got[~nan_got]) == np.signbit(ref[~nan_ref])).all()


def test_e2m1_decode_closed_form(orc):
    for c in range(16):
        mag = E2M1_MAG[c & 7]
        v = orc.e2m1_value(c)
        assert abs(v) == mag and (math.copysign(1, v) < 0) == bool(c & 8)


def _e4m3_positive_grid():
    vals = [(b, float(torch.tensor([b], dtype=torch.uint8).view(torch.float8_e4m3fn).float()))
            for b in range(0, 0x7F)]
    return vals  # bytes 0x00..0x7E with values 0 .. 448, increasing


def _brute_e4m3(a, grid):
    """Nearest grid value by exhaustive search, ties to the even byte,
    saturating above the grid."""
    best = None
    for b, v in grid:
        d = abs(a - v)
        if best is None or d < best[0] or (d == best[0] and b % 2 == 0):
            best = (d, b)
    return best[1]


def test_e4m3_encode_brute_force(orc):
    grid = _e4m3_positive_grid()
    vals = [v for _, v in grid]
    cases = []
    for i in range(len(vals) - 1):                     # every value and midpoint
        cases += [vals[i], (vals[i] + vals[i + 1]) / 2,
                  vals[i] + (vals[i + 1] - vals[i]) * 0.49, vals[i] + (vals[i + 1] - vals[i]) * 0.51]
    rng = np.random.default_rng(5)
    cases += list(np.exp(rng.uniform(math.log(1e-5), math.log(500.0), 3000)))
    cases += [448.0, 460.0, 463.99, 464.0, 1e4, 2.0 ** -10, 2.0 ** -11, 0.0]
    for a in cases:
        got = orc.e4m3_encode_pos(a)
        want = _brute_e4m3(a, grid) if a < 448.0 else 0x7E
        assert got == want, (a, hex(got), hex(want))


def test_e4m3_encode_matches_torch_cast(orc):
    rng = np.random.default_rng(6)
    a = np.concatenate([np.exp(rng.uniform(math.log(1e-4), math.log(460.0), 20000)),
                        rng.uniform(0, 1e-2, 2000)]).astype(np.float32)
    ref = torch.from_numpy(a).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_encode_pos(float(x)) for x in a], np.uint8)
    assert (got == ref).all()


def _brute_e2m1(r):
    best = None
    for c, v in enumerate(E2M1_MAG):
        d = abs(r - v)
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
            best = (d, c)
    return best[1]


def test_e2m1_encode_brute_force(orc):
    cases = []
    for i in range(7):
        lo, hi = E2M1_MAG[i], E2M1_MAG[i + 1]
        cases += [lo, (lo + hi) / 2, lo + (hi - lo) * 0.3, lo + (hi - lo) * 0.7,
                  np.nextafter((lo + hi) / 2, 0), np.nextafter((lo + hi) / 2, 10)]
    cases += list(np.random.default_rng(7).uniform(0, 6, 5000))
    for r in cases:
        assert orc.e2m1_encode_mag(r) == _brute_e2m1(r), r
    for r in [6.0, 6.0001, 7.5, 1e9]:
        assert orc.e2m1_encode_mag(r) == 7


# ---------------------------------------------------------------- quantise
def test_quantize_golden_groups(orc):
    n = 0
    for ln in _golden_lines("fp4_groups.txt"):
        name, xs, sb, cs = [p.strip() for p in ln.split(";")]
        x = [float(v) for v in xs.split()]
        bits = _bf16_bits(x)
        assert (torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
                == np.array(x, np.float32)).all(), name + ": value not bf16-exact"
        codes, scales = orc.quantize_kv_fp4(bits.reshape(1, 16))
        want = [int(c, 16) for c in cs.split()]
        packed = [want[2 * i] | (want[2 * i + 1] << 4) for i in range(8)]
        assert scales[0, 0] == int(sb, 16), name
        assert list(codes[0]) == packed, name
        n += 1
    assert n >= 8


def _rows(seed, R, D, scale=1.0, outliers=True):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(R, D, generator=g) * scale
    if outliers:
        x = torch.where(torch.rand(R, D, generator=g) < 0.01, x * 8, x)
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_quantize_brute_force_per_group(orc):
    """Scale byte = nearest E4M3 to amax/6 and each code = nearest E2M1
    magnitude of |x|/s, both by exhaustive search."""
    grid = _e4m3_positive_grid()
    bits = np.concatenate([_rows(1, 24, 64), _rows(2, 8, 64, scale=1e-3), _rows(3, 8, 64, scale=300.0)])
    codes, scales = orc.quantize_kv_fp4(bits)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    for r in range(x.shape[0]):
        for g in range(4):
            grp = x[r, 16 * g:16 * g + 16]
            amax = np.abs(grp).max()
            sb = _brute_e4m3(amax / 6.0, grid) if amax / 6.0 < 448 else 0x7E
            assert scales[r, g] == sb
            s = dict(grid)[sb]
            for c in range(16):
                ch = 16 * g + c
                code = (codes[r, ch // 2] >> (4 * (ch & 1))) & 0xF
                mag = 0 if s == 0 else (_brute_e2m1(abs(grp[c]) / s) if abs(grp[c]) / s < 6 else 7)
                sign = 8 if np.signbit(grp[c]) else 0
                assert code == (sign | mag), (r, ch, grp[c], s)


def test_quantize_one_hot_and_equal_groups(orc):
    # one-hot: [v, 0...]: v/s in (5, 6.x] -> code 7 unless the scale rounds to 0
    for v in [1.0, -2.5, 0.3, 100.0, -1e-2]:
        bits = _bf16_bits([v] + [0.0] * 15)
        codes, scales = orc.quantize_kv_fp4(bits.reshape(1, 16))
        assert (codes[0, 0] & 0x7) == 7
        assert (codes[0, 0] & 0x8) == (8 if v < 0 else 0)
        assert (codes[0, 1:] == 0).all()
    # all-equal groups with amax = 6 s exactly: every code is +-6 and dequant is exact
    for s in [0.5, 1.25, 2.0 ** -9, 448.0, 0.171875]:
        v = 6 * s
        bits = _bf16_bits([v, -v] * 8)
        codes, scales = orc.quantize_kv_fp4(bits.reshape(1, 16))
        deq = orc.dequant_fp4(codes, scales)
        assert (deq[0] == np.array([v, -v] * 8)).all()


def test_dequant_error_bound(orc):
    bits = _rows(11, 64, 576)
    codes, scales = orc.quantize_kv_fp4(bits)
    deq = orc.dequant_fp4(codes, scales)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    s = np.array([[orc.e4m3_value(b) for b in row] for row in scales]).repeat(16, axis=1)
    r = np.abs(x) / np.where(s > 0, s, 1)
    # half of the local grid step: 0.25 below 2, 0.5 in [2,4), 1 in [4,6]
    half = np.where(r < 2, 0.25, np.where(r < 4, 0.5, 1.0)) * s
    sat = np.maximum(np.abs(x) - 6 * s, 0)
    assert (np.abs(deq - x) <= np.maximum(half, sat) + 0 * s).all()
    # groups that contain a +-6 code are reproduced by re-quantising the dequantised values
    deq_bits = torch.from_numpy(deq).float().to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    c2, s2 = orc.quantize_kv_fp4(deq_bits)
    has6 = np.array([[((codes[r, 8 * g:8 * g + 8] & 0x7) == 7).any() or ((codes[r, 8 * g:8 * g + 8] >> 4 & 0x7) == 7).any()
                      for g in range(36)] for r in range(64)])
    assert (s2[has6] == scales[has6]).all()


def test_quantize_dst_slot_scatter(orc):
    bits = _rows(12, 5, 128)
    slots = np.array([7, 0, 3, 9, 4])
    c1, s1 = orc.quantize_kv_fp4(bits)
    c2, s2 = orc.quantize_kv_fp4(bits, dst_slot=slots, n_slots=10)
    assert (c2[slots] == c1).all() and (s2[slots] == s1).all()
    untouched = np.setdiff1d(np.arange(10), slots)
    assert (c2[untouched] == 0).all()


def test_quantize_rejects_nonfinite(orc):
    bits = _bf16_bits([float("inf")] + [0.0] * 15)
    with pytest.raises(ValueError):
        orc.quantize_kv_fp4(bits.reshape(1, 16))
