"""Mutation check of the oracle's pins (CPU only).

Each entry below plants one plausible mistake -- a dropped term, a wrong
sign, bias, index, rounding rule or operand -- in a copy of the oracle's C
source, builds that copy into a library of its own and runs the oracle's pin
modules against it in a child process.  Every mutant must make at least one
pin fail; the unchanged copy (the control) must pass them all.  The mistakes
are planted only in copies on the CPU; every mutant keeps its memory accesses
inside the buffers the pins pass (no index can move past the data).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "csa2_oracle.c")
PINS = ["tests/test_oracle_formats.py", "tests/test_oracle_path.py", "tests/test_oracle_rope.py",
        "tests/test_oracle_swa.py", "tests/test_dense_bound.py"]

# name -> list of (exact text, replacement); each text occurs once in the source
MUTANTS = {
    "control (unchanged)": [],
    # element formats
    "e4m3 subnormal step 2^-10": [("v = ldexp((double)m, -9);", "v = ldexp((double)m, -10);")],
    "e4m3 exponent bias 8": [("v = ldexp(1.0 + m / 8.0, e - 7);", "v = ldexp(1.0 + m / 8.0, e - 8);")],
    "e4m3 0x7F decoded as a number": [("if (e == 15 && m == 7) return NAN;", "")],
    "e2m1 exponent bias 0": [("v = ldexp(1.0 + m / 2.0, e - 1);", "v = ldexp(1.0 + m / 2.0, e);")],
    "e2m1 sign in bit 2": [("int sign = (c >> 3) & 1;", "int sign = (c >> 2) & 1;")],
    "e4m3 encode ties away from zero": [("n = rne((sig - 1.0) * 8.0);", "n = floor((sig - 1.0) * 8.0 + 0.5);")],
    "e4m3 encode truncates": [("n = rne((sig - 1.0) * 8.0);", "n = floor((sig - 1.0) * 8.0);")],
    "e4m3 encode subnormal ties away": [("n = rne(a / ldexp(1.0, -9));", "n = floor(a / ldexp(1.0, -9) + 0.5);")],
    "e4m3 saturates to the NaN code": [("if (a >= 448.0) return 0x7E;", "if (a >= 448.0) return 0x7F;")],
    "e2m1 encode ties away in [1, 2)": [("return (uint8_t)(2 + rne((r - 1.0) / 0.5));",
                                        "return (uint8_t)(2 + floor((r - 1.0) / 0.5 + 0.5));")],
    "e2m1 saturates to code 6": [("if (r >= 6.0) return 7;", "if (r >= 6.0) return 6;")],
    "e2m1 step 4 in [4, 6)": [("return (uint8_t)(6 + rne((r - 4.0) / 2.0));",
                               "return (uint8_t)(6 + rne((r - 4.0) / 4.0));")],
    "e4m3 subnormals flushed to zero": [("n = rne(a / ldexp(1.0, -9));", "n = 0.0 * a;")],
    "e2m1 step 0.25 below 1": [("if (r < 1.0) return (uint8_t)rne(r / 0.5);", "if (r < 1.0) return (uint8_t)rne(r / 0.25);")],
    # quantiser
    "scale amax / 4": [("sbyte = orc_e4m3_encode_pos(amax / 6.0);", "sbyte = orc_e4m3_encode_pos(amax / 4.0);")],
    "amax over 8 channels": [("for (c = 16 * g; c < 16 * g + 16; ++c) {\n                double v",
                              "for (c = 16 * g; c < 16 * g + 8; ++c) {\n                double v")],
    "amax of signed values": [("if (fabs(v) > amax) amax = fabs(v);", "if (v > amax) amax = v;")],
    "nibble order swapped": [("crow[c / 2] = code;", "crow[c / 2] = (uint8_t)(code << 4);"),
                             ("crow[c / 2] |= (uint8_t)(code << 4);", "crow[c / 2] |= code;")],
    "sign dropped when the code is zero": [("uint8_t code = (uint8_t)((sign << 3) | mag);",
                                            "uint8_t code = (uint8_t)((mag ? sign << 3 : 0) | mag);")],
    "dst_slot ignored": [("int64_t slot = dst_slot ? dst_slot[r] : r;", "int64_t slot = r;")],
    # RoPE
    "rotation by -angle": [("const float ra = ac - bs, rb = as + bc;", "const float ra = ac + bs, rb = bc - as;")],
    "rotation with fused multiply-add": [("const float ra = ac - bs, rb = as + bc;",
                                          "const float ra = fmaf(a, cs, -bs), rb = fmaf(a, sn, bc);")],
    "cos and sin swapped": [("const float cs = cos_sin[(p * (rope_dim / 2) + i) * 2];",
                             "const float cs = cos_sin[(p * (rope_dim / 2) + i) * 2 + 1];"),
                            ("const float sn = cos_sin[(p * (rope_dim / 2) + i) * 2 + 1];",
                             "const float sn = cos_sin[(p * (rope_dim / 2) + i) * 2];")],
    "rotated halves instead of interleaved pairs": [
        ("const float a = bf16_to_f32(x[D - rope_dim + 2 * i]);", "const float a = bf16_to_f32(x[D - rope_dim + i]);"),
        ("const float b = bf16_to_f32(x[D - rope_dim + 2 * i + 1]);",
         "const float b = bf16_to_f32(x[D - rope_dim / 2 + i]);"),
        ("y[D - rope_dim + 2 * i] = f32_to_bf16_rne(ra);", "y[D - rope_dim + i] = f32_to_bf16_rne(ra);"),
        ("y[D - rope_dim + 2 * i + 1] = f32_to_bf16_rne(rb);", "y[D - rope_dim / 2 + i] = f32_to_bf16_rne(rb);")],
    "bf16 rounding truncates": [("u += 0x7FFFu + ((u >> 16) & 1u);", "u += 0u;")],
    "RoPE on the first channels": [
        ("const float a = bf16_to_f32(x[D - rope_dim + 2 * i]);", "const float a = bf16_to_f32(x[2 * i]);"),
        ("const float b = bf16_to_f32(x[D - rope_dim + 2 * i + 1]);", "const float b = bf16_to_f32(x[2 * i + 1]);")],
    # indexer scores
    "ReLU dropped": [("s += (double)w[woff + h] * (dot > 0.0 ? dot : 0.0);", "s += (double)w[woff + h] * dot;")],
    "head 0's weight for every head": [("s += (double)w[woff + h] * (dot > 0.0 ? dot : 0.0);",
                                        "s += (double)w[woff] * (dot > 0.0 ? dot : 0.0);")],
    "head 0's query for every head": [("double qv = elem_value(q, q_dt, qoff + h * ORC_IDX_DIM + d);",
                                       "double qv = elem_value(q, q_dt, qoff + d);")],
    "Full mask admits entry kv_len": [("if (j < len)\n", "if (j <= len)\n")],
    "Reindex candidate blk + i": [("int64_t j = (int64_t)blk * 8 + i;", "int64_t j = (int64_t)blk + i;")],
    "Reindex reads sequence 0's keys": [
        ("if (blk >= 0 && j < len)\n                            score_one(q, q_dt, qoff, w, woff, k, k_dt, ((int64_t)b * N + j)",
         "if (blk >= 0 && j < len)\n                            score_one(q, q_dt, qoff, w, woff, k, k_dt, ((int64_t)j)")],
    # pool
    "block maximum skips the 8th position": [("for (j = beta * G; j < beta * G + G && j < len; ++j) {",
                                              "for (j = beta * G; j < beta * G + G - 1 && j < len; ++j) {")],
    "block score is its first position": [("if (v > m) m = v;", "if (m == -INFINITY) m = v;")],
    "partial last block never scores": [("for (j = beta * G; j < beta * G + G && j < len; ++j) {",
                                         "for (j = beta * G; j < beta * G + G && beta * G + G <= len; ++j) {")],
    # selection
    "ties go to the higher position": [("return (x->i < y->i) ? -1 : (x->i > y->i);",
                                        "return (x->i > y->i) ? -1 : (x->i < y->i);")],
    "-inf can be selected": [("if (v[i] > -INFINITY) { buf[n].v", "if (v[i] >= -INFINITY) { buf[n].v")],
    "Top-K admits position kv_len": [("if (j >= len) x = -INFINITY;", "if (j > len) x = -INFINITY;")],
    "Reindex output drops the offset in the block": [
        ("idx[bt * K + s] = (int32_t)((int64_t)pool[bt * P + l / 8] * 8 + l % 8);",
         "idx[bt * K + s] = (int32_t)((int64_t)pool[bt * P + l / 8] * 8);")],
    # attention
    "V is the last dv channels": [("for (c = 0; c < dv; ++c) o[c] += p * kh[(int64_t)i * D + c];",
                                   "for (c = 0; c < dv; ++c) o[c] += p * kh[(int64_t)i * D + (D - dv) + c];")],
    "logits without sm_scale": [("acc += bf16_value(qr[c]) * kh[(int64_t)i * D + c];\n                z[i] = sm_scale * acc;",
                                 "acc += bf16_value(qr[c]) * kh[(int64_t)i * D + c];\n                z[i] = acc;")],
    "lse in base 2": [("l = m + log(sum);", "l = m + log2(sum);")],
    "weights not normalised": [("double p = exp(z[i] - l);", "double p = exp(z[i] - m);")],
    "one scale per 32 channels": [("orc_e4m3_value(srow[c / 16]);", "orc_e4m3_value(srow[c / 32]);")],
    "dequant reads the nibbles swapped": [("uint8_t code = (c & 1) ? (byte >> 4) : (byte & 0xF);",
                                           "uint8_t code = (c & 1) ? (byte & 0xF) : (byte >> 4);")],
    "sm_scale applied twice": [("acc += bf16_value(qr[c]) * kh[(int64_t)i * D + c];\n                z[i] = sm_scale * acc;",
                                "acc += bf16_value(qr[c]) * kh[(int64_t)i * D + c];\n                z[i] = sm_scale * sm_scale * acc;")],
    "query channels beyond dv ignored": [("for (c = 0; c < D; ++c) acc += bf16_value(qr[c]) * kh[(int64_t)i * D + c];",
                                          "for (c = 0; c < dv; ++c) acc += bf16_value(qr[c]) * kh[(int64_t)i * D + c];")],
    # sliding window + merge
    "window logits without sm_scale": [("for (c = 0; c < D; ++c) acc += bf16_value(qr[c]) * orc_e4m3_value(kr[c]);\n                z[i] = sm_scale * acc;",
                                        "for (c = 0; c < D; ++c) acc += bf16_value(qr[c]) * orc_e4m3_value(kr[c]);\n                z[i] = acc;")],
    "merge weights swapped": [("o[c] = (a * ow[c] + cs * os) / (a + cs);", "o[c] = (cs * ow[c] + a * os) / (a + cs);")],
    "merged lse is the window's": [("if (lse) lse[bt * H + h] = M + log(a + cs);", "if (lse) lse[bt * H + h] = lw;")],
    "window V is the last dv channels": [("for (c = 0; c < dv; ++c) ow[c] += p * orc_e4m3_value(kr[c]);",
                                          "for (c = 0; c < dv; ++c) ow[c] += p * orc_e4m3_value(kr[D - dv + c]);")],
}

_DRIVER = """
import sys
sys.path.insert(0, {root!r})
import oracle
oracle._SRC, oracle._LIB, oracle._lib = {src!r}, {lib!r}, None
import pytest
sys.exit(pytest.main(["-x", "-q", "-p", "no:cacheprovider", *{pins!r}]))
"""


def _mutate(subs):
    with open(SRC) as f:
        s = f.read()
    for old, new in subs:
        assert s.count(old) == 1, "mutant text not unique in the oracle: %r" % old
        s = s.replace(old, new)
    return s


def _run(name, subs, work):
    d = os.path.join(work, "m%02d" % list(MUTANTS).index(name))
    os.makedirs(d)
    src, lib = os.path.join(d, "mutant.c"), os.path.join(d, "libmutant.so")
    with open(src, "w") as f:
        f.write(_mutate(subs))
    r = subprocess.run([sys.executable, "-c", _DRIVER.format(root=ROOT, src=src, lib=lib, pins=PINS)],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    return r.returncode, (r.stdout + r.stderr)[-1500:]


@pytest.fixture(scope="module")
def results(tmp_path_factory):
    work = str(tmp_path_factory.mktemp("oracle_mutants"))
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        futs = {n: ex.submit(_run, n, subs, work) for n, subs in MUTANTS.items()}
        return {n: f.result() for n, f in futs.items()}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_pins_catch_planted_mistake(results, name):
    rc, tail = results[name]
    if not MUTANTS[name]:
        assert rc == 0, "the unchanged oracle copy fails its pins:\n" + tail
    else:
        # pytest exit code 1: a pin failed (not a crash, an error or no tests)
        assert rc == 1, "mutant %r was not caught by a pin (exit %d):\n%s" % (name, rc, tail)
