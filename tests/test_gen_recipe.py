"""The seeded input recipe (gen/) is what the documentation states (CPU only):
deterministic per (seed, stream), decode lengths U{32768..65536} tokens at
4 tokens per entry, causal prefill lengths, RMS-normalised KV rows with 0.1%
x8 outliers and RoPE on the last 64 channels, valid FP8 bytes, w in [0, 1)."""
from __future__ import annotations

import numpy as np
import torch

import gen


def test_same_seed_and_stream_give_the_same_bytes_and_streams_differ():
    a = gen.kv_rows(1, 10, 64, 576)
    assert torch.equal(a, gen.kv_rows(1, 10, 64, 576))
    assert not torch.equal(a, gen.kv_rows(1, 11, 64, 576))
    assert not torch.equal(a, gen.kv_rows(2, 10, 64, 576))
    assert torch.equal(gen.normal_e4m3(3, 1, (4, 64)), gen.normal_e4m3(3, 1, (4, 64)))


def test_decode_lengths_follow_the_recipe():
    w = gen.FULL_BATCHED_DECODE
    n = gen.kv_lengths(w).numpy()
    L = gen.seq_lengths(w.seed, 90, w.B, w.len_lo, w.len_hi).numpy()
    assert n.shape == (32,) and (n == L // 4).all()
    assert (L >= 32768).all() and (L <= 65536).all()
    assert abs(n.mean() - 12288) < 1500                      # U{8192..16384} entries, 32 draws
    assert (gen.query_positions(w).numpy() == 4 * n).all()


def test_prefill_lengths_are_causal():
    w = gen.PREFILL_CHUNK
    n = gen.kv_lengths(w).numpy()
    p = gen.query_positions(w).numpy()
    assert (p == 126976 + np.arange(4096)).all()
    assert (n == (p + 1) // 4).all() and n[0] == 31744 and n[-1] == 32768


def test_kv_rows_are_rms_normalised_with_rope_on_the_last_64_channels():
    w = gen.scaled(gen.FULL_BATCHED_DECODE, B=2, N=512)
    x = gen.kv_cache_rows(w).view(torch.bfloat16).double()
    rms = x.pow(2).mean(-1).sqrt()
    assert (rms - 1).abs().max() < 1e-2                       # bf16 rounding and fp32 cos/sin only
    # RoPE at position 4j rotates the pairs (2i, 2i+1) of the last 64 channels only: the same
    # draw without RoPE agrees on the 512 latent channels everywhere and on all channels of
    # entry 0 (position 0)
    raw = gen.kv_rows(w.seed, 10, w.B * w.N, w.D, rms=True, rope_pos=None)
    rot = gen.kv_cache_rows(w)
    assert torch.equal(raw[:, :512], rot[:, :512])
    assert torch.equal(raw[0], rot[0]) and torch.equal(raw[w.N], rot[w.N])
    assert (raw[1:w.N, 512:] != rot[1:w.N, 512:]).any(1).all()


def test_outliers_are_one_in_a_thousand_times_eight():
    x = gen.kv_rows(7, 1, 4096, 512, rms=False).view(torch.bfloat16).float()
    frac = float((x.abs() > 5).float().mean())
    # P(|8 z| > 5) = P(|z| > 0.625) = 0.532 for an outlier; P(|z| > 5) = 5.7e-7 otherwise
    assert 0.8 * 0.532e-3 < frac < 1.2 * 0.532e-3
    assert abs(float(x.std()) - (1 + 1e-3 * 63) ** 0.5) < 0.01


def test_append_rows_are_not_normalised():
    x = gen.kv_cache_rows(gen.APPEND_POOL, rows=256).view(torch.bfloat16).double()
    assert (x.pow(2).mean(-1).sqrt() - 1).abs().max() > 0.05


def test_fp8_inputs_are_valid_e4m3_and_w_is_in_the_unit_interval():
    b = gen.normal_e4m3(5, 1, (1 << 16,)).numpy()
    assert not np.isin(b, [0x7F, 0xFF]).any()                  # no NaN codes
    assert np.isin(b & 0x7F, np.arange(0x60, 0x7F)).sum() == 0  # |z| < 16 for N(0,1) draws of this size
    w = gen.uniform01(5, 2, (1 << 16,)).numpy()
    assert (w >= 0).all() and (w < 1).all()


def test_entry_bytes_of_the_workloads():
    assert gen.FULL_BATCHED_DECODE.entry_bytes == 324 and gen.TINY_FULL_DECODE.entry_bytes == 72
