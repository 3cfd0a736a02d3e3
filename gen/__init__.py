"""Seeded synthetic inputs for the CSA2 FP4 decode path.

This module only draws random numbers and lays them out; it holds none of the
path's arithmetic (no quantisation, scoring, selection or attention).  Both
the CUDA library's tests/benchmark and the CPU oracle take their inputs from
here, so the two sides always see identical bytes.

Shapes and value distributions stand in for the workloads the pages describe
(DeepSeek-V4.1-Flash: 4:1 compressed entries of 512 latent + 64 RoPE
channels, contexts from 4K to 1M tokens, Top-512, a 2048 x 8 candidate pool).
The pages print no tensor shapes, so the five workloads below are synthetic
stand-ins with the sizes stated in their docstrings.

Randomness comes from ``torch.Generator`` seeded per tensor (seed, stream
id), on the CPU for sizes the oracle handles and optionally on a CUDA device
for full-size workloads (the oracle then receives the sampled rows it needs).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

ROPE_DIMS = 64          # last 64 channels of every KV entry / query carry RoPE
ROPE_THETA = 1.0e4
COMPRESS = 4            # one compressed entry per 4 tokens
IDX_HEADS, IDX_DIM = 4, 64


def _g(seed: int, stream: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1_000_003 + int(stream) * 7919) & 0x7FFF_FFFF_FFFF)
    return g


def bf16_bits(x: torch.Tensor) -> torch.Tensor:
    """fp32 -> bf16 (round to nearest even, torch's cast) as int16 bit patterns."""
    return x.to(torch.bfloat16).view(torch.int16)


def e4m3_bytes(x: torch.Tensor) -> torch.Tensor:
    """fp32 -> FP8 E4M3 bytes via torch's cast (inputs are clamped to +-448)."""
    return x.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)


def rope_interleaved(x: torch.Tensor, pos: torch.Tensor) -> torch.Tensor:
    """Rotate the last 64 channels of x [..., n, D] by position pos [..., n]
    (pairs (2i, 2i+1), theta = 1e4).  Input synthesis only: the path's
    inputs are post-RoPE rows."""
    d = x.shape[-1]
    r = x[..., d - ROPE_DIMS:].reshape(*x.shape[:-1], ROPE_DIMS // 2, 2)
    inv = ROPE_THETA ** (-torch.arange(0, ROPE_DIMS, 2, dtype=torch.float64, device=x.device) / ROPE_DIMS)
    ang = pos.to(torch.float64)[..., None] * inv
    c, s = torch.cos(ang).to(x.dtype), torch.sin(ang).to(x.dtype)
    a, b = r[..., 0], r[..., 1]
    rot = torch.stack((a * c - b * s, a * s + b * c), dim=-1).reshape(*x.shape[:-1], ROPE_DIMS)
    return torch.cat((x[..., : d - ROPE_DIMS], rot), dim=-1)


def rope_table(n_pos, rope_dim=None, theta=None, device="cpu") -> torch.Tensor:
    """fp32 [n_pos, rope_dim/2, 2] table of (cos, sin) of position * theta^(-2i/rope_dim),
    evaluated in fp64 and rounded to fp32 (an input of the fused RoPE + quantise call)."""
    rope_dim = ROPE_DIMS if rope_dim is None else rope_dim
    theta = ROPE_THETA if theta is None else theta
    inv = theta ** (-torch.arange(0, rope_dim, 2, dtype=torch.float64) / rope_dim)
    ang = torch.arange(n_pos, dtype=torch.float64)[:, None] * inv
    return torch.stack((torch.cos(ang), torch.sin(ang)), dim=-1).to(torch.float32).to(device)


def kv_rows(seed, stream, rows, D, *, rms=True, rope_pos=None, outlier_p=1e-3, outlier_mul=8.0,
            device="cpu") -> torch.Tensor:
    """bf16 bit patterns [rows, D] of post-RoPE KV rows: N(0,1) with each
    element independently multiplied by ``outlier_mul`` with probability
    ``outlier_p``, optionally RMS-normalised (no gain), then RoPE on the last
    64 channels at token position ``rope_pos[r]``."""
    g = _g(seed, stream, device)
    x = torch.randn(rows, D, generator=g, device=device, dtype=torch.float32)
    if outlier_p > 0:
        m = torch.rand(rows, D, generator=g, device=device) < outlier_p
        x = torch.where(m, x * outlier_mul, x)
    if rms:
        x = x * torch.rsqrt(x.pow(2).mean(dim=-1, keepdim=True) + 1e-6)
    if rope_pos is not None:
        x = rope_interleaved(x, rope_pos.to(device))
    return bf16_bits(x)


def normal_bf16(seed, stream, shape, *, device="cpu", rope_pos=None) -> torch.Tensor:
    g = _g(seed, stream, device)
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if rope_pos is not None:
        x = rope_interleaved(x, rope_pos.to(device))
    return bf16_bits(x)


def normal_e4m3(seed, stream, shape, *, device="cpu") -> torch.Tensor:
    g = _g(seed, stream, device)
    return e4m3_bytes(torch.randn(*shape, generator=g, device=device, dtype=torch.float32))


def uniform01(seed, stream, shape, *, device="cpu") -> torch.Tensor:
    g = _g(seed, stream, device)
    return torch.rand(*shape, generator=g, device=device, dtype=torch.float32)


def seq_lengths(seed, stream, B, lo, hi) -> torch.Tensor:
    """Token lengths L_b ~ U{lo..hi} (inclusive), int64 [B]."""
    g = _g(seed, stream)
    return torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64)


@dataclass(frozen=True)
class Workload:
    """Shape of one synthetic workload.  ``N`` is the per-sequence entry
    capacity; ``kv_len`` per query token is derived by ``kv_lengths``."""
    name: str
    seed: int
    B: int
    T: int
    N: int
    D: int
    dv: int
    H: int
    K: int = 512
    P: int = 2048
    idx_dtype: str = "fp8"          # "fp8" or "bf16" for the indexer q and keys
    len_lo: int = 0                 # token-length range (decode); 0 = full N
    len_hi: int = 0
    prefill_first_pos: int = -1     # >= 0: T causal queries at consecutive positions
    extra: dict = field(default_factory=dict)

    @property
    def entry_bytes(self) -> int:
        return self.D // 2 + self.D // 16


def kv_lengths(w: Workload) -> torch.Tensor:
    """Visible entry count per query token, int32 [B*T].  Entry j covers
    tokens [4j, 4j+4); a query at token position p sees j < (p+1)//4."""
    if w.prefill_first_pos >= 0:
        pos = torch.arange(w.prefill_first_pos, w.prefill_first_pos + w.T, dtype=torch.int64)
        per_q = (pos + 1) // COMPRESS
        return per_q.repeat(w.B).clamp(max=w.N).to(torch.int32)
    if w.len_hi > 0:
        L = seq_lengths(w.seed, 90, w.B, w.len_lo, w.len_hi)
        n = (L // COMPRESS).clamp(max=w.N)
        return n.repeat_interleave(w.T).to(torch.int32)
    return torch.full((w.B * w.T,), w.N, dtype=torch.int32)


def query_positions(w: Workload) -> torch.Tensor:
    """Token position of every query, int64 [B*T] (used for RoPE on Q)."""
    if w.prefill_first_pos >= 0:
        pos = torch.arange(w.prefill_first_pos, w.prefill_first_pos + w.T, dtype=torch.int64)
        return pos.repeat(w.B)
    n = kv_lengths(w).to(torch.int64)
    return n * COMPRESS


# The five workloads (seed = workload number - 1).
TINY_FULL_DECODE = Workload("tiny_full_decode_b1_n1024_d128_h16", 0, B=1, T=1, N=1024, D=128, dv=64,
                            H=16, idx_dtype="bf16")
FULL_BATCHED_DECODE = Workload("full_decode_b32_ctx64k_n16384_d576_h64", 1, B=32, T=1, N=16384, D=576,
                               dv=512, H=64, len_lo=32768, len_hi=65536)
REINDEX_REUSE_1M = Workload("reindex_reuse_group_b8_ctx1m_n262144_d576_h64", 2, B=8, T=1, N=262144,
                            D=576, dv=512, H=64)
PREFILL_CHUNK = Workload("prefill_chunk_t4096_ctx128k_n32768_d576_h64", 3, B=1, T=4096, N=32768,
                         D=576, dv=512, H=64, prefill_first_pos=126976)
APPEND_POOL = Workload("append_1m_rows_d576_pool_b16_n65536", 4, B=16, T=1, N=65536, D=576, dv=512,
                       H=64)

WORKLOADS = [TINY_FULL_DECODE, FULL_BATCHED_DECODE, REINDEX_REUSE_1M, PREFILL_CHUNK, APPEND_POOL]

# The decoder's layer schedule ("DeepSeek-V4.1-Flash：把 KV Cache 压缩到极限的百万上下文
# MoE", CSA2 section): 20 layers in 5 groups of 4, the first group 1 Full + 3
# Reuse, the other four 1 Reindex + 3 Reuse.  A constant of the workload, kept
# here so that the oracle's timing leg can use it without loading the CUDA
# library.
DECODER_SCHEDULE = ("full", "reuse", "reuse", "reuse") + ("reindex", "reuse", "reuse", "reuse") * 4


def scaled(w: Workload, **changes) -> Workload:
    """A smaller copy of a workload (same distributions) for oracle-sized tests."""
    d = dict(w.__dict__)
    d.update(changes)
    return Workload(**d)


# ------------------------------------------------------------- tensor sets
def kv_cache_rows(w: Workload, stream=10, device="cpu", rows=None) -> torch.Tensor:
    """bf16 KV rows for all B*N entries (or the first ``rows``), RoPE at
    token position 4j of entry j.  The append workload uses iid N(0,1)
    rows with outliers and no RMS norm or RoPE."""
    R = w.B * w.N if rows is None else rows
    if w is APPEND_POOL or w.name.startswith("append"):
        return kv_rows(w.seed, stream, R, w.D, rms=False, rope_pos=None, device=device)
    j = torch.arange(R, dtype=torch.int64) % w.N
    return kv_rows(w.seed, stream, R, w.D, rms=True, rope_pos=j * COMPRESS, device=device)


def indexer_inputs(w: Workload, layer=0, device="cpu"):
    """(q [B,T,4,64], w fp32 [B,T,4], k [B,N,64]) for the indexer of one
    layer.  q/k are FP8 E4M3 bytes (uint8) or bf16 bits (int16)."""
    s = 20 + 3 * layer
    if w.idx_dtype == "bf16":
        q = normal_bf16(w.seed, s, (w.B, w.T, IDX_HEADS, IDX_DIM), device=device)
        k = normal_bf16(w.seed, 19, (w.B, w.N, IDX_DIM), device=device)
    else:
        q = normal_e4m3(w.seed, s, (w.B, w.T, IDX_HEADS, IDX_DIM), device=device)
        k = normal_e4m3(w.seed, 19, (w.B, w.N, IDX_DIM), device=device)
    wt = uniform01(w.seed, s + 1, (w.B, w.T, IDX_HEADS), device=device)
    return q, wt, k


def attn_query(w: Workload, layer=0, device="cpu") -> torch.Tensor:
    """Attention Q [B,T,H,D] bf16 bits, N(0,1) with RoPE at the query's position."""
    pos = query_positions(w).reshape(w.B, w.T, 1).expand(w.B, w.T, w.H)
    return normal_bf16(w.seed, 200 + layer, (w.B, w.T, w.H, w.D), device=device, rope_pos=pos)


def random_indices(w: Workload, kv_len: torch.Tensor, stream=300, frac_pad=0.0) -> torch.Tensor:
    """int32 [B,T,K] distinct valid positions < kv_len per row (for testing the
    attention step on its own), with an optional fraction of -1 padding."""
    g = _g(w.seed, stream)
    out = torch.full((w.B * w.T, w.K), -1, dtype=torch.int32)
    for r in range(w.B * w.T):
        n = int(kv_len[r])
        k = min(w.K, n)
        sel = torch.randperm(n, generator=g)[:k].to(torch.int32)
        if frac_pad > 0:
            keep = torch.rand(k, generator=g) >= frac_pad
            sel = torch.where(keep, sel, torch.full_like(sel, -1))
        out[r, :k] = sel
    return out.reshape(w.B, w.T, w.K)


def softmax_scale(D: int) -> float:
    """1/sqrt(D) (the pages state no softmax scale)."""
    return 1.0 / math.sqrt(D)


def as_numpy(t: torch.Tensor) -> np.ndarray:
    """Host NumPy view with unsigned bit-pattern types where relevant."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.int16:
        return t.numpy().view(np.uint16)
    return t.numpy()


def fp4_planes(seed, stream, rows, D, device="cpu"):
    """Random FP4 cache planes (codes uint8 [rows, D/2], scales uint8
    [rows, D/16]) for timing-only work: uniform code bytes and scale bytes in
    [0x20, 0x38) (E4M3 values 0.125 .. 0.9, the range N(0,1) groups give)."""
    g = _g(seed, stream, device)
    codes = torch.randint(0, 256, (rows, D // 2), generator=g, device=device, dtype=torch.int32).to(torch.uint8)
    scales = torch.randint(0x20, 0x38, (rows, D // 16), generator=g, device=device, dtype=torch.int32).to(torch.uint8)
    return codes, scales
