"""CPU oracle for the CSA2 FP4 decode path -- TEST INFRASTRUCTURE ONLY.

Plain fp64 C code (``csa2_oracle.c``) behind a ctypes wrapper that takes and
returns NumPy arrays.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the product library
never does.  It shares no code with the CUDA library.

Every function follows a passage of the pages about the DeepSeek-V4.1-Flash
report (cited in ``csa2_oracle.c``):

* ``quantize_kv_fp4`` -- "DeepSeek-V4.1-Flash：把 KV Cache 压缩到极限的百万上下文 MoE",
  section "效率组件四件", item 4 (E2M1 + one E4M3 scale per 16 channels,
  quantised after RoPE, no global scale).
* ``index_score`` -- same page, "Hierarchical Sparse Indexer" (Full scores
  every entry, Reindex only the pool); the score formula itself is not on
  the pages (read as sum_h w_h ReLU(q_h . k)).
* ``build_pool`` -- same page, "Hierarchical Sparse Indexer" (<= 2048 blocks
  x 8 positions).
* ``topk`` -- same page, CSA2 section (Top-512).
* ``sparse_attn`` -- MLA-style attention over the selected FP4 entries
  (reading; the pages give no formula).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csa2_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

BF16, FP8_E4M3, FP32 = 0, 1, 2
FULL, REINDEX, REUSE = 0, 1, 2

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with plain gcc (no fast-math, no SIMD flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                               "-fno-fast-math", "-ffp-contract=off",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.orc_rounding_mode_ok.restype = i32
        lib.orc_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.orc_e4m3_value.restype = dbl
        lib.orc_e2m1_value.argtypes = [ctypes.c_uint8]
        lib.orc_e2m1_value.restype = dbl
        lib.orc_bf16_value.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_value.restype = dbl
        lib.orc_e4m3_encode_pos.argtypes = [dbl]
        lib.orc_e4m3_encode_pos.restype = ctypes.c_uint8
        lib.orc_e2m1_encode_mag.argtypes = [dbl]
        lib.orc_e2m1_encode_mag.restype = ctypes.c_uint8
        lib.orc_quantize_kv_fp4.argtypes = [P, i64, i32, i64, P, P, P]
        lib.orc_quantize_kv_fp4.restype = i32
        lib.orc_dequant_fp4.argtypes = [P, P, i64, i32, P]
        lib.orc_dequant_fp4.restype = None
        lib.orc_index_score.argtypes = [i32, i32, i32, i64, P, i32, P, P, i32, P, P, i32, P, P]
        lib.orc_index_score.restype = i32
        lib.orc_build_pool.argtypes = [i32, i32, i64, P, P, i32, i32, P]
        lib.orc_build_pool.restype = i32
        lib.orc_topk.argtypes = [i32, i32, i32, i64, P, P, P, i32, i32, P]
        lib.orc_topk.restype = i32
        lib.orc_sparse_attn.argtypes = [i32, i32, i32, i32, i32, P, P, P, i64, P, i32, P, dbl, P, P]
        lib.orc_sparse_attn.restype = i64
        lib.orc_rope_bf16.argtypes = [P, i64, i32, i64, P, P, i64, i32, P]
        lib.orc_rope_bf16.restype = i32
        lib.orc_swa_attn_merge.argtypes = [i32, i32, i32, i32, i32, P, P, i32, P, dbl, P, P, P, P]
        lib.orc_swa_attn_merge.restype = i32
        if not lib.orc_rounding_mode_ok():
            raise RuntimeError("oracle needs the round-to-nearest-even FP mode")
        _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ----------------------------------------------------------------- formats
def e4m3_value(b: int) -> float:
    return _load().orc_e4m3_value(int(b))


def e2m1_value(c: int) -> float:
    return _load().orc_e2m1_value(int(c))


def bf16_value(h: int) -> float:
    return _load().orc_bf16_value(int(h))


def e4m3_encode_pos(a: float) -> int:
    return int(_load().orc_e4m3_encode_pos(float(a)))


def e2m1_encode_mag(r: float) -> int:
    return int(_load().orc_e2m1_encode_mag(float(r)))


# ----------------------------------------------------------------- the path
def quantize_kv_fp4(kv_bf16_bits: np.ndarray, dst_slot=None, n_slots=None):
    """kv: uint16 bf16 bits [R, D] -> (codes uint8 [S, D/2], scales uint8 [S, D/16])."""
    kv = _c(kv_bf16_bits, np.uint16)
    R, D = kv.shape
    S = R if n_slots is None else n_slots
    codes = np.zeros((S, D // 2), np.uint8)
    scales = np.zeros((S, D // 16), np.uint8)
    slot = None if dst_slot is None else _c(dst_slot, np.int64)
    rc = _load().orc_quantize_kv_fp4(_p(kv), R, D, D, _p(slot), _p(codes), _p(scales))
    if rc != 0:
        raise ValueError("oracle quantize: non-finite input or bad D")
    return codes, scales


def rope_bf16(kv_bf16_bits: np.ndarray, pos, cos_sin, rope_dim=64):
    """RoPE (interleaved pairs of the last rope_dim channels, fp32 table
    cos_sin [n_pos, rope_dim/2, 2], fp32 arithmetic without FMA) -> bf16 bits."""
    kv = _c(kv_bf16_bits, np.uint16)
    R, D = kv.shape
    ps = _c(pos, np.int32)
    cs = _c(cos_sin, np.float32)
    out = np.zeros((R, D), np.uint16)
    rc = _load().orc_rope_bf16(_p(kv), R, D, D, _p(ps), _p(cs), cs.shape[0], rope_dim, _p(out))
    if rc != 0:
        raise ValueError("oracle rope: bad shape or position")
    return out


def rope_quantize_kv_fp4(kv_bf16_bits, pos, cos_sin, rope_dim=64, dst_slot=None, n_slots=None):
    """Pre-RoPE bf16 rows -> RoPE (rope_bf16) -> quantize_kv_fp4."""
    return quantize_kv_fp4(rope_bf16(kv_bf16_bits, pos, cos_sin, rope_dim), dst_slot=dst_slot, n_slots=n_slots)


def dequant_fp4(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    R = codes.shape[0]
    D = codes.shape[1] * 2
    out = np.zeros((R, D), np.float64)
    _load().orc_dequant_fp4(_p(codes), _p(scales), R, D, _p(out))
    return out


def index_score(mode, q, q_dt, w, k, k_dt, kv_len, pool=None, with_mag=False):
    """q [B,T,4,64], w fp32 [B,T,4], k [B,N,64]; returns fp64 scores
    [B,T,N] (FULL) or [B,T,8P] (REINDEX), and optionally the magnitudes."""
    B, T = q.shape[0], q.shape[1]
    N = k.shape[1]
    qa = _c(q, np.uint16 if q_dt == BF16 else np.uint8)
    ka = _c(k, np.uint16 if k_dt == BF16 else np.uint8)
    wa = _c(w, np.float32)
    kl = _c(kv_len, np.int32)
    if mode == REINDEX:
        pa = _c(pool, np.int32)
        P = pa.shape[-1]
        M = 8 * P
    else:
        pa, P, M = None, 0, N
    out = np.zeros((B, T, M), np.float64)
    mag = np.zeros((B, T, M), np.float64) if with_mag else None
    rc = _load().orc_index_score(mode, B, T, N, _p(qa), q_dt, _p(wa), _p(ka), k_dt, _p(kl),
                                 _p(pa), P, _p(out), _p(mag))
    if rc != 0:
        raise ValueError("oracle index_score: bad arguments")
    return (out, mag) if with_mag else out


def build_pool(scores_f32, kv_len, P=2048, G=8):
    s = _c(scores_f32, np.float32)
    B, T, N = s.shape
    kl = _c(kv_len, np.int32)
    out = np.zeros((B, T, P), np.int32)
    rc = _load().orc_build_pool(B, T, N, _p(s), _p(kl), P, G, _p(out))
    if rc != 0:
        raise MemoryError("oracle build_pool")
    return out


def topk(mode, scores_f32, kv_len=None, pool=None, K=512):
    s = _c(scores_f32, np.float32)
    B, T, M = s.shape
    kl = None if kv_len is None else _c(kv_len, np.int32)
    pa = None if pool is None else _c(pool, np.int32)
    P = 0 if pa is None else pa.shape[-1]
    idx = np.full((B, T, K), -7, np.int32)
    rc = _load().orc_topk(mode, B, T, M, _p(s), _p(kl), _p(pa), P, K, _p(idx))
    if rc != 0:
        raise ValueError("oracle topk: bad arguments")
    return idx


def sparse_attn(q_bf16_bits, codes, scales, N, idx, kv_len, sm_scale, dv):
    """q [B,T,H,D] bf16 bits; codes [B*N, D/2]; scales [B*N, D/16];
    idx int32 [B,T,K] -> (out fp64 [B,T,H,dv], lse fp64 [B,T,H], n_bad)."""
    q = _c(q_bf16_bits, np.uint16)
    B, T, H, D = q.shape
    ia = _c(idx, np.int32)
    K = ia.shape[-1]
    kl = None if kv_len is None else _c(kv_len, np.int32)
    out = np.zeros((B, T, H, dv), np.float64)
    lse = np.zeros((B, T, H), np.float64)
    bad = _load().orc_sparse_attn(B, T, H, D, dv, _p(q), _p(_c(codes, np.uint8)),
                                  _p(_c(scales, np.uint8)), N, _p(ia), K, _p(kl),
                                  float(sm_scale), _p(out), _p(lse))
    if bad < 0:
        raise MemoryError("oracle sparse_attn")
    return out, lse, int(bad)


def swa_attn_merge(q_bf16_bits, kv_e4m3, swa_len, sm_scale, dv, o_sparse=None, lse_sparse=None):
    """q uint16 [B,T,H,D]; kv uint8 E4M3 [B,W,D]; swa_len int32 [B*T]; optional
    fp64/fp32 o_sparse [B,T,H,dv] and lse_sparse [B,T,H] -> (out fp64 [B,T,H,dv],
    lse fp64 [B,T,H]): the window branch merged with the sparse branch."""
    qa = _c(q_bf16_bits, np.uint16)
    B, T, H, D = qa.shape
    ka = _c(kv_e4m3, np.uint8)
    W = ka.shape[1]
    sl = _c(swa_len, np.int32)
    os_ = None if o_sparse is None else _c(o_sparse, np.float64)
    ls = None if lse_sparse is None else _c(lse_sparse, np.float64)
    out = np.zeros((B, T, H, dv), np.float64)
    lse = np.zeros((B, T, H), np.float64)
    rc = _load().orc_swa_attn_merge(B, T, H, D, dv, _p(qa), _p(ka), W, _p(sl), ctypes.c_double(sm_scale),
                                    _p(os_), _p(ls), _p(out), _p(lse))
    if rc != 0:
        raise MemoryError("oracle swa_attn_merge")
    return out, lse
