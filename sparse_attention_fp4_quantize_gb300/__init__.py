"""Python binding of libcsa2 -- the CSA2 decode hot path over an FP4 main KV
cache, as hand-written CUDA kernels for GB300 (sm_103a).

Argument marshalling only: every function passes torch tensors' device
pointers, shapes and the current CUDA stream to the C ABI declared in
``include/csa2.h`` and raises ``Csa2Error`` on a non-OK status.  Since the C
calls see bare pointers, the binding first refuses (TypeError / ValueError)
tensors whose element size does not match what the call reads or writes and
buffers smaller than the call touches.  There is no CPU fallback: if the
shared library is missing the import fails loudly.

Names follow the C ABI: ``csa2_quantize_kv_fp4``, ``csa2_rope_quantize_kv_fp4``
(RoPE fused ahead of the quantiser), ``csa2_index_score``, ``csa2_build_pool``,
``csa2_topk``, ``csa2_index_topk`` (fused decode indexer),
``csa2_index_topk_dense`` (fused indexer for many query tokens),
``csa2_sparse_attn_fp4`` (and ``csa2_sparse_attn_fp4_noalloc``),
``csa2_swa_attn_fp8`` (sliding-window branch and merge),
``csa2_selftest_bounded_wait`` and the ``*_workspace_bytes`` helpers.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcsa2.so")

MODE_FULL, MODE_REINDEX, MODE_REUSE = 0, 1, 2
BF16, FP8_E4M3, FP32 = 0, 1, 2
FLAG_BAD_INDEX, FLAG_BAD_POOL, FLAG_BAD_SLOT, FLAG_TIMEOUT = 0x1, 0x2, 0x4, 0x8
INDEX_HEADS, INDEX_DIM, POOL_BLOCK, MAX_POOL, MAX_K = 4, 64, 8, 2048, 2048

STATUS = {0: "CSA2_OK", 1: "CSA2_ERR_INVALID_ARG", 2: "CSA2_ERR_UNSUPPORTED", 3: "CSA2_ERR_WORKSPACE",
          4: "CSA2_ERR_CUDA", 5: "CSA2_ERR_DEVICE_FLAG", 6: "CSA2_ERR_TIMEOUT"}


class Csa2Error(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__("%s: %s" % (STATUS.get(status, status), detail))
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError("libcsa2.so is not built (run __graft_entry__.build() or "
                          "python sparse_attention_fp4_quantize_gb300/build.py)")
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, i64, u64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    sig = {
        "csa2_quantize_kv_fp4": ([P, i64, i32, i64, P, i64, P, P, P, P], i32),
        "csa2_rope_quantize_kv_fp4": ([P, i64, i32, i64, P, P, i64, i32, P, i64, P, P, P, P], i32),
        "csa2_index_score": ([i32, i32, i32, i64, P, i32, P, P, i32, P, P, i32, P, P, P], i32),
        "csa2_build_pool": ([i32, i32, i64, P, P, i32, i32, P, P, u64, P], i32),
        "csa2_build_pool_workspace_bytes": ([i32, i32, i64, i32], u64),
        "csa2_topk": ([i32, i32, i32, i64, P, P, P, i32, i32, P, P, u64, P], i32),
        "csa2_topk_workspace_bytes": ([i32, i32, i64, i32], u64),
        "csa2_index_topk": ([i32, i32, i32, i64, P, i32, P, P, i32, P, P, i32, i32, P, P, i32, P, P], i32),
        "csa2_index_topk_dense": ([i32, i32, i64, P, i32, P, P, i32, P, i32, P, P, P, u64, P], i32),
        "csa2_index_topk_dense_workspace_bytes": ([i32, i32, i64, i32], u64),
        "csa2_sparse_attn_fp4": ([i32, i32, i32, i32, i32, i32, P, P, P, i64, P, i32, P, f32, P, i32, P, P,
                                  P, u64, P], i32),
        "csa2_sparse_attn_workspace_bytes": ([i32, i32, i32, i32, i32, i32], u64),
        "csa2_sparse_attn_fp4_prefetch": ([i32, i32, i32, i32, i32, i32, P, P, P, i64, P, i32, P, f32, P, i32, P, P,
                                           P, u64, P, P, P], i32),
        "csa2_swa_attn_fp8": ([i32, i32, i32, i32, i32, P, P, i32, P, f32, P, P, P, P, P, P], i32),
        "csa2_sparse_attn_fp4_noalloc": ([i32, i32, i32, i32, i32, i32, P, P, P, i64, P, i32, P, f32, P, i32, P,
                                          P, P], i32),
        "csa2_sparse_attn_noalloc_max_scratch_bytes": ([], u64),
        "csa2_selftest_bounded_wait": ([ctypes.c_uint32, P, P], i32),
        "csa2_status_string": ([i32], ctypes.c_char_p),
        "csa2_last_error": ([], ctypes.c_char_p),
        "csa2_version": ([], i32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


_lib = _load()


def exported_symbols():
    return ["csa2_quantize_kv_fp4", "csa2_rope_quantize_kv_fp4", "csa2_index_score", "csa2_build_pool", "csa2_build_pool_workspace_bytes",
            "csa2_topk", "csa2_topk_workspace_bytes", "csa2_index_topk", "csa2_index_topk_dense",
            "csa2_index_topk_dense_workspace_bytes", "csa2_sparse_attn_fp4", "csa2_sparse_attn_workspace_bytes",
            "csa2_sparse_attn_fp4_prefetch", "csa2_swa_attn_fp8",
            "csa2_sparse_attn_fp4_noalloc", "csa2_sparse_attn_noalloc_max_scratch_bytes",
            "csa2_selftest_bounded_wait", "csa2_status_string", "csa2_last_error", "csa2_version"]


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(rc: int):
    if rc != 0:
        raise Csa2Error(rc, _lib.csa2_last_error().decode())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return FP8_E4M3
    if t.dtype in (torch.bfloat16, torch.int16):
        return BF16
    raise TypeError("indexer tensors must be FP8 E4M3 (uint8/float8_e4m3fn) or bf16 (bfloat16/int16 bits)")


def _on_device(t) -> bool:
    return t.is_cuda


def _cuda(*ts):
    for t in ts:
        if t is not None and (not _on_device(t) or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def _elem(t, name, sizes, floating=None):
    """The C call reads or writes t's memory as elements of one of these
    byte sizes (and of this kind, when given)."""
    if t is None:
        return
    if t.element_size() not in sizes or (floating is not None and t.is_floating_point() != floating):
        raise TypeError("%s: %s elements do not fit this call" % (name, t.dtype))


def _bf16(t, name):
    """The C call reads t as bf16 values: only torch.bfloat16 or its int16
    bit patterns are accepted (a float16 tensor has the same element size
    but other values)."""
    if t is not None and t.dtype not in (torch.bfloat16, torch.int16):
        raise TypeError("%s: %s elements are not bf16 (pass torch.bfloat16 or int16 bit patterns)" % (name, t.dtype))


def _room(t, name, n):
    """t must hold every element the call touches (the C side sees only a pointer)."""
    if t is not None and t.numel() < n:
        raise ValueError("%s holds %d elements, the call touches %d" % (name, t.numel(), n))


def _flag(err_flag):
    _elem(err_flag, "err_flag", (4,), False)
    _room(err_flag, "err_flag", 1)


def _indexer_operands(q_idx, w, k_idx, kv_len, B, T, N):
    _elem(q_idx, "q_idx", (1, 2))
    _elem(k_idx, "k_idx", (1, 2))
    _elem(w, "w", (4,), True)
    _elem(kv_len, "kv_len", (4,), False)
    _room(q_idx, "q_idx", B * T * INDEX_HEADS * INDEX_DIM)
    _room(k_idx, "k_idx", B * N * INDEX_DIM)
    _room(w, "w", B * T * INDEX_HEADS)
    _room(kv_len, "kv_len", B * T)


def csa2_selftest_bounded_wait(err_flag, max_polls=4096, stream=None):
    """The kernels' bounded mbarrier wait on an arrival that never comes:
    sets FLAG_TIMEOUT in err_flag (int32/uint32 CUDA tensor) and returns."""
    _cuda(err_flag)
    _check(_lib.csa2_selftest_bounded_wait(int(max_polls), _ptr(err_flag), _stream(stream)))


def version() -> int:
    return _lib.csa2_version()


def _plane_args(kv, codes, scales, dst_slot, err_flag, R, D, n_slots):
    _bf16(kv, "kv")
    _elem(codes, "codes", (1,))
    _elem(scales, "scales", (1,))
    _elem(dst_slot, "dst_slot", (8,), False)
    _flag(err_flag)
    if codes.dim() != 2 or codes.shape[1] != D // 2:
        raise ValueError("codes must be [slots, D/2] = [*, %d], got %s" % (D // 2, tuple(codes.shape)))
    _room(scales, "scales", n_slots * (D // 16))
    _room(dst_slot, "dst_slot", R)


def csa2_quantize_kv_fp4(kv, codes, scales, dst_slot=None, err_flag=None, stream=None):
    """kv bf16 [R, D] (or int16 bits) -> codes uint8 [S, D/2], scales uint8 [S, D/16]."""
    _cuda(codes, scales, dst_slot, err_flag)
    R, D = kv.shape
    if not _on_device(kv) or kv.stride(1) != 1:
        raise ValueError("kv must be a CUDA tensor with contiguous rows (any row stride)")
    n_slots = codes.shape[0]
    _plane_args(kv, codes, scales, dst_slot, err_flag, R, D, n_slots)
    _check(_lib.csa2_quantize_kv_fp4(_ptr(kv), R, D, kv.stride(0), _ptr(dst_slot), n_slots, _ptr(codes),
                                     _ptr(scales), _ptr(err_flag), _stream(stream)))


def csa2_rope_quantize_kv_fp4(kv, pos, cos_sin, codes, scales, dst_slot=None, err_flag=None, stream=None):
    """Pre-RoPE kv bf16 [R, D] (or int16 bits), pos int32 [R], cos_sin fp32
    [n_pos, rope_dim/2, 2] -> codes uint8 [S, D/2], scales uint8 [S, D/16]."""
    _cuda(kv, pos, cos_sin, codes, scales, dst_slot, err_flag)
    R, D = kv.shape
    _plane_args(kv, codes, scales, dst_slot, err_flag, R, D, codes.shape[0])
    _elem(pos, "pos", (4,), False)
    _elem(cos_sin, "cos_sin", (4,), True)
    _room(pos, "pos", R)
    if cos_sin.dim() != 3 or cos_sin.shape[2] != 2:
        raise ValueError("cos_sin must be [n_pos, rope_dim/2, 2], got %s" % (tuple(cos_sin.shape),))
    n_pos, half = cos_sin.shape[0], cos_sin.shape[1]
    _check(_lib.csa2_rope_quantize_kv_fp4(_ptr(kv), R, D, D, _ptr(pos), _ptr(cos_sin), n_pos, 2 * half,
                                          _ptr(dst_slot), codes.shape[0], _ptr(codes), _ptr(scales),
                                          _ptr(err_flag), _stream(stream)))


def csa2_index_score(mode, q_idx, w, k_idx, kv_len, scores, pool_blocks=None, err_flag=None, stream=None):
    """q_idx [B,T,4,64], w fp32 [B,T,4], k_idx [B,N,64], kv_len int32 [B*T] ->
    scores fp32 [B,T,N] (FULL) or [B,T,8P] (REINDEX)."""
    _cuda(q_idx, w, k_idx, kv_len, scores, pool_blocks, err_flag)
    B, T = q_idx.shape[0], q_idx.shape[1]
    N = k_idx.shape[1]
    P = 0 if pool_blocks is None else pool_blocks.shape[-1]
    if int(mode) != MODE_REUSE:
        _indexer_operands(q_idx, w, k_idx, kv_len, B, T, N)
        _elem(scores, "scores", (4,), True)
        _elem(pool_blocks, "pool_blocks", (4,), False)
        _flag(err_flag)
        _room(scores, "scores", B * T * (8 * P if int(mode) == MODE_REINDEX else N))
        _room(pool_blocks, "pool_blocks", B * T * P)
    _check(_lib.csa2_index_score(int(mode), B, T, N, _ptr(q_idx), _dtype_code(q_idx), _ptr(w), _ptr(k_idx),
                                 _dtype_code(k_idx), _ptr(kv_len), _ptr(pool_blocks), P, _ptr(scores),
                                 _ptr(err_flag), _stream(stream)))


def csa2_build_pool(scores, kv_len, pool_blocks, workspace=None, stream=None):
    """scores fp32 [B,T,N], kv_len int32 [B*T] -> pool_blocks int32 [B,T,P]."""
    _cuda(scores, kv_len, pool_blocks, workspace)
    B, T, N = scores.shape
    P = pool_blocks.shape[-1]
    _elem(scores, "scores", (4,), True)
    _elem(kv_len, "kv_len", (4,), False)
    _elem(pool_blocks, "pool_blocks", (4,), False)
    _room(kv_len, "kv_len", B * T)
    _room(pool_blocks, "pool_blocks", B * T * P)
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.csa2_build_pool(B, T, N, _ptr(scores), _ptr(kv_len), P, POOL_BLOCK, _ptr(pool_blocks),
                                _ptr(workspace), ws, _stream(stream)))


def csa2_topk(mode, scores, idx, kv_len=None, pool_blocks=None, workspace=None, stream=None):
    """scores fp32 [B,T,M] -> idx int32 [B,T,K]."""
    _cuda(scores, idx, kv_len, pool_blocks, workspace)
    B, T, M = scores.shape
    K = idx.shape[-1]
    P = 0 if pool_blocks is None else pool_blocks.shape[-1]
    if int(mode) != MODE_REUSE:
        _elem(scores, "scores", (4,), True)
        for t, name in ((idx, "idx"), (kv_len, "kv_len"), (pool_blocks, "pool_blocks")):
            _elem(t, name, (4,), False)
        _room(idx, "idx", B * T * K)
        _room(kv_len, "kv_len", B * T)
        _room(pool_blocks, "pool_blocks", B * T * P)
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.csa2_topk(int(mode), B, T, M, _ptr(scores), _ptr(kv_len), _ptr(pool_blocks), P, K, _ptr(idx),
                          _ptr(workspace), ws, _stream(stream)))


def csa2_index_topk(mode, q_idx, w, k_idx, kv_len, idx, pool_blocks=None, pool_out=None, err_flag=None,
                    stream=None):
    """Fused decode indexer (FP8): the scores of csa2_index_score feed the
    Top-K of csa2_topk (and, for FULL with pool_out, the pool of
    csa2_build_pool) without being written out.  q_idx [B,T,4,64], w fp32
    [B,T,4], k_idx [B,N,64], kv_len int32 [B*T] -> idx int32 [B,T,K]
    (+ pool_out int32 [B,T,P_out])."""
    _cuda(q_idx, w, k_idx, kv_len, idx, pool_blocks, pool_out, err_flag)
    B, T = q_idx.shape[0], q_idx.shape[1]
    N = k_idx.shape[1]
    P = 0 if pool_blocks is None else pool_blocks.shape[-1]
    P_out = 0 if pool_out is None else pool_out.shape[-1]
    if int(mode) != MODE_REUSE:
        if q_idx.element_size() == 1 and k_idx.element_size() == 1:   # other dtypes: rejected by the call
            _indexer_operands(q_idx, w, k_idx, kv_len, B, T, N)
        for t, name in ((idx, "idx"), (pool_blocks, "pool_blocks"), (pool_out, "pool_out")):
            _elem(t, name, (4,), False)
        _flag(err_flag)
        _room(idx, "idx", B * T * idx.shape[-1])
        _room(pool_blocks, "pool_blocks", B * T * P)
        _room(pool_out, "pool_out", B * T * P_out)
    _check(_lib.csa2_index_topk(int(mode), B, T, N, _ptr(q_idx), _dtype_code(q_idx), _ptr(w), _ptr(k_idx),
                                _dtype_code(k_idx), _ptr(kv_len), _ptr(pool_blocks), P, idx.shape[-1], _ptr(idx),
                                _ptr(pool_out), P_out, _ptr(err_flag), _stream(stream)))


def csa2_index_topk_dense_workspace_bytes(B, T, N, K) -> int:
    return int(_lib.csa2_index_topk_dense_workspace_bytes(B, T, N, K))


def csa2_index_topk_dense(q_idx, w, k_idx, kv_len, idx, workspace=None, err_flag=None, stream=None):
    """Fused dense indexer for many query tokens (FP8, Full mode): the Top-K
    of csa2_index_score's scores, as csa2_topk selects it, without the score
    matrix.  q_idx [B,T,4,64], w fp32 [B,T,4], k_idx [B,N,64], kv_len int32
    [B*T] -> idx int32 [B,T,K].  workspace: a CUDA byte tensor of at least
    csa2_index_topk_dense_workspace_bytes(B, T, N, K) bytes (allocated here
    when None)."""
    _cuda(q_idx, w, k_idx, kv_len, idx, workspace, err_flag)
    B, T = q_idx.shape[0], q_idx.shape[1]
    N, K = k_idx.shape[1], idx.shape[-1]
    if q_idx.element_size() == 1 and k_idx.element_size() == 1:       # other dtypes: rejected by the call
        _indexer_operands(q_idx, w, k_idx, kv_len, B, T, N)
    _elem(idx, "idx", (4,), False)
    _flag(err_flag)
    _room(idx, "idx", B * T * K)
    if workspace is None:
        workspace = torch.empty(max(1, csa2_index_topk_dense_workspace_bytes(B, T, N, K)), dtype=torch.uint8,
                                device=idx.device)
    ws = workspace.numel() * workspace.element_size()
    _check(_lib.csa2_index_topk_dense(B, T, N, _ptr(q_idx), _dtype_code(q_idx), _ptr(w), _ptr(k_idx),
                                      _dtype_code(k_idx), _ptr(kv_len), K, _ptr(idx), _ptr(err_flag),
                                      _ptr(workspace), ws, _stream(stream)))


def csa2_swa_attn_fp8(q, swa_kv, swa_len, out, sm_scale, o_sparse=None, lse_sparse=None, lse=None, err_flag=None,
                      stream=None):
    """Sliding-window branch: q bf16 [B,T,H,D], swa_kv E4M3 [B,W,D] (uint8 or
    float8_e4m3fn), swa_len int32 [B*T] -> out fp32 [B,T,H,dv] (and lse),
    merged with (o_sparse, lse_sparse) when given; out may be o_sparse."""
    _cuda(q, swa_kv, swa_len, out, o_sparse, lse_sparse, lse, err_flag)
    B, T, H, D = q.shape
    W = swa_kv.shape[1]
    dv = out.shape[-1]
    _bf16(q, "q")
    _elem(swa_kv, "swa_kv", (1,))
    _elem(swa_len, "swa_len", (4,), False)
    for t, name in ((out, "out"), (o_sparse, "o_sparse"), (lse_sparse, "lse_sparse"), (lse, "lse")):
        _elem(t, name, (4,), True)
    _flag(err_flag)
    _room(swa_kv, "swa_kv", B * W * D)
    _room(swa_len, "swa_len", B * T)
    _room(out, "out", B * T * H * dv)
    _room(o_sparse, "o_sparse", B * T * H * dv)
    _room(lse_sparse, "lse_sparse", B * T * H)
    _room(lse, "lse", B * T * H)
    _check(_lib.csa2_swa_attn_fp8(B, T, H, D, out.shape[-1], _ptr(q), _ptr(swa_kv), W, _ptr(swa_len),
                                  float(sm_scale), _ptr(o_sparse), _ptr(lse_sparse), _ptr(out), _ptr(lse),
                                  _ptr(err_flag), _stream(stream)))


def csa2_sparse_attn_workspace_bytes(B, T, H, D, dv, K) -> int:
    return int(_lib.csa2_sparse_attn_workspace_bytes(B, T, H, D, dv, K))


def _attn_args(q, codes, scales, N, idx, out, kv_len, lse, err_flag, B, T, H, D, dv, K):
    _bf16(q, "q")
    _elem(codes, "codes", (1,))
    _elem(scales, "scales", (1,))
    _elem(idx, "idx", (4,), False)
    _elem(kv_len, "kv_len", (4,), False)
    _elem(out, "out", (4,), True)
    _elem(lse, "lse", (4,), True)
    _flag(err_flag)
    _room(codes, "codes", B * int(N) * (D // 2))
    _room(scales, "scales", B * int(N) * (D // 16))
    _room(idx, "idx", B * T * K)
    _room(kv_len, "kv_len", B * T)
    _room(out, "out", B * T * H * dv)
    _room(lse, "lse", B * T * H)


def csa2_sparse_attn_fp4(mode, q, codes, scales, N, idx, out, sm_scale, kv_len=None, lse=None, err_flag=None,
                         workspace=None, stream=None):
    """q bf16 [B,T,H,D]; codes [B*N, D/2], scales [B*N, D/16]; idx int32
    [B,T,K] -> out fp32 [B,T,H,dv], lse fp32 [B,T,H] (optional)."""
    _cuda(q, codes, scales, idx, out, kv_len, lse, err_flag, workspace)
    B, T, H, D = q.shape
    dv = out.shape[-1]
    K = idx.shape[-1]
    _attn_args(q, codes, scales, N, idx, out, kv_len, lse, err_flag, B, T, H, D, dv, K)
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.csa2_sparse_attn_fp4(int(mode), B, T, H, D, dv, _ptr(q), _ptr(codes), _ptr(scales), int(N),
                                     _ptr(idx), K, _ptr(kv_len), float(sm_scale), _ptr(out), FP32, _ptr(lse),
                                     _ptr(err_flag), _ptr(workspace), ws, _stream(stream)))


def csa2_sparse_attn_fp4_prefetch(mode, q, codes, scales, N, idx, out, sm_scale, next_codes=None, next_scales=None,
                                  kv_len=None, lse=None, err_flag=None, workspace=None, stream=None):
    """csa2_sparse_attn_fp4 plus an L2 prefetch hint: the rows idx selects in
    (next_codes, next_scales), the planes of the layer that attends next with
    the same indices."""
    _cuda(q, codes, scales, idx, out, kv_len, lse, err_flag, workspace, next_codes, next_scales)
    B, T, H, D = q.shape
    dv = out.shape[-1]
    K = idx.shape[-1]
    _attn_args(q, codes, scales, N, idx, out, kv_len, lse, err_flag, B, T, H, D, dv, K)
    if (next_codes is None) != (next_scales is None):
        raise ValueError("next_codes and next_scales go together")
    if next_codes is not None:
        _elem(next_codes, "next_codes", (1,))
        _elem(next_scales, "next_scales", (1,))
        _room(next_codes, "next_codes", B * int(N) * (D // 2))
        _room(next_scales, "next_scales", B * int(N) * (D // 16))
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.csa2_sparse_attn_fp4_prefetch(int(mode), B, T, H, D, dv, _ptr(q), _ptr(codes), _ptr(scales), int(N),
                                              _ptr(idx), K, _ptr(kv_len), float(sm_scale), _ptr(out), FP32,
                                              _ptr(lse), _ptr(err_flag), _ptr(workspace), ws, _ptr(next_codes),
                                              _ptr(next_scales), _stream(stream)))


def workspace_for_attn(B, T, H, D, dv, K, device="cuda"):
    """Allocate (through torch) the scratch csa2_sparse_attn_fp4 needs, or None."""
    n = csa2_sparse_attn_workspace_bytes(B, T, H, D, dv, K)
    return None if n == 0 else torch.empty(n, dtype=torch.uint8, device=device)


def csa2_sparse_attn_fp4_noalloc(mode, q, codes, scales, N, idx, out, sm_scale, kv_len=None, lse=None,
                                 err_flag=None, stream=None):
    """csa2_sparse_attn_fp4 for callers that may not allocate device memory:
    the split-KV scratch is the library's built-in array (see the header)."""
    _cuda(q, codes, scales, idx, out, kv_len, lse, err_flag)
    B, T, H, D = q.shape
    dv = out.shape[-1]
    K = idx.shape[-1]
    _attn_args(q, codes, scales, N, idx, out, kv_len, lse, err_flag, B, T, H, D, dv, K)
    _check(_lib.csa2_sparse_attn_fp4_noalloc(int(mode), B, T, H, D, dv, _ptr(q), _ptr(codes), _ptr(scales), int(N),
                                             _ptr(idx), K, _ptr(kv_len), float(sm_scale), _ptr(out), FP32,
                                             _ptr(lse), _ptr(err_flag), _stream(stream)))


def noalloc_max_scratch_bytes() -> int:
    return int(_lib.csa2_sparse_attn_noalloc_max_scratch_bytes())
