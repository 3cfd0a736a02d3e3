"""One decode step of the CSA2 decoder layers, as a sequence of libcsa2 calls.

The layer schedule is the decoder's as the pages give it ("DeepSeek-V4.1-Flash：
把 KV Cache 压缩到极限的百万上下文 MoE", CSA2 section): 20 layers in 5 groups of
4, the first group 1 Full + 3 Reuse, the other four 1 Reindex + 3 Reuse, Top-512
everywhere; the first Full layer also builds the hierarchical candidate pool
("Hierarchical Sparse Indexer") that the Reindex layers score inside.

This module owns no arithmetic: it allocates the device buffers (through
torch), then issues the calls of the C library in order on one stream, so the
whole step can be captured in a CUDA graph.  Per step:
  1. csa2_quantize_kv_fp4 appends each KV-owning layer's new post-RoPE row for
     every sequence (one launch for all layers);
  2. per group: the Full layer scores all entries, builds the pool and takes
     its Top-512; a Reindex layer scores the pool with its own indexer query
     against the Full layer's index keys and takes its Top-512 (with FP8
     indexer tensors each of these is one fused csa2_index_topk call, the
     scores staying on chip; otherwise csa2_index_score, csa2_build_pool and
     csa2_topk);
  3. every layer attends over its FP4 KV with its group's indices (Reuse
     layers consume the group's index buffer unchanged).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from gen import DECODER_SCHEDULE  # the schedule as a workload constant (no arithmetic)

from . import (MODE_FULL, MODE_REINDEX, MODE_REUSE, csa2_build_pool, csa2_index_score, csa2_index_topk,
               csa2_quantize_kv_fp4, csa2_sparse_attn_fp4, csa2_sparse_attn_fp4_prefetch, csa2_topk,
               workspace_for_attn)


@dataclass
class StepShape:
    B: int
    N: int
    D: int = 576
    dv: int = 512
    H: int = 64
    K: int = 512
    P: int = 2048
    idx_fp8: bool = True
    kv_per_layer: bool = True        # each layer attends over its own FP4 KV
    fused_indexer: bool = True       # FP8 only: csa2_index_topk instead of score + pool + topk
    prefetch_next: bool = True       # a layer followed by a Reuse layer hints that layer's selected rows into L2
    schedule: tuple = DECODER_SCHEDULE


class DecoderStep:
    """Device buffers and call sequence for one decode step (T = 1 query token
    per sequence).  Inputs live in ``self.inputs``; outputs in ``self.out``
    and ``self.lse`` (one per layer)."""

    def __init__(self, shape: StepShape, device="cuda"):
        s = self.shape = shape
        dev = self.device = torch.device(device)
        L = len(s.schedule)
        assert s.schedule[0] == "full"
        self.L = L
        self.groups = [i for i, m in enumerate(s.schedule) if m != "reuse"]
        self.n_kv = L if s.kv_per_layer else 1
        R = self.n_kv * s.B * s.N
        self.codes = torch.zeros(R, s.D // 2, dtype=torch.uint8, device=dev)
        self.scales = torch.zeros(R, s.D // 16, dtype=torch.uint8, device=dev)
        idt = torch.uint8 if s.idx_fp8 else torch.int16
        self.k_idx = torch.zeros(s.B, s.N, 64, dtype=idt, device=dev)
        self.kv_len = torch.zeros(s.B, dtype=torch.int32, device=dev)
        # per-step inputs
        self.inputs = {
            "q": torch.zeros(L, s.B, 1, s.H, s.D, dtype=torch.int16, device=dev),
            "q_idx": torch.zeros(len(self.groups), s.B, 1, 4, 64, dtype=idt, device=dev),
            "w_idx": torch.zeros(len(self.groups), s.B, 1, 4, dtype=torch.float32, device=dev),
            "new_rows": torch.zeros(self.n_kv * s.B, s.D, dtype=torch.int16, device=dev),
            "new_slots": torch.zeros(self.n_kv * s.B, dtype=torch.int64, device=dev),
        }
        self.scores = torch.empty(s.B, 1, s.N, dtype=torch.float32, device=dev)
        self.rscores = torch.empty(s.B, 1, 8 * s.P, dtype=torch.float32, device=dev)
        self.pool = torch.empty(s.B, 1, s.P, dtype=torch.int32, device=dev)
        self.idx = torch.empty(len(self.groups), s.B, 1, s.K, dtype=torch.int32, device=dev)
        self.out = torch.empty(L, s.B, 1, s.H, s.dv, dtype=torch.float32, device=dev)
        self.lse = torch.empty(L, s.B, 1, s.H, dtype=torch.float32, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.ws = workspace_for_attn(s.B, 1, s.H, s.D, s.dv, s.K, device=dev)
        self.sm_scale = 1.0 / float(s.D) ** 0.5

    @property
    def token_layers(self) -> int:
        return self.shape.B * self.L

    def kv_planes(self, layer: int):
        s = self.shape
        kv = layer if s.kv_per_layer else 0
        r0 = kv * s.B * s.N
        return self.codes[r0:r0 + s.B * s.N], self.scales[r0:r0 + s.B * s.N]

    def set_append_slots(self):
        """Append slot of every KV-owning layer's new row: the entry kv_len-1
        of each sequence (the step completes a 4-token chunk)."""
        s = self.shape
        b = torch.arange(s.B, device=self.device, dtype=torch.int64)
        last = self.kv_len.to(torch.int64) - 1
        slots = [(kv * s.B + b) * s.N + last for kv in range(self.n_kv)]
        self.inputs["new_slots"].copy_(torch.cat(slots))

    def run(self, stream=None):
        s = self.shape
        x = self.inputs
        csa2_quantize_kv_fp4(x["new_rows"], self.codes, self.scales, dst_slot=x["new_slots"], err_flag=self.err,
                             stream=stream)
        gi = -1
        fused = s.fused_indexer and s.idx_fp8
        L = len(s.schedule)
        for layer, mode in enumerate(s.schedule):
            if mode != "reuse" and fused:
                gi += 1
                if mode == "full":
                    csa2_index_topk(MODE_FULL, x["q_idx"][gi], x["w_idx"][gi], self.k_idx, self.kv_len, self.idx[gi],
                                    pool_out=self.pool if layer == 0 else None, err_flag=self.err, stream=stream)
                else:
                    csa2_index_topk(MODE_REINDEX, x["q_idx"][gi], x["w_idx"][gi], self.k_idx, self.kv_len,
                                    self.idx[gi], pool_blocks=self.pool, err_flag=self.err, stream=stream)
            elif mode != "reuse":
                gi += 1
                if mode == "full":
                    csa2_index_score(MODE_FULL, x["q_idx"][gi], x["w_idx"][gi], self.k_idx, self.kv_len,
                                     self.scores, err_flag=self.err, stream=stream)
                    if layer == 0:
                        csa2_build_pool(self.scores, self.kv_len, self.pool, stream=stream)
                    csa2_topk(MODE_FULL, self.scores, self.idx[gi], kv_len=self.kv_len, stream=stream)
                else:
                    csa2_index_score(MODE_REINDEX, x["q_idx"][gi], x["w_idx"][gi], self.k_idx, self.kv_len,
                                     self.rscores, pool_blocks=self.pool, err_flag=self.err, stream=stream)
                    csa2_topk(MODE_REINDEX, self.rscores, self.idx[gi], pool_blocks=self.pool, stream=stream)
            else:
                # Reuse: no indexer, no selection -- the group's idx buffer as is
                csa2_topk(MODE_REUSE, self.scores, self.idx[gi], stream=stream)
            codes, scales = self.kv_planes(layer)
            mode_id = {"full": MODE_FULL, "reindex": MODE_REINDEX, "reuse": MODE_REUSE}[mode]
            nxt = layer + 1
            if s.prefetch_next and s.kv_per_layer and nxt < L and s.schedule[nxt] == "reuse":
                # the next layer attends with this group's idx over its own planes
                nc, ns = self.kv_planes(nxt)
                csa2_sparse_attn_fp4_prefetch(mode_id, x["q"][layer], codes, scales, s.N, self.idx[gi],
                                              self.out[layer], self.sm_scale, next_codes=nc, next_scales=ns,
                                              kv_len=self.kv_len, lse=self.lse[layer], err_flag=self.err,
                                              workspace=self.ws, stream=stream)
            else:
                csa2_sparse_attn_fp4(mode_id, x["q"][layer], codes, scales, s.N, self.idx[gi], self.out[layer],
                                     self.sm_scale, kv_len=self.kv_len, lse=self.lse[layer], err_flag=self.err,
                                     workspace=self.ws, stream=stream)

    def launches_per_step(self) -> int:
        """Kernel launches of one step (Reuse-mode scoring/selection launch nothing)."""
        s = self.shape
        split = self.ws is not None
        n = 1                                              # quantise
        fused = s.fused_indexer and s.idx_fp8
        L = len(s.schedule)
        for layer, mode in enumerate(s.schedule):
            if mode != "reuse" and fused:
                n += 1                                     # fused score + (pool) + topk
            elif mode == "full":
                n += 2 + (1 if layer == 0 else 0)         # score, topk (+ pool)
            elif mode == "reindex":
                n += 2
            n += 2 if split else 1                         # attention (+ combine)
        return n
