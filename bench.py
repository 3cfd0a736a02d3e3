#!/usr/bin/env python
"""Benchmark: decode steps of the CSA2 decoder over an FP4 main KV cache.

Workload (the batched Full-mode decode shapes): 32 sequences with
L_b ~ U{32768..65536} tokens (n_b = L_b/4 compressed entries, capacity
16384), 576-channel FP4 entries (512 latent + 64 RoPE), 64 query heads, FP8
indexer 4 x 64, Top-512, pool of 2048 x 8.  One step is one decode token
through the decoder's 20 CSA2 layers as the pages schedule them (group 0: 1
Full + 3 Reuse; groups 1-4: 1 Reindex + 3 Reuse), so every row of the path
runs each step: FP4 append (quantise), Full scoring, pool build, Reindex
scoring, Top-512, sparse FP4 attention, Reuse.  Each layer attends over its
own FP4 KV (the worst case for bytes).

Metric: CSA2 decode token-layers per second (B x 20 per step), plus the
dominant kernel's achieved HBM bandwidth against the measured GB300 copy
bandwidth.  Inputs are resident in HBM; four disjoint input sets rotate so no
step finds the previous step's data in L2.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode CSA2 token-layers/s (B x layers per decode step)"
UNIT = "token-layers/s"
B, NCAP, D, DV, H, K, P = 32, 16384, 576, 512, 64, 512, 2048
LAYERS = 20
ROTATE = 4


def _workload_config(extra=None):
    cfg = {"workload": "csa2_decoder_step_b32_ctx32k-64k_n16384_d576_h64_top512_pool2048x8_20layers",
           "batch": B, "entries_cap": NCAP, "D": D, "dv": DV, "heads": H, "topk": K, "pool_blocks": P,
           "layers": LAYERS, "schedule": "1Full+3Reuse, 4x(1Reindex+3Reuse)", "kv": "FP4 E2M1 + E4M3/16, per layer",
           "indexer": "FP8 E4M3 4x64, fused score->pool->Top-512 (scores stay on chip)", "l2": "4 rotating disjoint input sets, each step's working set > L2"}
    if extra:
        cfg.update(extra)
    return cfg


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _bf16_peak_tflops():
    """Measured dense bf16 burst rate (cuBLAS) from MEASURED_PEAKS.json, else
    the fallback 1900 TFLOP/s."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        if j.get("bf16_tflops"):
            return float(j["bf16_tflops"])
    return 1900.0


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _rank_seed(rank, r):
    """Seed of input set r on `rank`: every rank serves its own sequences, so
    the work per GPU is fixed as ranks are added (weak scaling)."""
    return 1 + 1000 * rank + 17 * r


def _max_over_ranks(sec, device=None):
    """The slowest rank's seconds, on every rank (the job ends with it); the
    value itself with one rank or no process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(sec)
    dev = device if (device is not None and dist.get_backend() == "nccl") else "cpu"
    t = torch.tensor([float(sec)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _job_rate(units_per_rank_step, steps, world, sec):
    """Whole-job throughput: the units all ranks processed over the slowest
    rank's time."""
    return units_per_rank_step * steps * world / sec


class ClockSampler:
    """nvidia-smi clocks/throttle sampling in the background (100 ms)."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for ln in self.proc.stdout:
            self.samples.append((time.time(), ln.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = []
        for ts, ln in self.samples:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((ts, float(f[1]), float(f[2]), f[5:9]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 <= r[0] <= t1]
        if not inside and rows:  # timed region shorter than the sampling period: nearest samples
            inside = sorted(rows, key=lambda r: min(abs(r[0] - t0), abs(r[0] - t1)))[:3]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside)}


# ------------------------------------------------------------------ GPU arm
def _fill_instance(st, seed):
    import torch
    import gen
    w = gen.scaled(gen.FULL_BATCHED_DECODE, seed=seed)
    dev = st.device
    st.kv_len.copy_(gen.kv_lengths(w).to(dev))
    for layer in range(st.n_kv):
        rows = gen.kv_rows(seed, 100 + layer, B * NCAP, D, rms=True, device=dev)
        c, s = st.kv_planes(layer)
        import sparse_attention_fp4_quantize_gb300 as csa2
        csa2.csa2_quantize_kv_fp4(rows, c, s)
        del rows
    st.k_idx.copy_(gen.normal_e4m3(seed, 19, (B, NCAP, 64), device=dev))
    for gi in range(len(st.groups)):
        st.inputs["q_idx"][gi].copy_(gen.normal_e4m3(seed, 20 + 3 * gi, (B, 1, 4, 64), device=dev))
        st.inputs["w_idx"][gi].copy_(gen.uniform01(seed, 21 + 3 * gi, (B, 1, 4), device=dev))
    for layer in range(LAYERS):
        st.inputs["q"][layer].copy_(gen.normal_bf16(seed, 200 + layer, (B, 1, H, D), device=dev))
    st.inputs["new_rows"].copy_(gen.kv_rows(seed, 70, st.n_kv * B, D, device=dev))
    st.set_append_slots()
    torch.cuda.synchronize()


def _algorithmic_bytes(st):
    """Indexer keys read + selected FP4 entries gathered + outputs, per step."""
    import torch
    n = st.kv_len.to(torch.int64)
    keys_full = int(n.sum()) * 64
    # Reindex layers score the pool's candidates: min(n, 8 * 2048) keys per sequence
    keys_re = int(torch.clamp(n, max=8 * P).sum()) * 64
    n_full = sum(1 for m in st.shape.schedule if m == "full")
    n_re = sum(1 for m in st.shape.schedule if m == "reindex")
    gathered = LAYERS * B * K * (D // 2 + D // 16)
    outputs = LAYERS * B * H * DV * 4
    return {"keys": keys_full * n_full + keys_re * n_re, "gathered": gathered, "outputs": outputs,
            "attn_per_launch": B * K * (D // 2 + D // 16) + B * H * DV * 4}


def _kernel_breakdown(steps, stream, rounds):
    """Device time per launch of each kernel kind, with CUDA events on the
    launching stream: for every input set, a CUDA graph holding only that
    kind's launches of one decode step (the other calls are left out; their
    output buffers still hold the previous step's valid data) is replayed
    ``rounds`` times in rotation between two events."""
    import torch
    import sparse_attention_fp4_quantize_gb300 as csa2
    import sparse_attention_fp4_quantize_gb300.decode as dec
    kinds = {"quantize": ("csa2_quantize_kv_fp4",), "index_score": ("csa2_index_score",),
             "build_pool": ("csa2_build_pool",), "topk": ("csa2_topk",), "index_topk": ("csa2_index_topk",),
             "sparse_attn": ("csa2_sparse_attn_fp4", "csa2_sparse_attn_fp4_prefetch")}
    orig = {fn: getattr(dec, fn) for names in kinds.values() for fn in names}
    out = {}
    for kind, keep in kinds.items():
        count, dry = [0], [True]

        def make(fn_name, fn):
            def inner(*a, **kw):
                if fn_name not in keep:
                    return None
                if fn_name in ("csa2_index_score", "csa2_topk", "csa2_index_topk") and a[0] == csa2.MODE_REUSE:
                    return None if dry[0] else fn(*a, **kw)          # no launch
                count[0] += 1
                return None if dry[0] else fn(*a, **kw)
            return inner

        for fn_name, fn in orig.items():
            setattr(dec, fn_name, make(fn_name, fn))
        try:
            # count this kind's calls first (nothing launched): a kind the
            # step never calls gets no (empty) graph
            steps[0].run(stream=stream)
            if count[0] == 0:
                continue
            dry[0] = False
            graphs = []
            for st in steps:
                count[0] = 0
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    st.run(stream=stream)
                graphs.append(g)
            per_graph = count[0]
        finally:
            for fn_name, fn in orig.items():
                setattr(dec, fn_name, fn)
        if per_graph == 0:
            continue
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for i in range(len(graphs)):
                graphs[i].replay()
            e0.record(stream)
            for i in range(rounds):
                graphs[i % len(graphs)].replay()
            e1.record(stream)
        torch.cuda.synchronize()
        sec = e0.elapsed_time(e1) * 1e-3
        out[kind] = {"launches_per_step": per_graph, "avg_s": sec / (rounds * per_graph),
                     "total_s_per_step": sec / rounds}
    return out


def _traffic_record(kernel):
    """DRAM bytes per launch from the committed ncu summary, valid only while
    the kernel's source is unchanged."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f).get(kernel)
    if not rec:
        return None
    src = os.path.join(ROOT, rec["source"])
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] if os.path.exists(src) else None
    if h != rec.get("source_sha256_16"):
        return None
    return rec.get("dram_bytes_per_launch")


def _time_graph(fn, stream, reps, warm=3):
    """Capture fn() as a CUDA graph on `stream`, replay it `warm` times, then
    time `reps` replays with events; seconds per replay."""
    import torch
    with torch.cuda.stream(stream):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    with torch.cuda.stream(stream):
        for _ in range(warm):
            g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e-3 / reps


def _extra_workloads(dev, stream, peak_gbs):
    """The other synthetic workloads, each timed on the device: the 1M-row FP4
    append, the 4096-query prefill scoring, the Reindex + 3 Reuse group at 1M
    context, the pool build, and the tiny Full-layer chain."""
    import torch
    import gen
    import sparse_attention_fp4_quantize_gb300 as csa2
    res = {}
    # append: quantise 1,048,576 x 576 rows (two output sets alternate; the 1.2 GB input exceeds L2)
    w5 = gen.APPEND_POOL
    R = w5.B * w5.N
    rows = gen.kv_rows(w5.seed, 10, R, 576, rms=False, device=dev)
    outs = [(torch.empty(R, 288, dtype=torch.uint8, device=dev), torch.empty(R, 36, dtype=torch.uint8, device=dev))
            for _ in range(2)]
    t = _time_graph(lambda: [csa2.csa2_quantize_kv_fp4(rows, c, s_, stream=stream) for c, s_ in outs], stream, 20) / 2
    qbytes = R * 576 * 2 + R * (288 + 36)
    res["append_quantize_1m_rows"] = {"us": t * 1e6, "bytes": qbytes, "gbs": qbytes / t / 1e9,
                                     "hbm_frac": qbytes / t / 1e9 / peak_gbs}
    # the same append from pre-RoPE rows: RoPE (fp32 table of 131072 positions) fused ahead of the quantiser
    tab = gen.rope_table(131072, device=dev)
    pos = torch.randint(0, 131072, (R,), generator=torch.Generator(device=dev).manual_seed(7), device=dev,
                        dtype=torch.int32)
    t = _time_graph(lambda: [csa2.csa2_rope_quantize_kv_fp4(rows, pos, tab, c, s_, stream=stream)
                             for c, s_ in outs], stream, 20) / 2
    rbytes = qbytes + R * 4
    res["append_rope_quantize_1m_rows"] = {"us": t * 1e6, "bytes": rbytes, "gbs": rbytes / t / 1e9,
                                          "hbm_frac": rbytes / t / 1e9 / peak_gbs}
    del rows, outs, tab, pos
    # decode rows: Top-512 of 32 rows x 16384 scores, csa2_topk against torch.topk
    w2 = gen.FULL_BATCHED_DECODE
    q2, ww2, k2 = gen.indexer_inputs(w2, device=dev)
    kl2 = gen.kv_lengths(w2).to(dev)
    sc2 = torch.empty(w2.B, 1, w2.N, device=dev)
    csa2.csa2_index_score(0, q2, ww2, k2, kl2, sc2, stream=stream)
    i2 = torch.empty(w2.B, 1, 512, dtype=torch.int32, device=dev)
    t_c = _time_graph(lambda: csa2.csa2_topk(0, sc2, i2, kv_len=kl2, stream=stream), stream, 50)
    v2 = torch.empty(w2.B, 1, 512, device=dev)
    x2 = torch.empty(w2.B, 1, 512, dtype=torch.int64, device=dev)
    t_t = _time_graph(lambda: torch.topk(sc2, 512, dim=2, out=(v2, x2)), stream, 50)
    res["topk_b32_n16384"] = {"csa2_us": t_c * 1e6, "torch_topk_us": t_t * 1e6, "csa2_topk_speedup": t_t / t_c}
    del q2, ww2, k2, sc2, i2, v2, x2
    # pool for 16 x 65536 entries from Full scores
    q5, w5w, k5 = gen.indexer_inputs(w5, device=dev)
    kl5 = gen.kv_lengths(w5).to(dev)
    sc5 = torch.empty(w5.B, 1, w5.N, device=dev)
    csa2.csa2_index_score(0, q5, w5w, k5, kl5, sc5, stream=stream)
    pool5 = torch.empty(w5.B, 1, 2048, dtype=torch.int32, device=dev)
    t = _time_graph(lambda: csa2.csa2_build_pool(sc5, kl5, pool5, stream=stream), stream, 50)
    res["pool_build_b16_n65536"] = {"us": t * 1e6, "score_bytes_read": w5.B * w5.N * 4}
    t = _time_graph(lambda: csa2.csa2_index_score(0, q5, w5w, k5, kl5, sc5, stream=stream), stream, 20)
    res["full_score_b16_n65536"] = {"us": t * 1e6, "key_gbs": w5.B * w5.N * 64 / t / 1e9,
                                    "hbm_frac": w5.B * w5.N * 68 / t / 1e9 / peak_gbs}
    del q5, w5w, k5, sc5
    # prefill: 4096 causal queries x 32768 keys (FP8), scores materialised
    w4 = gen.PREFILL_CHUNK
    q4, ww4, k4 = gen.indexer_inputs(w4, device=dev)
    kl4 = gen.kv_lengths(w4).to(dev)
    sc4 = torch.empty(1, w4.T, w4.N, device=dev)
    t = _time_graph(lambda: csa2.csa2_index_score(0, q4, ww4, k4, kl4, sc4, stream=stream), stream, 5)
    flops = 2.0 * w4.T * 4 * 64 * w4.N
    res["prefill_score_t4096_n32768"] = {"us": t * 1e6, "tflops": flops / t / 1e12,
                                         "score_write_gbs": w4.T * w4.N * 4 / t / 1e9}
    idx4 = torch.empty(1, w4.T, 512, dtype=torch.int32, device=dev)
    t = _time_graph(lambda: csa2.csa2_topk(0, sc4, idx4, kv_len=kl4, stream=stream), stream, 5)
    res["prefill_topk_t4096_n32768"] = {"us": t * 1e6, "score_read_gbs": w4.T * w4.N * 4 / t / 1e9}
    # context for the pages' DeepSelect claim (2-20x over torch.topk, no hardware stated): torch.topk on the
    # same rows, here and on the decode rows below
    vals = torch.empty(1, w4.T, 512, device=dev)
    tix = torch.empty(1, w4.T, 512, dtype=torch.int64, device=dev)
    t = _time_graph(lambda: torch.topk(sc4, 512, dim=2, out=(vals, tix)), stream, 5)
    res["torch_topk_t4096_n32768"] = {"us": t * 1e6,
                                      "csa2_topk_speedup": t * 1e6 / res["prefill_topk_t4096_n32768"]["us"]}
    del vals, tix
    # the same Top-512 by the fused dense indexer (block maxima -> threshold -> candidates -> Top-K):
    # two tensor-core scoring passes, no score matrix
    ws4 = torch.empty(csa2.csa2_index_topk_dense_workspace_bytes(1, w4.T, w4.N, 512), dtype=torch.uint8, device=dev)
    idx4d = torch.empty(1, w4.T, 512, dtype=torch.int32, device=dev)
    t = _time_graph(lambda: csa2.csa2_index_topk_dense(q4, ww4, k4, kl4, idx4d, workspace=ws4, stream=stream),
                    stream, 10)
    fp8_peak = 2.0 * _bf16_peak_tflops()   # FP8 dense = 2 x the measured bf16 burst rate (nominal ratio)
    res["prefill_index_topk_dense_t4096_n32768"] = {
        "us": t * 1e6, "tflops": flops / t / 1e12, "passes": 2,
        "fp8_peak_tflops": fp8_peak, "fp8_peak_frac": flops / t / 1e12 / fp8_peak,
        "vs_unfused_us": res["prefill_score_t4096_n32768"]["us"] + res["prefill_topk_t4096_n32768"]["us"]}
    del ws4, idx4d
    # the chunk's attention: 4096 queries x 64 heads over their Top-512 of the FP4 cache
    c4, s4 = gen.fp4_planes(w4.seed, 50, w4.N, 576, device=dev)
    qa4 = gen.normal_bf16(w4.seed, 51, (1, w4.T, 64, 576), device=dev)
    oa4 = torch.empty(1, w4.T, 64, 512, device=dev)
    t = _time_graph(lambda: csa2.csa2_sparse_attn_fp4(0, qa4, c4, s4, w4.N, idx4, oa4, 1 / 24.0, kv_len=kl4,
                                                      stream=stream), stream, 5)
    aflops = 2.0 * w4.T * 64 * 512 * (576 + 512)
    res["prefill_attention_t4096_k512"] = {"us": t * 1e6, "tflops": aflops / t / 1e12}
    del q4, ww4, k4, sc4, idx4, c4, s4, qa4, oa4
    # Reindex + 3 Reuse group at 1M context, B = 8, each layer over its own FP4 KV
    w3 = gen.REINDEX_REUSE_1M
    q0, w0, k3 = gen.indexer_inputs(w3, layer=0, device=dev)
    q1, w1, _ = gen.indexer_inputs(w3, layer=1, device=dev)
    kl3 = gen.kv_lengths(w3).to(dev)
    full3 = torch.empty(w3.B, 1, w3.N, device=dev)
    csa2.csa2_index_score(0, q0, w0, k3, kl3, full3, stream=stream)
    pool3 = torch.empty(w3.B, 1, 2048, dtype=torch.int32, device=dev)
    csa2.csa2_build_pool(full3, kl3, pool3, stream=stream)
    idx3 = torch.empty(w3.B, 1, 512, dtype=torch.int32, device=dev)
    planes = [gen.fp4_planes(w3.seed, 40 + l, w3.B * w3.N, 576, device=dev) for l in range(4)]
    qs = [gen.normal_bf16(w3.seed, 200 + l, (w3.B, 1, 64, 576), device=dev) for l in range(4)]
    outs3 = [torch.empty(w3.B, 1, 64, 512, device=dev) for _ in range(4)]
    ws3 = csa2.workspace_for_attn(w3.B, 1, 64, 576, 512, 512, device=dev)

    def group():   # the fused Reindex indexer (score + Top-512 in the pool, one launch), as in the decode step
        csa2.csa2_index_topk(1, q1, w1, k3, kl3, idx3, pool_blocks=pool3, stream=stream)
        for l in range(4):   # the next Reuse layer's selected rows are hinted into L2 (as in the decode step)
            nxt = planes[l + 1] if l < 3 else (None, None)
            csa2.csa2_sparse_attn_fp4_prefetch(1 if l == 0 else 2, qs[l], planes[l][0], planes[l][1], w3.N, idx3,
                                               outs3[l], 1 / 24.0, next_codes=nxt[0], next_scales=nxt[1],
                                               kv_len=kl3, workspace=ws3, stream=stream)
    t = _time_graph(group, stream, 50)
    gbytes = w3.B * 16384 * 64 + 4 * w3.B * 512 * 324 + 4 * w3.B * 64 * 512 * 4
    res["reindex_reuse_group_b8_1m"] = {"us": t * 1e6, "token_layers_per_s": w3.B * 4 / t,
                                        "algorithmic_bytes": gbytes, "gbs": gbytes / t / 1e9}
    t = _time_graph(lambda: csa2.csa2_build_pool(full3, kl3, pool3, stream=stream), stream, 50)
    res["pool_build_b8_n262144"] = {"us": t * 1e6, "score_bytes_read": w3.B * w3.N * 4}
    del planes, qs, outs3, k3, full3
    torch.cuda.empty_cache()
    # sliding-window branch (FP8 window of 128 tokens) merged in place with a sparse-branch output, B=32
    qs_ = gen.normal_bf16(11, 1, (32, 1, 64, 576), device=dev)
    kvw = gen.e4m3_bytes(torch.randn(32, 128, 576, generator=torch.Generator(device=dev).manual_seed(3), device=dev))
    slw = torch.full((32,), 128, dtype=torch.int32, device=dev)
    osp = torch.randn(32, 1, 64, 512, device=dev)
    lsp = torch.randn(32, 1, 64, device=dev)
    t = _time_graph(lambda: csa2.csa2_swa_attn_fp8(qs_, kvw, slw, osp, 1 / 24.0, o_sparse=osp, lse_sparse=lsp,
                                                   lse=lsp, stream=stream), stream, 50)
    sb = 32 * 128 * 576 + 2 * 32 * 64 * 512 * 4
    res["swa_merge_b32_w128"] = {"us": t * 1e6, "algorithmic_bytes": sb, "gbs": sb / t / 1e9}
    del qs_, kvw, osp, lsp
    # attention alone at larger token counts (T=1 decode tokens, H=64, Top-512 of 16384 entries):
    # the same kernel once the launch holds more than one token per SM group; two
    # rotating input sets whose gathered rows exceed L2
    for nb in (128, 512):
        wa = gen.scaled(gen.FULL_BATCHED_DECODE, B=nb)
        kla = torch.full((nb,), 16384, dtype=torch.int32, device=dev)
        sets = []
        for r_ in range(2):
            codes, scales = gen.fp4_planes(wa.seed, 60 + r_, nb * 16384, 576, device=dev)
            qa = gen.normal_bf16(wa.seed, 70 + r_, (nb, 1, 64, 576), device=dev)
            ia = torch.randint(0, 16384, (nb, 1, 512), generator=torch.Generator(device=dev).manual_seed(80 + r_),
                               device=dev, dtype=torch.int32)
            oa = torch.empty(nb, 1, 64, 512, device=dev)
            sets.append((codes, scales, qa, ia, oa))
        t = _time_graph(lambda: [csa2.csa2_sparse_attn_fp4(2, qa_, c_, s_, 16384, ia_, oa_, 1 / 24.0, kv_len=kla,
                                                           stream=stream)
                                 for c_, s_, qa_, ia_, oa_ in sets], stream, 20) / 2
        ab = nb * 512 * 324 + nb * 64 * 512 * 4
        res["attention_b%d" % nb] = {"us": t * 1e6, "algorithmic_bytes": ab, "gbs": ab / t / 1e9,
                                     "hbm_frac": ab / t / 1e9 / peak_gbs}
        del sets
        torch.cuda.empty_cache()
    return res


def run_gpu(args):
    import torch
    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.device_count() >= world else "gloo")
    import sparse_attention_fp4_quantize_gb300 as csa2  # noqa: F401  (fails loudly without libcsa2.so)
    from sparse_attention_fp4_quantize_gb300.decode import DecoderStep, StepShape

    steps = []
    for r in range(ROTATE):
        st = DecoderStep(StepShape(B=B, N=NCAP, D=D, dv=DV, H=H, K=K, P=P), device=dev)
        _fill_instance(st, seed=_rank_seed(rank, r))
        steps.append(st)
    stream = torch.cuda.Stream(device=dev)
    # warm the library (attributes, module load) eagerly, then capture one graph per input set
    with torch.cuda.stream(stream):
        for st in steps:
            st.run(stream=stream)
    torch.cuda.synchronize()
    graphs = []
    for st in steps:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            st.run(stream=stream)
        graphs.append(g)
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # ---- device-resident timed region
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            graphs[i % ROTATE].replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(args.steps):
            graphs[i % ROTATE].replay()
        e1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier()
    time.sleep(0.15)
    clocks.stop()
    sec = _max_over_ranks(e0.elapsed_time(e1) * 1e-3, dev)
    st0 = steps[0]
    tl = st0.token_layers
    value = _job_rate(tl, args.steps, world, sec)
    errs = [int(s.err.item()) for s in steps]

    # ---- end to end through the public API with pinned host buffers
    host_in = []
    for st in steps:
        host_in.append({k: v.to("cpu").pin_memory() for k, v in st.inputs.items()})
    host_out = torch.empty_like(st0.out[-1], device="cpu").pin_memory()
    host_lse = torch.empty_like(st0.lse[-1], device="cpu").pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host_in[0].values())
    d2h = host_out.numel() * host_out.element_size() + host_lse.numel() * host_lse.element_size()
    # a fixed, longer window than a short --steps run: the first step's input copy
    # cannot overlap anything, so a 20-step window would mostly measure that fill
    e2e_steps = max(100, min(args.steps, 400))
    barrier()
    torch.cuda.synchronize()
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    # A serving loop: step i+1's inputs are copied host -> device on a copy stream
    # while step i computes; step i's output is read back after it finishes.  An
    # input set is overwritten only after the step that used it (i - ROTATE) is
    # done, and its outputs only after they were read back.
    cs = torch.cuda.Stream(device=dev)
    in_ready = [torch.cuda.Event() for _ in range(e2e_steps)]
    done = [torch.cuda.Event() for _ in range(e2e_steps)]
    read = [torch.cuda.Event() for _ in range(e2e_steps)]

    def copy_in(i):
        st = steps[i % ROTATE]
        if i >= ROTATE:
            cs.wait_event(read[i - ROTATE])   # step i - ROTATE computed and its output read
        with torch.cuda.stream(cs):
            for k_, v in host_in[i % ROTATE].items():
                st.inputs[k_].copy_(v, non_blocking=True)
            in_ready[i].record(cs)

    f0.record(stream)
    cs.wait_stream(stream)
    copy_in(0)
    for i in range(e2e_steps):
        if i + 1 < e2e_steps:
            copy_in(i + 1)
        stream.wait_event(in_ready[i])
        with torch.cuda.stream(stream):
            graphs[i % ROTATE].replay()
            done[i].record(stream)
        cs.wait_event(done[i])
        with torch.cuda.stream(cs):
            st = steps[i % ROTATE]
            host_out.copy_(st.out[-1], non_blocking=True)
            host_lse.copy_(st.lse[-1], non_blocking=True)
            read[i].record(cs)
    stream.wait_event(read[e2e_steps - 1])
    f1.record(stream)
    torch.cuda.synchronize()
    e2e_sec = _max_over_ranks(f0.elapsed_time(f1) * 1e-3, dev)
    e2e_value = _job_rate(tl, e2e_steps, world, e2e_sec)

    # ---- per-kernel durations (events around each call, eager steps on the same stream)
    brk = _kernel_breakdown(steps, stream, rounds=max(40, min(args.steps, 400)))
    alg = _algorithmic_bytes(st0)
    peak, peak_kind = _peaks()
    dom = max(brk.items(), key=lambda kv: kv[1]["total_s_per_step"])
    per_launch_bytes = {"sparse_attn": alg["attn_per_launch"],
                        "index_score": None, "topk": None, "build_pool": None, "quantize": None}
    kname = dom[0]
    if kname == "sparse_attn":
        ab = alg["attn_per_launch"]
    elif kname == "index_score":
        ab = alg["keys"] / 5
    else:
        ab = None
    achieved = (ab / dom[1]["avg_s"] / 1e9) if ab else None
    roof = {"bound": "hbm", "kernel": kname, "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": (achieved / peak) if achieved else None,
            "peak_kind": "burst copy (%s; the kernel is timed alone)" % peak_kind,
            "algorithmic_bytes_per_launch": ab,
            "traffic": _traffic_record({"sparse_attn": "sparse_attn_tc_kernel", "index_topk": "index_topk_kernel",
                                        "quantize": "quantize_fp4_kernel"}.get(kname, kname)),
            "avg_launch_us": dom[1]["avg_s"] * 1e6}
    path_bytes = alg["keys"] + alg["gathered"] + alg["outputs"]

    extras = None
    if not args.no_extras:
        extras = _extra_workloads(dev, stream, peak)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(budget_s=args.cpu_budget)
        if args.cpu_workers != 1:
            cpu["all_cores"] = cpu_baseline_all_cores(LAYERS / cpu["value"], budget_s=args.cpu_budget,
                                                      workers=args.cpu_workers or None)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": sec / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp4/fp8 in, f16 mma, f32 accumulate",
        "data": "synthetic (seeded; shapes of the pages' 64K-context batched decode)",
        "config": _workload_config(),
        "path_hbm_gbs": path_bytes / (sec / args.steps) / 1e9,
        "path_bytes_per_step": path_bytes,
        "roofline": roof,
        "kernels": {k: {"avg_us": v["avg_s"] * 1e6, "launches_per_step": v["launches_per_step"],
                        "share": v["total_s_per_step"] / sum(x["total_s_per_step"] for x in brk.values())}
                    for k, v in brk.items()},
        "kernels_timing": "per kind: CUDA graphs of that kind's launches, replayed alone with events",
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps, "pipeline": "step i+1's host->device copies overlap step i on a copy stream"},
        "gpu_launches": st0.launches_per_step() * args.steps,
        "clocks": clocks.summary(t0, t1),
        "device_error_flags": errs,
        "cpu_baseline": cpu,
        "workloads": extras,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------------------ oracle (CPU) arm
def _oracle_sample(n_seq, n_layers=LAYERS, seed=1):
    """Inputs of n_seq sequences for the oracle decode step (CPU, seeded)."""
    import gen
    w = gen.scaled(gen.FULL_BATCHED_DECODE, seed=seed)
    kv_len = gen.as_numpy(gen.kv_lengths(w))[:n_seq].copy()
    k = gen.as_numpy(gen.normal_e4m3(seed, 19, (n_seq, NCAP, 64)))
    q_idx = [gen.as_numpy(gen.normal_e4m3(seed, 20 + 3 * g, (n_seq, 1, 4, 64))) for g in range(5)]
    w_idx = [gen.as_numpy(gen.uniform01(seed, 21 + 3 * g, (n_seq, 1, 4))) for g in range(5)]
    q = [gen.as_numpy(gen.normal_bf16(seed, 200 + l, (n_seq, 1, H, D))) for l in range(n_layers)]
    planes = [tuple(gen.as_numpy(t) for t in gen.fp4_planes(seed, 100 + l, n_seq * NCAP, D)) for l in range(n_layers)]
    new_rows = gen.as_numpy(gen.kv_rows(seed, 70, n_layers * n_seq, D))
    return dict(kv_len=kv_len, k=k, q_idx=q_idx, w_idx=w_idx, q=q, planes=planes, new_rows=new_rows)


def _oracle_step(orc, s, n_seq, schedule):
    """The decode step of the oracle on the sample (all sequences at once)."""
    import numpy as np
    sm = 1.0 / D ** 0.5
    L = len(schedule)
    orc.quantize_kv_fp4(s["new_rows"][: L * n_seq])             # the step's FP4 appends
    gi = -1
    pool = idx = None
    for layer, mode in enumerate(schedule):
        if mode == "full":
            gi += 1
            sc = orc.index_score(orc.FULL, s["q_idx"][gi], orc.FP8_E4M3, s["w_idx"][gi], s["k"], orc.FP8_E4M3,
                                 s["kv_len"]).astype(np.float32)
            if layer == 0:
                pool = orc.build_pool(sc, s["kv_len"], P=P)
            idx = orc.topk(orc.FULL, sc, s["kv_len"], K=K)
        elif mode == "reindex":
            gi += 1
            rs = orc.index_score(orc.REINDEX, s["q_idx"][gi], orc.FP8_E4M3, s["w_idx"][gi], s["k"], orc.FP8_E4M3,
                                 s["kv_len"], pool=pool).astype(np.float32)
            idx = orc.topk(orc.REINDEX, rs, None, pool=pool, K=K)
        codes, scales = s["planes"][layer]
        orc.sparse_attn(s["q"][layer], codes, scales, NCAP, idx, s["kv_len"], sm, DV)


def cpu_baseline(budget_s=15.0):
    """Time the oracle as it stands (single-threaded C, fp64) on a bounded
    sample of the workload: whole sequences through the 20-layer schedule."""
    import oracle as orc
    from gen import DECODER_SCHEDULE
    orc.build()
    s1 = _oracle_sample(1)
    t = time.perf_counter()
    _oracle_step(orc, s1, 1, DECODER_SCHEDULE)
    t1 = time.perf_counter() - t
    n_seq = int(max(1, min(B, budget_s // max(t1, 1e-3))))
    s = _oracle_sample(n_seq)
    t = time.perf_counter()
    _oracle_step(orc, s, n_seq, DECODER_SCHEDULE)
    el = time.perf_counter() - t
    return {"value": n_seq * LAYERS / el, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": "%d of %d sequences x %d layers (one decode step), single-threaded C fp64, %s; %.1f s"
                      % (n_seq, B, LAYERS, _cpu_model(), el)}


def _cpu_model():
    """CPU model string for the report (``model name`` on x86, the Arm part
    number otherwise), with the architecture."""
    import platform
    name = None
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                k, _, v = ln.partition(":")
                if k.strip() in ("model name", "CPU part") and v.strip():
                    name = v.strip() if k.strip() == "model name" else "Arm CPU part " + v.strip()
                    break
    except OSError:
        pass
    return "%s (%s)" % (name or "unknown", platform.machine())


def _oracle_worker(seed, n_seq, schedule, barrier, out_q):
    """One process of the all-cores CPU baseline: its own seeded sequences
    through the same oracle step, timed from a common start."""
    import oracle as orc
    try:
        s = _oracle_sample(n_seq, seed=seed)
        barrier.wait(timeout=600)
        t0 = time.monotonic()
        _oracle_step(orc, s, n_seq, schedule)
        out_q.put((t0, time.monotonic(), n_seq, None))
    except Exception as e:  # reported to the parent, which raises
        out_q.put((0.0, 0.0, 0, repr(e)))


def cpu_baseline_all_cores(per_seq_s, budget_s=10.0, workers=None):
    """The oracle as it stands, one process per host core (the rows spread
    over cores; each process runs whole sequences of its own seed through the
    20-layer step).  Value = all processes' token-layers / (last end - first
    start).  Processes are spawned, never forked, so no CUDA state is shared."""
    import multiprocessing as mp
    import oracle as orc
    from gen import DECODER_SCHEDULE
    orc.build()
    n = int(workers or os.cpu_count() or 1)
    n_seq = int(max(1, min(4, budget_s // max(per_seq_s, 1e-3))))
    ctx = mp.get_context("spawn")
    barrier, q = ctx.Barrier(n), ctx.Queue()
    procs = [ctx.Process(target=_oracle_worker, args=(1000 + i, n_seq, list(DECODER_SCHEDULE), barrier, q))
             for i in range(n)]
    for pr in procs:
        pr.start()
    import queue
    res, deadline = [], time.monotonic() + 1800
    try:
        while len(res) < n:
            try:
                res.append(q.get(timeout=1.0))
            except queue.Empty:
                # a process that died (or every process ended) without its result
                if any(pr.exitcode not in (None, 0) for pr in procs) or time.monotonic() > deadline or \
                        not any(pr.is_alive() for pr in procs):
                    raise RuntimeError("oracle workers ended without a result (exit codes %s)"
                                       % [pr.exitcode for pr in procs])
    finally:
        for pr in procs:
            pr.join(timeout=5 if len(res) < n else 60)
            if pr.is_alive():
                pr.terminate()
                pr.join(timeout=10)
    errs = [r[3] for r in res if r[3]]
    if errs:
        raise RuntimeError("oracle worker failed: " + errs[0])
    el = max(r[1] for r in res) - min(r[0] for r in res)
    total = sum(r[2] for r in res)
    return {"value": total * LAYERS / el, "unit": UNIT, "cores": n, "kind": "oracle",
            "sample": "%d processes x %d sequences x %d layers (one decode step each), C fp64, %s; %.2f s"
                      % (n, n_seq, LAYERS, _cpu_model(), el)}


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return
    import oracle as orc
    from gen import DECODER_SCHEDULE
    orc.build()
    s1 = _oracle_sample(1)
    t = time.perf_counter()
    _oracle_step(orc, s1, 1, DECODER_SCHEDULE)
    t_full = time.perf_counter() - t
    # each step: one sequence through the schedule (or its first group if K+W steps would run too long)
    sched = DECODER_SCHEDULE if t_full * (args.steps + args.warmup) <= 240 else DECODER_SCHEDULE[:4]
    for _ in range(args.warmup):
        _oracle_step(orc, s1, 1, sched)
    t = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(orc, s1, 1, sched)
    el = time.perf_counter() - t
    value = len(sched) * args.steps / el
    sample = "1 of %d sequences x %d layers per step, single-threaded C fp64" % (B, len(sched))
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "config": _workload_config({"sample": sample}),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_profile_case(args):
    """Small, self-terminating cases for full ncu captures of one kernel:
    decode: one input set (about 3.6 GB on the device), three eager decode steps;
    append: the 1,048,576-row quantise, twice (about 1.6 GB);
    prefill: the 4096 x 32768 fused dense indexer, twice (about 0.3 GB)."""
    import torch
    import gen
    import sparse_attention_fp4_quantize_gb300 as csa2
    case = args.profile_case
    if case == "append":
        w5 = gen.APPEND_POOL
        R = w5.B * w5.N
        rows = gen.kv_rows(w5.seed, 10, R, D, rms=False, device="cuda")
        c = torch.empty(R, D // 2, dtype=torch.uint8, device="cuda")
        s = torch.empty(R, D // 16, dtype=torch.uint8, device="cuda")
        for _ in range(2):
            csa2.csa2_quantize_kv_fp4(rows, c, s)
        torch.cuda.synchronize()
        print(json.dumps({"profile_case": "append_quantize_1m_rows", "calls": 2}))
        return
    if case == "prefill_attn":
        # the many-token attention kernel on 1024 of the prefill chunk's queries, twice (about 0.3 GB)
        w4 = gen.scaled(gen.PREFILL_CHUNK, T=1024)
        kl4 = gen.kv_lengths(w4).to("cuda")
        c4, s4 = gen.fp4_planes(3, 1, w4.N, D, device="cuda")
        idx4 = gen.random_indices(w4, kl4.cpu()).to("cuda")
        qa4 = gen.normal_bf16(3, 2, (1, w4.T, H, D), device="cuda")
        oa4 = torch.empty(1, w4.T, H, DV, device="cuda")
        flag = torch.zeros(1, dtype=torch.int32, device="cuda")
        for _ in range(2):
            csa2.csa2_sparse_attn_fp4(0, qa4, c4, s4, w4.N, idx4, oa4, 1 / D ** 0.5, kv_len=kl4, err_flag=flag)
        torch.cuda.synchronize()
        print(json.dumps({"profile_case": "prefill_attention_t1024_k512", "calls": 2, "error_flag": int(flag.item())}))
        return
    if case == "prefill":
        w4 = gen.PREFILL_CHUNK
        q4, ww4, k4 = gen.indexer_inputs(w4, device="cuda")
        kl4 = gen.kv_lengths(w4).to("cuda")
        ws = torch.empty(csa2.csa2_index_topk_dense_workspace_bytes(1, w4.T, w4.N, K), dtype=torch.uint8,
                         device="cuda")
        idx = torch.empty(1, w4.T, K, dtype=torch.int32, device="cuda")
        flag = torch.zeros(1, dtype=torch.int32, device="cuda")
        for _ in range(2):
            csa2.csa2_index_topk_dense(q4, ww4, k4, kl4, idx, workspace=ws, err_flag=flag)
        torch.cuda.synchronize()
        print(json.dumps({"profile_case": "prefill_index_topk_dense_t4096_n32768", "calls": 2,
                          "error_flag": int(flag.item())}))
        return
    from sparse_attention_fp4_quantize_gb300.decode import DecoderStep, StepShape
    st = DecoderStep(StepShape(B=B, N=NCAP, D=D, dv=DV, H=H, K=K, P=P), device="cuda")
    _fill_instance(st, seed=1)
    for _ in range(3):
        st.run()
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": "decoder_step", "steps": 3, "error_flag": int(st.err.item())}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-workers", type=int, default=0,
                    help="processes for the all-cores oracle baseline (0: one per host core; 1: skip it)")
    ap.add_argument("--no-extras", action="store_true", help="skip the other workloads' timings")
    ap.add_argument("--profile-case", nargs="?", const="decode", default=None, choices=["decode", "append", "prefill", "prefill_attn"],
                    help="a small case for ncu: 3 eager decode steps (default), the 1M-row append, the prefill indexer, "
                         "or the many-token attention on 1024 prefill queries")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.profile_case:
        run_profile_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
