"""Host logic of the benchmark, on the CPU (no GPU and no CUDA call).

bench.py under torchrun runs one replica per GPU (the decode path shards by
sequence and has no exchange step): every rank draws its own sequences, times
its own steps, and the job's time is the slowest rank's.  These tests run
that logic with two gloo ranks, and check the all-cores oracle baseline, the
DRAM traffic record's validity rule and the clock summary.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, secs, out_dir):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, _ = bench._dist()
        assert (w, r) == (world, rank)
        dist.barrier()
        slowest = bench._max_over_ranks(secs[rank])
        rate = bench._job_rate(640, 10, w, slowest)
        # the second reduction must see the same answer on every rank
        again = bench._max_over_ranks(slowest)
        with open(os.path.join(out_dir, "rank%d.txt" % rank), "w") as f:
            f.write("%r %r %r\n" % (slowest, rate, again))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_gloo_two_ranks(tmp_path):
    world = 2
    secs = [0.25, 0.4]   # rank 1 is slower: the job takes its time
    mp.start_processes(_rank_main, args=(world, _free_port(), secs, str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    got = []
    for r in range(world):
        slowest, rate, again = (float(x) for x in open(tmp_path / ("rank%d.txt" % r)).read().split())
        got.append((slowest, rate, again))
    for slowest, rate, again in got:
        assert slowest == pytest.approx(0.4)
        assert again == pytest.approx(0.4)
        # 640 token-layers per rank-step, 10 steps, both ranks' work over the slowest time
        assert rate == pytest.approx(640 * 10 * world / 0.4)


def test_single_process_is_identity():
    assert not dist.is_initialized()
    assert bench._max_over_ranks(0.123) == pytest.approx(0.123)
    assert bench._job_rate(640, 10, 1, 0.5) == pytest.approx(12800.0)


def test_rank_seeds_are_disjoint():
    seeds = {(rank, r): bench._rank_seed(rank, r) for rank in range(8) for r in range(bench.ROTATE)}
    assert len(set(seeds.values())) == len(seeds)
    assert bench._rank_seed(0, 0) == 1   # rank 0's first input set is the single-GPU workload's seed


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")

    class Args:
        steps, warmup = 1, 3

    # must return at once: no oracle build, no output
    assert bench.run_reference(Args()) is None
    assert capsys.readouterr().out == ""


def test_all_cores_cpu_baseline_spawns_workers_and_counts_their_work():
    """The all-cores oracle baseline: two spawned processes, one sequence
    each through the 20-layer oracle step; the value counts both."""
    r = bench.cpu_baseline_all_cores(per_seq_s=100.0, budget_s=0.0, workers=2)
    assert r["cores"] == 2 and r["kind"] == "oracle" and r["unit"] == bench.UNIT
    assert r["sample"].startswith("2 processes x 1 sequences x 20 layers")
    el = float(r["sample"].rsplit(";", 1)[1].strip().rstrip("s"))
    assert r["value"] == pytest.approx(2 * bench.LAYERS / el, rel=0.03)


def test_traffic_record_is_used_only_while_the_source_is_unchanged(tmp_path, monkeypatch):
    import hashlib
    import json
    src = tmp_path / "k.cu"
    src.write_text("kernel v1\n")
    (tmp_path / "profiles").mkdir()
    rec = {"k_kernel": {"source": "k.cu", "source_sha256_16": hashlib.sha256(b"kernel v1\n").hexdigest()[:16],
                        "dram_bytes_per_launch": 1234}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._traffic_record("k_kernel") == 1234
    assert bench._traffic_record("other_kernel") is None
    src.write_text("kernel v2\n")                        # the kernel changed since the capture
    assert bench._traffic_record("k_kernel") is None


def test_clock_summary_takes_the_timed_window_and_the_active_reasons():
    c = bench.ClockSampler(0)
    row = "0, {sm}, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, {cap}"
    c.samples = [(9.0, row.format(sm=1000, cap="Not Active")),          # before the timed region
                 (10.1, row.format(sm=2070, cap="Not Active")),
                 (10.2, row.format(sm=1965, cap="Active")),
                 (10.3, "garbage line"),
                 (10.4, row.format(sm=2055, cap="Not Active")),
                 (12.0, row.format(sm=500, cap="Not Active"))]          # after it
    s = c.summary(10.0, 11.0)
    assert s["samples"] == 3 and s["sm_mhz"] == 2055 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]
    assert c.summary(10.45, 10.5)["samples"] == 3                        # shorter than a period: nearest samples
    assert bench.ClockSampler(0).summary(0, 1)["reasons"] == ["nvidia-smi unavailable"]
