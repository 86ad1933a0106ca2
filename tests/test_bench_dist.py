"""Multi-rank host logic of bench.py on CPU: two gloo ranks.

The GPU benchmark runs one process per GPU (torchrun).  Every rank decodes
its own batch (batch-sharded replicas), the job's time is the slowest rank's
and its work is the sum of all ranks' bytes.  These tests run that host
logic with the gloo backend; no GPU and no NCCL are involved.
"""
import os
import socket

import pytest

import bench


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, queue):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r: step time 10 + r ms, stage-1 time 5 (r + 1) ms, 1e9 (r + 1) bytes
        (step_ms, s1_ms), (total,) = bench.reduce_over_ranks(
            dist, [10.0 + rank, 5.0 * (rank + 1)], [1e9 * (rank + 1)])
        (e2e_ms,), empty = bench.reduce_over_ranks(dist, [3.0 - rank], [])
        queue.put((rank, step_ms, s1_ms, total, e2e_ms, empty, bench.rank_seed(4, rank)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_max_time_and_sum_work():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    results = [queue.get(timeout=180) for _ in procs]
    for p in procs:
        p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs)
    assert sorted(r[0] for r in results) == [0, 1]
    for _, step_ms, s1_ms, total, e2e_ms, empty, _ in results:
        assert step_ms == 11.0 and s1_ms == 10.0       # the slowest rank's times
        assert total == 3e9                             # both ranks' bytes
        assert e2e_ms == 3.0 and empty == []
    assert len({r[6] for r in results}) == 2           # every rank its own batch
    # whole-job throughput: 3e9 bytes over the slowest rank's 11 ms
    assert bench.aggregate_gbs(3e9, 11.0) == pytest.approx(3e9 / 11e-3 / 1e9)


def test_single_process_reduction_is_identity():
    assert bench.reduce_over_ranks(None, [1.5, 2.5], [7]) == ([1.5, 2.5], [7.0])
    assert bench.rank_seed(4, 0) == 4


def test_nvml_clock_samples_are_kept_from_the_timed_window_only():
    # the sampler's summary (no NVML call: the samples are injected) keeps the
    # samples inside the timed window and decodes NVML's clock-event bits
    s = bench.NvmlSampler.__new__(bench.NvmlSampler)
    s.max_mhz = 2070
    s.samples = [(0.5, 900, 0x1),           # idle, before the window
                 (1.0, 2070, 0x4),          # sw power cap
                 (1.2, 2040, 0x0),
                 (1.5, 2070, 0x40),         # hw thermal slowdown
                 (3.0, 500, 0x8 | 0x20)]    # after the window
    s.window = (0.9, 2.0)
    got = s.summary()
    assert got["samples"] == 3 and got["window"] == "timed region"
    assert got["sm_mhz"] == 2070 and got["sm_max_mhz"] == 2070
    assert got["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    # a window that no sample falls in reports the whole sampling period
    s.window = (10.0, 11.0)
    got = s.summary()
    assert got["samples"] == 5 and got["window"] == "whole sampling period"
    assert got["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap",
                              "sw_thermal_slowdown"]


def test_reference_arm_prints_its_json_line():
    # `bench.py --impl reference` (the fp64 oracle on the host cores) needs no
    # GPU: one JSON line with the bench contract's keys and the reference
    # arm's own (impl, cpu_baseline, an e2e with no copies)
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    # run the arm as bench.py's __main__, then list what the process mapped:
    # the oracle's library, never the CUDA decode library
    code = ("import runpy, sys; sys.argv = ['bench.py', '--impl', 'reference', '--config', "
            "'bs4_kv1024_bf16', '--steps', '1', '--warmup', '0']; "
            "runpy.run_path('bench.py', run_name='__main__'); "
            "maps = open('/proc/self/maps').read(); "
            "print('MAPS', 'libmla_decode' in maps, 'libmla_oracle' in maps, "
            "'mla_decode_stage1_gb300' in sys.modules)")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300,
                       cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert lines[-1] == "MAPS False True False", lines[-1]
    d = json.loads(lines[-2])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["config"]["workload"] == "bs4_kv1024_bf16" and d["steps"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
