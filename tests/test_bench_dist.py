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
