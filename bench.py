#!/usr/bin/env python3
"""Benchmark of single-token MLA decode on GB300 through libmla_decode.

One step = one full decode call (stage-1 split kernel + stage-2 merge) over
one batch of synthetic input that is already resident in HBM.  The default
workload is the HBM-bound headline shape: bs=256 requests x 8192 tokens,
fp8-e4m3 KV and fp8 q (per-tensor scales), page size 8 with a permuted page
table (1.21 GB of KV, larger than L2, so no L2 flush is needed).

Prints ONE JSON line (rank 0).  Multi-GPU (torchrun): every rank decodes its
own batch of the same shape (batch-sharded replicas, no collective on the
data path); timing is the max over ranks.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--config NAME] [--no-e2e] [--no-cpu-baseline] [--no-per-config]

The line's `value` is the configuration named by --config (default: the
headline shape); `per_config` adds every configuration of the suite, each
timed the same way in the same run with its own clock record.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA decode µs/call and achieved HBM GB/s (% of 8 TB/s) per (bs, kv_len, KV dtype)"
DEFAULT_CONFIG = "bs256_kv8192_fp8_page8"
L2_BYTES = 129 * 2**20
NOMINAL_HBM_GBS = 8000.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=8)
    ap.add_argument("--bs", type=int, default=0,
                    help="override the batch size of the configuration (profiling runs)")
    ap.add_argument("--q-len", type=int, default=1,
                    help="query tokens per request (causal over the last q_len positions)")
    ap.add_argument("--per-config", dest="per_config", action="store_true", default=True,
                    help="also measure every other configuration of the suite (default)")
    ap.add_argument("--no-per-config", dest="per_config", action="store_false")
    ap.add_argument("--per-config-steps", type=int, default=50,
                    help="timed steps of each other configuration")
    ap.add_argument("--unit-tokens", type=int, default=0,
                    help="plan option: tokens between cut points (32, 64, 128; 0 = 128)")
    ap.add_argument("--item-cost", type=int, default=0,
                    help="plan option: cost of an extra request in a CTA (0 = 1)")
    ap.add_argument("--autotune", dest="autotune", action="store_true", default=False,
                    help="choose each configuration's plan with mla_decode_autotune (untimed)")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def rank_seed(base_seed, rank):
    """Seed of a rank's own batch: every rank decodes a different batch of
    the same shape (batch-sharded replicas)."""
    return base_seed + 1000 * rank


def reduce_over_ranks(dist, max_values, sum_values, device="cpu"):
    """Max over ranks of the times (the slowest rank sets the job's time) and
    sum over ranks of the work counts.  Without a process group (dist is None)
    the values are returned as they are."""
    max_values = [float(v) for v in max_values]
    sum_values = [float(v) for v in sum_values]
    if dist is None:
        return max_values, sum_values
    import torch
    out = []
    for vals, op in ((max_values, dist.ReduceOp.MAX), (sum_values, dist.ReduceOp.SUM)):
        if vals:
            t = torch.tensor(vals, dtype=torch.float64, device=device)
            dist.all_reduce(t, op=op)
            vals = t.tolist()
        out.append(vals)
    return out[0], out[1]


def aggregate_gbs(total_bytes, ms):
    """Whole-job throughput: the bytes of all ranks over the slowest rank's time."""
    return total_bytes / (ms * 1e-3) / 1e9


def config_meta(name, w):
    import workloads as synth
    c = synth.CONFIGS[name]
    return {"workload": name, "bs": w.bs,
            "kv_len": c["kv_len"] if c["kv_len"] is not None else "U[512,8192]",
            "q_dtype": w.q_dtype, "kv_dtype": w.kv_dtype, "page_size": w.page_size,
            "page_table": "permuted" if w.kv_indices is not None else "identity",
            "heads": 16, "qk_dim": 576, "v_dim": 512,
            "parallelism": "batch-sharded replicas (one batch per GPU)",
            **({"q_len": w.q_len} if w.q_len > 1 else {})}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def stage1_traffic(workload):
    """DRAM bytes per stage-1 launch from the committed ncu summary, if it was
    taken on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "stage1_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    src = os.path.join(ROOT, "mla_decode_stage1_gb300", "csrc", "stage1.cu")
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    entry = d.get(workload)
    if not entry or entry.get("stage1_sha") != h:
        return None
    return float(entry["dram_bytes_per_launch"])


class NvmlSampler:
    """SM clock and clock-event reasons read through NVML (read only: no
    setting is changed) about every millisecond in a thread, so that even a
    timed region of a few milliseconds holds samples.  summary() keeps the
    samples taken inside the window given to mark()."""

    # NVML clock-event reason bits (nvml.h); the hardware power brake is a
    # hardware slowdown too
    REASONS = (("hw_slowdown", 0x8 | 0x80), ("hw_thermal_slowdown", 0x40),
               ("sw_thermal_slowdown", 0x20), ("sw_power_cap", 0x4))
    CLOCK_SM = 1

    def __init__(self, index, uuid=None):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit_v2 failed")
        self.dev = ctypes.c_void_p()
        mx = ctypes.c_uint()
        # the CUDA device by its UUID (NVML numbers devices on its own), else by index
        found = uuid is not None and self.lib.nvmlDeviceGetHandleByUUID(
            ("GPU-" + str(uuid)).encode(), ctypes.byref(self.dev)) == 0
        if not found:
            found = self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.dev)) == 0
        if not found or self.lib.nvmlDeviceGetMaxClockInfo(self.dev, self.CLOCK_SM, ctypes.byref(mx)) != 0:
            self.lib.nvmlShutdown()
            raise OSError("NVML device query failed")
        self.max_mhz = mx.value
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.samples, self.window, self.thread = [], None, None
        self.stop = None

    def _poll(self):
        ct = self.ct
        mhz, rs = ct.c_uint(), ct.c_ulonglong()
        while not self.stop.is_set():
            t = time.perf_counter()
            if (self.lib.nvmlDeviceGetClockInfo(self.dev, self.CLOCK_SM, ct.byref(mhz)) == 0
                    and self.reasons_fn(self.dev, ct.byref(rs)) == 0):
                self.samples.append((t, mhz.value, rs.value))
            time.sleep(0.0005)

    def __enter__(self):
        import threading
        self.stop = threading.Event()
        self.thread = threading.Thread(target=self._poll, daemon=True)
        self.thread.start()
        return self

    def __exit__(self, *a):
        self.stop.set()
        self.thread.join(timeout=5)
        self.lib.nvmlShutdown()

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def summary(self):
        rows = self.samples
        where = "whole sampling period"
        if self.window is not None:
            inside = [r for r in rows if self.window[0] <= r[0] <= self.window[1]]
            if inside:
                rows, where = inside, "timed region"
        if not rows:
            return None
        sm = sorted(r[1] for r in rows)
        reasons = sorted({name for r in rows for name, bit in self.REASONS if r[2] & bit})
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(rows), "source": "nvml", "window": where}


def clock_sampler(index):
    """The NVML sampler where the driver library loads, else nvidia-smi."""
    try:
        import torch
        uuid = getattr(torch.cuda.get_device_properties(index), "uuid", None)
    except Exception:
        uuid = None
    try:
        return NvmlSampler(index, uuid)
    except (OSError, AttributeError):
        return ClockSampler(index)


class ClockSampler:
    """nvidia-smi clock / throttle sampling (100 ms interval) around the
    timed region; the fallback when NVML cannot be loaded."""

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def mark(self, t0, t1):
        pass

    def summary(self):
        if self.path is None or not os.path.exists(self.path):
            return None
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        sm = sorted(r[0] for r in rows)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[2]) if v.lower() == "active"})
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": rows[0][1], "reasons": reasons,
                "samples": len(rows), "source": "nvidia-smi", "window": "around the timed region"}


def cpu_baseline(w, target_s=8.0):
    """The fp64 oracle, as it stands, on the host cores over a bounded sample
    of the workload's requests.  Returns (GB/s, cores, sample description)."""
    import oracle
    import workloads as synth
    cores = os.cpu_count() or 1
    n = max(1, min(w.bs, cores))
    args = synth.oracle_args(w)
    elapsed = 0.0
    done = 0
    nbytes = 0
    per_req_qo = w.q_len * (16 * 576 * (2 if w.q_dtype == "bf16" else 1) + 16 * 512 * 2)
    start = 0
    while elapsed < target_s and done < w.bs:
        sel = list(range(start, min(start + n, w.bs)))
        t0 = time.perf_counter()
        oracle.mla_decode(**dict(args, select=sel), nthreads=cores)
        elapsed += time.perf_counter() - t0
        done += len(sel)
        nbytes += sum(w.lengths[i] for i in sel) * w.kv_bytes_per_token() + len(sel) * per_req_qo
        start += len(sel)
        if elapsed > 0 and (target_s - elapsed) < elapsed / max(1, done) * n:
            break
    return nbytes / elapsed / 1e9, cores, f"{done} of {w.bs} requests ({nbytes/1e6:.1f} MB algorithmic), {elapsed:.1f} s"


def run_reference(args, world, rank):
    """Reference arm: the fp64 CPU oracle on the host cores, each step a
    bounded sample of the same workload (rank 0 only)."""
    if rank != 0:
        return
    import workloads as synth
    w = synth.make_config(args.config, device="cpu")
    import oracle
    oargs = synth.oracle_args(w)
    cores = os.cpu_count() or 1
    sample = list(range(min(w.bs, max(1, cores // 2))))
    per_req_qo = 16 * 576 * (2 if w.q_dtype == "bf16" else 1) + 16 * 512 * 2
    nbytes = sum(w.lengths[i] for i in sample) * w.kv_bytes_per_token() + len(sample) * per_req_qo
    for _ in range(args.warmup):
        oracle.mla_decode(**dict(oargs, select=sample[:1]), nthreads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.mla_decode(**dict(oargs, select=sample), nthreads=cores)
    dt = (time.perf_counter() - t0) / args.steps
    value = nbytes / dt / 1e9
    desc = f"{len(sample)} of {w.bs} requests per step"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_meta(args.config, w),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def build_workload(name, rank, dev, bs_override=0, q_len=1):
    """The seeded workload of configuration `name` for this rank, on `dev`."""
    import workloads as synth
    c = synth.CONFIGS[name]
    lengths = synth.config_lengths(name)
    if bs_override:
        lengths = (lengths * ((bs_override + len(lengths) - 1) // len(lengths)))[:bs_override]
    return synth.make_workload(bs=len(lengths), lengths=lengths, page_size=c["page_size"],
                               q_dtype=c["q_dtype"], kv_dtype=c["kv_dtype"],
                               permute_pages=c["permute_pages"], seed=rank_seed(c["seed"], rank),
                               device=dev, name=name, q_len=q_len)


class Decoder:
    """One configuration made ready to decode: its plan, workspace, outputs
    and (for inputs smaller than twice the L2) the buffer that flushes L2."""

    def __init__(self, mla, w, dev, unit_tokens=0, item_cost=0, autotune=False):
        import torch
        self.mla, self.w, self.d = mla, w, w.to(dev)
        self.out = torch.empty(w.bs * w.q_len, 16, 512, dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty(w.bs * w.q_len, 16, dtype=torch.float32, device=dev)
        self.tuned = None
        if autotune:
            d = self.d
            kw = dict(page_size=w.page_size, q_dtype=w.q_dtype, kv_dtype=w.kv_dtype,
                      q_scale=d.q_scale, kv_scale=d.kv_scale, kv_e8m0=d.kv_e8m0,
                      kv_indices=d.kv_indices, lse=self.lse, q_len=w.q_len)
            need = mla.mla_decode_autotune(w.kv_indptr, w.kv_last_page_len, d.q, d.kv, self.out, **kw)
            self.ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
            self.plan, self.tuned = mla.mla_decode_autotune(w.kv_indptr, w.kv_last_page_len, d.q,
                                                            d.kv, self.out, workspace=self.ws,
                                                            reps=5, **kw)
        else:
            self.plan = mla.mla_decode_plan(w.kv_indptr, w.kv_last_page_len, page_size=w.page_size,
                                            q_dtype=w.q_dtype, kv_dtype=w.kv_dtype, q_len=w.q_len,
                                            unit_tokens=unit_tokens, item_cost=item_cost)
            self.ws = torch.empty(max(self.plan.workspace_bytes, 256), dtype=torch.uint8,
                                  device=dev)
        self.info = self.plan.info()
        self.alg_bytes = w.algorithmic_bytes()
        self.kv_bytes = w.total_tokens() * w.kv_bytes_per_token()
        self.flush = self.kv_bytes < 2 * L2_BYTES
        self.scratch = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev) if self.flush else None

    def step(self, stream=None):
        d = self.d
        self.mla.mla_decode_run(self.plan, d.q, d.kv, self.out, workspace=self.ws, q_scale=d.q_scale,
                                kv_scale=d.kv_scale, kv_e8m0=d.kv_e8m0, kv_indices=d.kv_indices,
                                lse=self.lse, stream=stream)

    def measure(self, K, warmup, dist, local):
        """W untimed steps, then K steps timed with CUDA events on the
        launching stream (L2 flushed before each step when the inputs fit
        in it), bracketed by a barrier and a synchronize; then K more steps
        with events the library records around the stage-1 launch alone.
        Returns (ms per step, stage-1 ms, clocks, wall seconds), the times
        already the max over ranks."""
        import torch
        stream = torch.cuda.current_stream()
        for _ in range(max(3, warmup)):
            if self.flush:
                self.scratch.fill_(1)
            self.step()
        torch.cuda.synchronize()
        self.mla.mla_decode_check(self.plan, self.ws)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K)]
        ev_s1 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(K)]
        for a, b in ev_s1:   # torch creates the CUDA event on first record
            a.record(stream)
            b.record(stream)
        with clock_sampler(local) as clk:
            if dist is not None:
                dist.barrier()
            torch.cuda.synchronize()
            t_start = time.perf_counter()
            for i in range(K):
                if self.flush:
                    self.scratch.fill_(1)
                ev[i][0].record(stream)
                self.step()
                ev[i][1].record(stream)
            torch.cuda.synchronize()
            t_end = time.perf_counter()
            clk.mark(t_start, t_end)
            if dist is not None:
                dist.barrier()
            # second pass: the stage-1 kernel alone, between events the library
            # records around its launch (kept out of the headline loop because an
            # event between the two kernels would serialise their launches)
            for i in range(K):
                if self.flush:
                    self.scratch.fill_(1)
                self.plan.set_stage1_events(*ev_s1[i])
                self.step()
            torch.cuda.synchronize()
        self.plan.set_stage1_events(None, None)
        self.mla.mla_decode_check(self.plan, self.ws)
        step_ms = sum(a.elapsed_time(b) for a, b in ev) / K
        s1_ms = sum(a.elapsed_time(b) for a, b in ev_s1) / K
        (step_ms, s1_ms), _ = reduce_over_ranks(dist, [step_ms, s1_ms], [],
                                                device=torch.device("cuda", local))
        return step_ms, s1_ms, clk.summary(), t_end - t_start


def config_entry(dec, step_ms, s1_ms, clocks, total_bytes, peak):
    """The per-configuration figures of the bench line."""
    gbs = aggregate_gbs(total_bytes, step_ms)
    s1 = dec.alg_bytes / (s1_ms * 1e-3) / 1e9
    return {"us_per_call": step_ms * 1e3, "GBps": gbs,
            "pct_of_8TBps": 100.0 * (dec.alg_bytes / (step_ms * 1e-3) / 1e9) / NOMINAL_HBM_GBS,
            "stage1_us": s1_ms * 1e3, "stage1_GBps": s1, "stage1_frac": s1 / peak,
            "algorithmic_bytes": dec.alg_bytes, "num_ctas": dec.info.num_ctas,
            "num_partials": dec.info.num_partials, "plan": plan_meta(dec),
            "l2": "flushed between steps (2x L2 write)" if dec.flush else "inputs larger than L2",
            "clocks": clocks}


def plan_meta(dec):
    """The plan options in use (and, after autotune, every candidate's time)."""
    m = {"unit_tokens": dec.info.unit_tokens, "item_cost": dec.info.item_cost,
         "num_ctas": dec.info.num_ctas,
         "merge": "cluster of %d" % dec.info.cluster_size if dec.info.cluster_size else "stage 2"}
    if dec.tuned is not None:
        m["autotune"] = [dict(o, median_ms=ms) for o, ms in dec.tuned]
    return m


def main():
    args = parse()
    world, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    import torch
    import mla_decode_stage1_gb300 as mla
    import workloads as synth

    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peak, peak_kind = load_peaks()

    # every rank owns one batch of the configured shape (weak scaling)
    w = build_workload(args.config, rank, dev, args.bs, args.q_len)
    dec = Decoder(mla, w, dev, args.unit_tokens, args.item_cost, args.autotune)
    torch.cuda.empty_cache()
    info, alg_bytes = dec.info, dec.alg_bytes
    meta = dict(config_meta(args.config, w),
                l2="flushed between steps (2x L2 write)" if dec.flush else
                f"inputs larger than L2 ({dec.kv_bytes/1e9:.2f} GB KV)",
                algorithmic_bytes=alg_bytes, num_ctas=info.num_ctas,
                num_partials=info.num_partials, plan=plan_meta(dec))
    K = args.steps
    step_ms, s1_ms, clocks, t_wall = dec.measure(K, args.warmup, dist, local)
    (total_bytes,) = reduce_over_ranks(dist, [], [alg_bytes], device=dev)[1]

    # end to end through the public API: pinned host inputs -> device, decode,
    # output + lse -> pinned host, every step.  Inputs are double-buffered on
    # the device: step i+1's copy (on its own stream) overlaps step i's decode.
    e2e = None
    if not args.no_e2e:
        d, plan, out, lse, ws = dec.d, dec.plan, dec.out, dec.lse, dec.ws
        stream = torch.cuda.current_stream(dev)
        host = {k: (None if v is None else v.cpu().pin_memory())
                for k, v in (("q", d.q), ("kv", d.kv), ("q_scale", d.q_scale),
                             ("kv_scale", d.kv_scale), ("kv_e8m0", d.kv_e8m0),
                             ("kv_indices", d.kv_indices))}
        dev_in = [{k: (None if v is None else torch.empty_like(v, device=dev))
                   for k, v in host.items()} for _ in range(2)]
        out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
        d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * lse_h.element_size()
        E = max(1, args.e2e_steps)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        copy_stream = torch.cuda.Stream(dev)
        copied = [torch.cuda.Event() for _ in range(2)]   # buffer b holds its step's inputs
        released = [torch.cuda.Event() for _ in range(2)]  # the decode reading buffer b is done
        for ev in released:
            ev.record(stream)

        def e2e_step(i):
            b = i % 2
            copy_stream.wait_event(released[b])
            with torch.cuda.stream(copy_stream):
                for k, v in host.items():
                    if v is not None:
                        dev_in[b][k].copy_(v, non_blocking=True)
                copied[b].record(copy_stream)
            stream.wait_event(copied[b])
            x = dev_in[b]
            mla.mla_decode_run(plan, x["q"], x["kv"], out, workspace=ws, q_scale=x["q_scale"],
                               kv_scale=x["kv_scale"], kv_e8m0=x["kv_e8m0"],
                               kv_indices=x["kv_indices"], lse=lse, stream=stream)
            released[b].record(stream)
            out_h.copy_(out, non_blocking=True)
            lse_h.copy_(lse, non_blocking=True)

        e2e_step(0)                              # both input buffers once, untimed
        e2e_step(1)
        torch.cuda.synchronize()
        # Three timed batches of E steps; the median batch is reported.  The
        # host link is shared with the rest of the machine, and one batch in
        # a few can read at half speed while another job copies.
        batches = []
        for rep in range(3):
            if dist is not None:
                dist.barrier()
            e0.record(stream)
            copy_stream.wait_stream(stream)      # every timed copy starts after e0
            for i in range(2 + rep * E, 2 + (rep + 1) * E):
                e2e_step(i)
            e1.record(stream)
            torch.cuda.synchronize()
            batches.append(e0.elapsed_time(e1) / E)
        e2e_ms = sorted(batches)[1]
        (e2e_ms,), _ = reduce_over_ranks(dist, [e2e_ms], [], device=dev)
        e2e = {"value": aggregate_gbs(total_bytes, e2e_ms), "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "steps": E, "batches": 3, "batch_ms_per_step": [round(b, 4) for b in batches],
               "summary": "median of the three batches",
               "overlap": "double-buffered inputs: a step's copy overlaps the previous decode"}
        del dev_in, host, d, plan, out, lse, ws

    # every other configuration of the suite, measured the same way in the
    # same run (the headline configuration's entry is the measurement above)
    per_config = None
    if args.per_config and not args.bs and args.q_len == 1:
        per_config = {args.config: config_entry(dec, step_ms, s1_ms, clocks, total_bytes, peak)}
        w_cpu = w.to("cpu") if rank == 0 and not args.no_cpu_baseline else None
        del dec, w
        torch.cuda.empty_cache()
        for name in synth.CONFIGS:
            if name == args.config:
                continue
            other = Decoder(mla, build_workload(name, rank, dev), dev, args.unit_tokens,
                            args.item_cost, args.autotune)
            o_ms, o_s1, o_clk, _ = other.measure(min(K, args.per_config_steps), args.warmup,
                                                 dist, local)
            (o_total,) = reduce_over_ranks(dist, [], [other.alg_bytes], device=dev)[1]
            per_config[name] = config_entry(other, o_ms, o_s1, o_clk, o_total, peak)
            del other
            torch.cuda.empty_cache()
        per_config = {name: per_config[name] for name in synth.CONFIGS}
    else:
        w_cpu = w.to("cpu") if rank == 0 and not args.no_cpu_baseline else None

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    achieved = alg_bytes / (s1_ms * 1e-3) / 1e9
    # the committed DRAM counts are for the configuration as named
    traffic = stage1_traffic(args.config) if not args.bs and args.q_len == 1 else None
    gbs = aggregate_gbs(total_bytes, step_ms)
    cfg = synth.CONFIGS[args.config]
    line = {
        "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": step_ms, "us_per_call": step_ms * 1e3,
        "pct_of_8TBps": 100.0 * (alg_bytes / (step_ms * 1e-3) / 1e9) / NOMINAL_HBM_GBS,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": cfg["kv_dtype"] if cfg["q_dtype"] == cfg["kv_dtype"]
        else f"{cfg['q_dtype']}q/{cfg['kv_dtype']}kv",
        "data": "synthetic: seeded N(0,1) q and KV, per-tensor e4m3 quantisation (amax/448), "
                "MXFP4 per the OCP MX rule",
        "config": meta,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind, "traffic": traffic,
                     "kernel": "mla_stage1_kernel", "stage1_us": s1_ms * 1e3},
        # stage 1, plus stage 2 unless the plan merges inside clusters
        "gpu_launches": K * (1 + (1 if info.num_merge_jobs > 0 and info.cluster_size == 0 else 0)),
        "clocks": clocks,
        "wall_s_timed": t_wall,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if per_config is not None:
        line["per_config"] = per_config
    if w_cpu is not None:
        try:
            v, cores, sample = cpu_baseline(w_cpu)
            line["cpu_baseline"] = {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle",
                                    "sample": sample}
        except Exception as e:  # the oracle is optional for the GPU number itself
            line["cpu_baseline"] = {"value": None, "unit": "GB/s", "cores": os.cpu_count(),
                                    "kind": "oracle", "sample": f"failed: {e}"}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
