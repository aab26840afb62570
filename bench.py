#!/usr/bin/env python3
"""Benchmark: decode-attention KV-read throughput on one GB300 per rank.

A step is one decode_attn_run (the split kernel with its in-kernel LSE merge and range check,
plus in unified mode the recompute launch for flagged groups) over the named workload, inputs
resident in HBM. Default workload: long-context GQA, batch 1, 32 query heads over 8 KV heads,
head_dim 128, 32768 tokens, bf16 K/V, unified-max softmax with the heuristic (balanced)
split. Other workloads: tiny, mha, paged, stress, and gqa32k_fp8 / paged_fp8 (the same
draws over FP8 E4M3 caches). Before every timed step, outside the timed
events, the L2 is flushed: 256 MiB are written, then 256 MiB of another buffer are read so
that the written lines are evicted before the step rather than during it; a device-side spin
then gives the host time to enqueue the step before the GPU reaches its start event.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--mode MODE]
  python bench.py --impl reference ...   # the float64 CPU oracle on the host cores
  python bench.py --op logit_histogram --workload NAME   # the phi calibration pass

Under torchrun each rank runs an independent replica of the workload on its own GPU
(weak scaling); value = all ranks' KV bytes / the slowest rank's time.
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn KV-read GB/s (% of GB300 HBM peak); µs/decode step at 32K GQA"
FALLBACK_HBM_GBS = 6800.0
FLUSH_BYTES = 256 << 20
# Device-side spin (clock cycles, ~0.15 ms at 2 GHz) enqueued after each flush and before each
# timed step, outside the step's events: the host enqueues the step while the GPU spins, so
# the host's own call overhead never leaves the GPU idle inside the timed region.
HOST_AHEAD_CYCLES = 300_000


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="gqa32k")
    ap.add_argument("--mode", default="unified_local",
                    choices=["unified", "sync", "unified_local"])
    ap.add_argument("--num-splits", type=int, default=-1,
                    help="-1: the plan's heuristic; >0 uniform splits")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-side", action="store_true",
                    help="time only the named workload (no paged / MHA / stress / FP8 lines)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--op", default="attention", choices=["attention", "logit_histogram"],
                    help="attention: the decode step (default); logit_histogram: the phi "
                         "calibration pass over the same workload")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(values, device="cpu"):
    """Element-wise maximum of per-rank timings over the process group (identity on one rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "decode_attention_attn_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload_name, kernel="split_kernel"):
    """dram read+write bytes per launch of `kernel` from the committed ncu summary, or None
    when the summary is missing or was taken on different kernel sources."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload_name}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_hash = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", text)
    m_bytes = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    if not m_hash or not m_bytes or m_hash.group(1) != kernel_source_hash():
        return None
    return int(m_bytes.group(1))


class RawEvent:
    """A CUDA event created through the CUDA runtime directly, so that the library can record
    it inside decode_attn_run_ex (torch events only time what torch itself recorded)."""
    _rt = None

    @classmethod
    def runtime(cls):
        if cls._rt is None:
            import ctypes
            import ctypes.util
            cands = [os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "lib64",
                                  "libcudart.so"), "libcudart.so.13", "libcudart.so"]
            found = ctypes.util.find_library("cudart")
            if found:
                cands.append(found)
            for c in cands:
                try:
                    cls._rt = ctypes.CDLL(c)
                    break
                except OSError:
                    continue
            if cls._rt is None:
                raise RuntimeError("libcudart not found for raw CUDA events")
        return cls._rt

    def __init__(self):
        import ctypes
        h = ctypes.c_void_p()
        if self.runtime().cudaEventCreate(ctypes.byref(h)) != 0:
            raise RuntimeError("cudaEventCreate failed")
        self.cuda_event = h.value

    def elapsed_ms(self, end):
        import ctypes
        ms = ctypes.c_float()
        rc = self.runtime().cudaEventElapsedTime(ctypes.byref(ms), ctypes.c_void_p(self.cuda_event),
                                                 ctypes.c_void_p(end.cuda_event))
        if rc != 0:
            raise RuntimeError(f"cudaEventElapsedTime failed ({rc})")
        return ms.value


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        self.proc.wait()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.remove(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


class L2Flush:
    """Write a buffer larger than L2 (so no input stays cached), then read a second one so
    that the write's dirty lines are evicted before the timed region instead of inside it."""

    def __init__(self, device):
        import torch
        self.w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.r = torch.ones(FLUSH_BYTES // 8, dtype=torch.int64, device=device)
        self.n = 0

    def __call__(self):
        self.n += 1
        self.w.fill_(self.n & 0xFF)
        self.r.max()


def pct(xs, q):
    """The q-quantile of xs (nearest rank)."""
    ys = sorted(xs)
    return ys[min(len(ys) - 1, max(0, int(round(q * (len(ys) - 1)))))]


def spread(ms_list):
    """median / min / p90 / mean of per-step times, in µs."""
    us = [1e3 * m for m in ms_list]
    return {"median": round(statistics.median(us), 3), "min": round(min(us), 3),
            "p90": round(pct(us, 0.9), 3), "mean": round(sum(us) / len(us), 3)}


def time_step(attn, dev, wl, num_splits, steps, warmup, stream, flush, out, lse, flags,
              sampler=None):
    """Time `steps` decode steps (each after an L2 flush and a host-ahead spin) with CUDA
    events around the whole step, then the same steps again with events recorded by the
    library around the split kernel alone. Returns (step ms list, split-kernel ms list,
    clocks)."""
    import torch

    def step(split_events=None):
        attn.run(dev.q, dev.k, dev.v, dev.bt, dev.sl, wl.scale, num_splits, out=out,
                 out_lse=lse, row_flags=flags, stream=stream, split_events=split_events)

    for _ in range(max(3, warmup)):
        flush()
        step()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    clocks = None
    if sampler is not None:
        sampler.start()
    for i in range(steps):
        flush()
        torch.cuda._sleep(HOST_AHEAD_CYCLES)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    if sampler is not None:
        clocks = sampler.stop()
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    ks = [RawEvent() for _ in range(steps)]
    ke = [RawEvent() for _ in range(steps)]
    for i in range(steps):
        flush()
        torch.cuda._sleep(HOST_AHEAD_CYCLES)
        step(split_events=(ks[i], ke[i]))
    torch.cuda.synchronize()
    kern_ms = [a.elapsed_ms(b) for a, b in zip(ks, ke)]
    return step_ms, kern_ms, clocks


def launches_per_step(mode):
    return 2 if mode == "unified" else 1   # split kernel (+ the recompute launch)


# Workloads measured beside the headline by the default run: the other named configurations
# of the gate and the stress test's fallback rates (paged batch, Llama2-7B-shaped MHA, the
# unified-max stress in both unified modes), plus the FP8 caches.
# (workload, softmax mode, split override): the MHA step runs with its stated 16 splits of
# 256 tokens and once more with the library's balanced shares (None: the workload's own).
SIDE_WORKLOADS = [("mha", "unified_local", None), ("mha", "unified_local", 0),
                  ("paged", "unified_local", None), ("paged", "unified", None),
                  ("stress", "unified", None),
                  ("stress", "unified_local", None), ("gqa32k_fp8", "unified_local", None),
                  ("paged_fp8", "unified_local", None)]


def measure_side(name, mode, splits, args, dev_name, stream, flush, peak, peak_kind):
    """One side workload: step and split-kernel time spread, GB/s, roofline and fallback rates."""
    import torch
    from decode_attention_attn_gb300 import binding, harness, workloads
    wl = workloads.get(name).replace(mode=mode)
    if splits is not None:
        wl = wl.replace(num_splits=splits)
    inp = workloads.generate(wl)
    kv_bytes = inp.kv_bytes()
    dev = harness.DeviceInputs(inp, dev_name)
    attn = binding.DecodeAttention(harness.problem_for(inp, mode=mode), wl.num_splits)
    B, H, d = wl.batch, wl.num_q_heads, wl.head_dim
    out = torch.empty((B, H, d), dtype=workloads.TORCH_DTYPES[wl.out_dtype], device=dev_name)
    lse = torch.empty((B, H), dtype=torch.float32, device=dev_name)
    flags = torch.empty((B, H), dtype=torch.uint8, device=dev_name)
    steps = max(10, min(args.steps, 30))
    step_ms, kern_ms, clocks = time_step(attn, dev, wl, -1, steps, args.warmup, stream, flush,
                                         out, lse, flags, ClockSampler(torch.cuda.current_device()))
    stats = attn.run(dev.q, dev.k, dev.v, dev.bt, dev.sl, wl.scale, -1, want_stats=True)[3]
    ms = statistics.median(step_ms)
    km = statistics.median(kern_ms)
    res = {"workload": wl.name, "softmax": mode, "kv_dtype": wl.kv_storage,
           "splits": (f"{wl.num_splits} uniform splits" if wl.num_splits > 0
                      else "heuristic (balanced shares)"),
           "kv_bytes_per_step": kv_bytes, "us_per_step": spread(step_ms),
           "value": round(kv_bytes / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
           "pct_hbm_peak": round(100 * kv_bytes / (ms * 1e-3) / 1e9 / peak, 2),
           "roofline": {"bound": "hbm", "achieved": round(kv_bytes / (km * 1e-3) / 1e9, 1),
                        "peak": peak, "unit": "GB/s",
                        "frac": round(kv_bytes / (km * 1e-3) / 1e9 / peak, 4),
                        "peak_source": f"{peak_kind} hbm_gbs", "kernel": "decode_split_kernel",
                        "kernel_us": spread(kern_ms),
                        "traffic": profiled_traffic(wl.name) if splits is None else None},
           "clocks": clocks, "steps": steps, "gpu_launches": launches_per_step(mode) * steps,
           "grid_ctas": attn.info.grid_ctas,
           "split_tokens": [stats.split_tokens_min, stats.split_tokens]}
    if mode != "sync":
        rows = B * H
        res["rows_flagged"] = int(stats.rows_flagged)
        res["row_fallback_rate"] = round(stats.rows_flagged / rows, 6)
        res["splits_flagged"] = int(stats.splits_flagged)
    del dev, attn, inp, out, lse, flags
    torch.cuda.empty_cache()
    return res


def run_ours(args):
    import torch
    import torch.distributed as dist
    from decode_attention_attn_gb300 import binding, harness, workloads

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev_name = f"cuda:{local}"
    wl = workloads.get(args.workload)
    wl = wl.replace(mode=args.mode)
    inp = workloads.generate(wl, offset=rank)
    kv_bytes = inp.kv_bytes()
    dev = harness.DeviceInputs(inp, dev_name)
    # the workload's own split choice (uniform splits for the MHA step) unless --num-splits
    plan_splits = wl.num_splits if args.num_splits < 0 else args.num_splits
    attn = binding.DecodeAttention(harness.problem_for(inp, mode=args.mode), plan_splits)
    stream = torch.cuda.current_stream()
    flush = L2Flush(dev_name)
    B, H, d = wl.batch, wl.num_q_heads, wl.head_dim
    out = torch.empty((B, H, d), dtype=workloads.TORCH_DTYPES[wl.out_dtype], device=dev_name)
    lse = torch.empty((B, H), dtype=torch.float32, device=dev_name)
    flags = torch.empty((B, H), dtype=torch.uint8, device=dev_name)

    # ---- timed region: whole steps; then the split kernel alone, same steps and flushes ----
    if world > 1:
        dist.barrier()
    t_wall0 = time.perf_counter()
    step_ms, kern_ms, clocks = time_step(attn, dev, wl, args.num_splits, args.steps, args.warmup,
                                         stream, flush, out, lse, flags, ClockSampler(local))
    t_wall = time.perf_counter() - t_wall0
    if world > 1:
        dist.barrier()
    ms, kern_med = max_over_ranks([statistics.median(step_ms), statistics.median(kern_ms)],
                                  dev_name)
    stats = attn.run(dev.q, dev.k, dev.v, dev.bt, dev.sl, wl.scale, args.num_splits,
                     want_stats=True)[3]

    # ---- end to end: pinned host inputs -> device -> run -> host results ----
    e2e = None
    if not args.no_e2e:
        hq = inp.q.pin_memory()
        hk = inp.k_cache.pin_memory()
        hv = inp.v_cache.pin_memory()
        hsl = inp.seq_lens.pin_memory()
        hbt = None if inp.block_table is None else inp.block_table.pin_memory()
        hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        hlse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hsl) + ((hbt,) if hbt is not None else ()))
        d2h = hout.numel() * hout.element_size() + hlse.numel() * hlse.element_size()
        e_steps = max(5, min(args.steps, 20))
        es = [torch.cuda.Event(enable_timing=True) for _ in range(e_steps)]
        ee = [torch.cuda.Event(enable_timing=True) for _ in range(e_steps)]
        for i in range(e_steps + 2):
            j = i - 2
            if j >= 0:
                es[j].record(stream)
            dev.q.copy_(hq, non_blocking=True)
            dev.k.copy_(hk, non_blocking=True)
            dev.v.copy_(hv, non_blocking=True)
            dev.sl.copy_(hsl, non_blocking=True)
            if hbt is not None:
                dev.bt.copy_(hbt, non_blocking=True)
            attn.run(dev.q, dev.k, dev.v, dev.bt, dev.sl, wl.scale, args.num_splits, out=out,
                     out_lse=lse, row_flags=flags, stream=stream)
            hout.copy_(out, non_blocking=True)
            hlse.copy_(lse, non_blocking=True)
            if j >= 0:
                ee[j].record(stream)
            stream.synchronize()
        e2e_ms = statistics.median([a.elapsed_time(b) for a, b in zip(es, ee)])
        e2e_ms = max_over_ranks([e2e_ms], dev_name)[0]
        e2e = {"value": round(world * kv_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": round(e2e_ms, 4)}

    peak, peak_kind = measured_peaks()
    side = []
    if rank == 0 and world == 1 and not args.no_side and args.workload == "gqa32k" \
            and args.num_splits < 0:
        side = [measure_side(n, m, sp, args, dev_name, stream, flush, peak, peak_kind)
                for n, m, sp in SIDE_WORKLOADS]

    if world > 1:
        dist.barrier()
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    achieved = kv_bytes / (kern_med * 1e-3) / 1e9
    value = world * kv_bytes / (ms * 1e-3) / 1e9
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 5),
        "us_per_step": spread(step_ms),
        "pct_hbm_peak": round(100 * value / world / peak, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded N(0,1), workloads.py recipe)",
        "config": {"workload": wl.name, "batch": wl.batch, "q_heads": wl.num_q_heads,
                   "kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim,
                   "kv_tokens_per_seq": int(inp.seq_lens.max()), "kv_dtype": wl.kv_storage,
                   "out_dtype": wl.out_dtype, "softmax": args.mode,
                   "splits": (args.num_splits if args.num_splits >= 0 else
                              (f"{wl.num_splits} uniform splits" if wl.num_splits > 0
                               else "heuristic (balanced shares)")),
                   "grid_ctas": attn.info.grid_ctas, "stages": attn.info.stages,
                   "split_tokens": [stats.split_tokens_min, stats.split_tokens],
                   "kv_bytes_per_step": kv_bytes,
                   "inputs_sha256": workloads.input_digest(inp),
                   "kv_heads_per_group": attn.info.kv_heads_per_group,
                   "timing": "value and ms_per_step from the median step; us_per_step gives median, min, p90 and mean",
                   "l2": f"flushed before every timed step: {FLUSH_BYTES >> 20} MiB written, then {FLUSH_BYTES >> 20} MiB of another buffer read (evicts the dirty lines)",
                   "host_ahead": f"a {HOST_AHEAD_CYCLES}-cycle device spin precedes each timed step, outside its events, so host call overhead is not timed as device time (e2e times it)",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_source": f"{peak_kind} hbm_gbs",
                     "kernel": "decode_split_kernel", "kernel_us": spread(kern_ms),
                     "traffic": profiled_traffic(wl.name)},
        "clocks": clocks,
        "gpu_launches": launches_per_step(args.mode) * args.steps,
        "e2e": e2e,
        "wall_s_timed": round(t_wall, 3),
    }
    if args.mode != "sync":
        line["rows_flagged"] = int(stats.rows_flagged)
        line["splits_flagged"] = int(stats.splits_flagged)
    if side:
        line["workloads"] = side
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp, args.cpu_seconds, out)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def cpu_baseline(inp, seconds, out=None):
    """The float64 CPU oracle, as it stands, on this host's cores over the same inputs: with
    one thread per host core (the headline baseline) and with a single thread. When `out`
    (the GPU result of the timed launch configuration on these inputs) is given, the oracle's
    result also checks it, within the parity tolerance."""
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import _parity
    import oracle
    threads = oracle.host_threads()
    rows = inp.wl.batch * inp.wl.num_q_heads

    def timed(nthreads, budget):
        t0 = time.perf_counter()
        n = 0
        ref = None
        while True:
            ref = _parity.run_oracle(inp, nthreads=nthreads)[0]
            n += 1
            if time.perf_counter() - t0 >= budget:
                break
        return (time.perf_counter() - t0) / n, n, ref

    dt, n, ref = timed(threads, seconds)
    if out is not None:
        _parity.compare(out, ref, inp.wl.out_dtype, where="bench output vs oracle")
    dt1, n1, _ = timed(1, seconds / 2)
    return {"value": round(inp.kv_bytes() / dt / 1e9, 4), "unit": "GB/s", "cores": threads,
            "kind": "oracle", "ms_per_step": round(dt * 1e3, 2),
            "sample": f"the whole workload ({rows} query rows, every token), {n} passes",
            "checked_gpu_output": out is not None,
            "single_thread": {"value": round(inp.kv_bytes() / dt1 / 1e9, 4), "unit": "GB/s",
                              "cores": 1, "ms_per_step": round(dt1 * 1e3, 2),
                              "sample": f"the whole workload, {n1} passes"}}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import _parity
    import oracle
    from decode_attention_attn_gb300 import workloads
    wl = workloads.get(args.workload).replace(mode=args.mode)
    inp = workloads.generate(wl)
    threads = oracle.host_threads()
    for _ in range(args.warmup):
        _parity.run_oracle(inp, nthreads=threads)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        _parity.run_oracle(inp, nthreads=threads)
        times.append(time.perf_counter() - t0)
    dt = sum(times) / len(times)
    value = inp.kv_bytes() / dt / 1e9
    rows = wl.batch * wl.num_q_heads
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,1), workloads.py recipe)",
        "config": {"workload": wl.name, "softmax": args.mode,
                   "kv_bytes_per_step": inp.kv_bytes()},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle",
                         "sample": f"the whole workload ({rows} query rows, every token) per step"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


HIST_LO, HIST_HI, HIST_BINS = -16.0, 16.0, 4096


def oracle_histogram(inp):
    """Histogram of the oracle's float64 logits, slots as the library lays them out."""
    import numpy as np
    import oracle
    from decode_attention_attn_gb300 import workloads
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import _parity
    bt = None if inp.block_table is None else inp.block_table.numpy()
    x = oracle.logits(_parity.oracle_shape(inp), workloads.bits(inp.q), workloads.bits(inp.k_cache),
                      bt, inp.seq_lens.numpy(), inp.wl.scale)
    w = (HIST_HI - HIST_LO) / HIST_BINS

    def slots(v):
        i = np.floor((v - HIST_LO) / w)
        return np.where(i < 0, 0, np.where(i >= HIST_BINS, HIST_BINS + 1, i + 1)).astype(np.int64)
    tol = 2e-5 * (1.0 + np.abs(x))
    edge = int(np.count_nonzero(slots(x - tol) != slots(x + tol)))
    return np.bincount(slots(x), minlength=HIST_BINS + 2), edge


def run_histogram(args):
    """The calibration pass (decode_attn_logit_histogram) timed like the decode step: one
    launch per step over the workload's K, L2 flushed before each step."""
    import numpy as np
    import torch
    from decode_attention_attn_gb300 import binding, harness, workloads

    rank, world, local = dist_env()
    if world > 1:
        print(json.dumps({"op": "logit_histogram", "unavailable": "one GPU only"}))
        return
    torch.cuda.set_device(local)
    wl = workloads.get(args.workload)
    inp = workloads.generate(wl)
    k_bytes = inp.kv_bytes() // 2
    dev = harness.DeviceInputs(inp)
    attn = binding.DecodeAttention(harness.problem_for(inp, mode="sync"), 0)
    stream = torch.cuda.current_stream()
    flush = L2Flush(f"cuda:{local}")
    counts = torch.zeros(HIST_BINS + 2, dtype=torch.int64, device=f"cuda:{local}")

    def step():
        binding.decode_attn_logit_histogram(
            attn.plan, dev.q.data_ptr(), dev.k.data_ptr(),
            None if dev.bt is None else dev.bt.data_ptr(), dev.sl.data_ptr(), wl.scale,
            HIST_LO, HIST_HI, HIST_BINS, counts.data_ptr(), stream.cuda_stream)

    for _ in range(max(3, args.warmup)):
        flush()
        step()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(local)
    torch.cuda.synchronize()
    sampler.start()
    for i in range(args.steps):
        flush()
        torch.cuda._sleep(HOST_AHEAD_CYCLES)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / args.steps

    # end to end: pinned q, K, lengths and table in; the counts out
    e2e = None
    hq, hk, hsl = inp.q.pin_memory(), inp.k_cache.pin_memory(), inp.seq_lens.pin_memory()
    hbt = None if inp.block_table is None else inp.block_table.pin_memory()
    hcounts = torch.empty(counts.shape, dtype=counts.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hsl) + ((hbt,) if hbt is not None else ()))
    d2h = hcounts.numel() * hcounts.element_size()
    e_steps = 1 if args.no_e2e else max(5, min(args.steps, 20))
    es = [torch.cuda.Event(enable_timing=True) for _ in range(e_steps)]
    ee = [torch.cuda.Event(enable_timing=True) for _ in range(e_steps)]
    for i in range(e_steps):   # (one untimed pass with --no-e2e: the counts the check reads)
        es[i].record(stream)
        dev.q.copy_(hq, non_blocking=True)
        dev.k.copy_(hk, non_blocking=True)
        dev.sl.copy_(hsl, non_blocking=True)
        if hbt is not None:
            dev.bt.copy_(hbt, non_blocking=True)
        counts.zero_()
        step()
        hcounts.copy_(counts, non_blocking=True)
        ee[i].record(stream)
        stream.synchronize()
    if not args.no_e2e:
        e2e_ms = sum(s.elapsed_time(e) for s, e in zip(es, ee)) / e_steps
        e2e = {"value": round(k_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": round(e2e_ms, 4)}

    # the oracle's logits plus a numpy histogram, timed on the host cores; its result also
    # checks the last GPU histogram (one step's, from the e2e loop): slots may differ only by
    # logits within the fp32 error of a bin edge
    cpu = None
    if not args.no_cpu_baseline:
        t0 = time.perf_counter()
        n = 0
        while n == 0 or time.perf_counter() - t0 < args.cpu_seconds:
            ref, edge = oracle_histogram(inp)
            n += 1
        cpu_dt = (time.perf_counter() - t0) / n
        diff = int(np.abs(hcounts.numpy() - ref).sum())
        assert diff <= 2 * edge, f"histogram differs from the oracle's by {diff} (> 2 x {edge})"
        cpu = {"value": round(k_bytes / cpu_dt / 1e9, 4), "unit": "GB/s", "cores": 1,
               "kind": "oracle", "ms_per_step": round(cpu_dt * 1e3, 2),
               "sample": f"the whole workload (every logit, float64) plus a numpy histogram, "
                         f"{n} passes", "checked_gpu_output": True}

    peak, peak_kind = measured_peaks()
    achieved = k_bytes / (ms * 1e-3) / 1e9
    line = {
        "op": "logit_histogram",
        "metric": "logit-histogram K-read GB/s (phi calibration pass)",
        "value": round(achieved, 2),
        "unit": "GB/s",
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 5),
        "us_per_step": round(ms * 1e3, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded N(0,1), workloads.py recipe)",
        "config": {"workload": wl.name, "k_bytes_per_step": k_bytes,
                   "bins": HIST_BINS, "range": [HIST_LO, HIST_HI],
                   "l2": f"flushed before every timed step: {FLUSH_BYTES >> 20} MiB written, then {FLUSH_BYTES >> 20} MiB of another buffer read"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_source": f"{peak_kind} hbm_gbs",
                     "kernel": ("logit_histogram_mma_kernel"
                                if wl.kv_storage in ("bf16", "e4m3") else "logit_histogram_kernel"),
                     "traffic": profiled_traffic(wl.name, "logit_histogram")},
        "clocks": clocks,
        "gpu_launches": args.steps,
        "e2e": e2e,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.op == "logit_histogram":
        run_histogram(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
