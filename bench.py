#!/usr/bin/env python3
"""Benchmark of the integer motion SAD + PSNR SSE hot path on GB300.

Default workload: 50 pairs of 3840x2160 8-bit 4:2:0 pictures (reference from
the smooth generator, distorted = reference + N(0, 3^2)).  One step = one pass
of the whole hot path over the 50 pairs: motion blur + SAD on the reference
luma and SSE of Y, U, V -- one fused launch (motion_psnr_yuv420_batch).
Inputs are resident in HBM before timing; the 1.24 GB working set is ~10x the
L2, so no flush is needed between steps.

Prints ONE JSON line (rank 0).  `value` is pairs/s over all ranks (weak
scaling: every rank processes its own 50 pairs); `roofline` reports the fused
kernel against the measured HBM copy bandwidth; `e2e` is the same metric
through the host-buffer entry point (pinned host pictures in, results out);
`cpu_baseline` is the CPU oracle on a bounded sample.  `--impl reference`
times the oracle itself as the reference arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import re
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "frames/s and HBM GB/s (fraction of roofline) for 4K 8-bit motion SAD + PSNR"
WORKLOAD = "yuv420_3840x2160_u8_pairs"
FALLBACK_HBM_GBS = 6800.0


def algorithmic_bytes_per_pair(w: int, h: int, bpc: int) -> int:
    """Minimum bytes one pair must move: every sample of the reference and the
    distorted picture read once (Y + U + V); the motion blur reuses the
    reference luma already read for the SSE."""
    s = 1 if bpc == 8 else 2
    cw, ch = (w + 1) // 2, (h + 1) // 2
    return 2 * (w * h + 2 * cw * ch) * s


def motion_tile_rows(w: int, h: int, batch: int, v2: bool = False) -> int:
    """Tile height (32 or 16) of a batched motion-only launch on this device:
    128 x 16 tiles when the 128 x 32 tiles fit in one wave of 4 per SM."""
    import torch

    import integer_image_filter_gb300 as iif
    slots = 4 * torch.cuda.get_device_properties(0).multi_processor_count
    return iif.motion_launch_shape(w, h, batch, slots, v2=v2)


def motion_kernel_name(bpc: int, v2: bool = False, tile_rows: int = 32) -> str:
    """The key of a motion-only launch in the recorded profiles."""
    return "motion_tma_kernel<%s, %s%s>" % ("uint8_t" if bpc == 8 else "uint16_t",
                                              "motion_v2" if v2 else "motion",
                                              "" if tile_rows == 32 else ", 16-row tiles")


def numa_placement(host_tensor) -> dict:
    """NUMA nodes of the host, the node the GPU is attached to, and the node
    that holds the first page of a pinned host buffer (move_pages query)."""
    import ctypes
    import glob

    import torch
    info = {}
    try:
        info["host_nodes"] = sorted(int(p.rsplit("node", 1)[1])
                                    for p in glob.glob("/sys/devices/system/node/node[0-9]*"))
    except Exception:
        info["host_nodes"] = None
    try:
        pr = torch.cuda.get_device_properties(0)
        bus = "%04x:%02x:%02x.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
        with open(f"/sys/bus/pci/devices/{bus}/numa_node") as f:
            info["gpu_node"] = int(f.read().strip())
    except Exception:
        info["gpu_node"] = None
    try:
        libc = ctypes.CDLL(None, use_errno=True)
        nr = 239 if os.uname().machine == "aarch64" else 279      # move_pages
        page = (ctypes.c_void_p * 1)(host_tensor.data_ptr())
        status = (ctypes.c_int * 1)(-1)
        rc = libc.syscall(nr, 0, ctypes.c_ulong(1), page, None, status, 0)
        info["pinned_pages_node"] = int(status[0]) if rc == 0 and status[0] >= 0 else None
    except Exception:
        info["pinned_pages_node"] = None
    return info


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# the sources that make up the fused TMA kernel; its recorded DRAM traffic is
# only reported while they are unchanged since the capture
KERNEL_SOURCES = ("motion_tma.cu", "tile_geometry.cuh", "motion_common.cuh", "motion_internal.h",
                  "bounds_check.cuh")


def _code_tokens(text: str) -> bytes:
    """The source without comments and with whitespace runs collapsed, so that
    a comment or layout edit does not count as a kernel change (string
    literals in these sources hold no comment markers)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split()).encode()


def kernel_source_hash() -> str:
    csrc = os.path.join(ROOT, "integer_image_filter_gb300", "csrc")
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(f.encode() + b"\0" + _code_tokens(fh.read()))
    return h.hexdigest()[:16]


# Warp instructions each unit can take per SM clock, from the measured rates
# (profiles/pipe_rates_gb300.md: every integer class at 64 lanes per SM clock
# = 2 warp instructions; the 4 schedulers issue one warp instruction each).
PIPE_WARP_INST_PER_SM_CLOCK = {"issue": 4.0, "alu": 2.0, "fmaheavy": 2.0}


def recorded_inst_mix(kernel: str, workload: str):
    """ncu instruction counts per launch (total and per pipe) from the committed
    record, or None when the kernel sources changed since the capture."""
    p = os.path.join(ROOT, "profiles", "inst_mix.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d[kernel][workload]
        if e.get("source_hash") != kernel_source_hash():
            return None
        return e
    except Exception:
        return None


def instruction_co_bound(kernel: str, workload: str, launch_ms: float, sm_mhz,
                         units: float | None = None, batch: int | None = None) -> dict:
    """The integer co-bound of a launch (or a step of `units` frames or pairs):
    for the issue slots (4 warp instructions per SM clock) and each integer pipe
    (ALU and FMA-heavy, 2 per SM clock), the time its recorded instruction count
    needs at that rate ÷ the measured time; the largest is the bound.  Counts
    are recorded per captured launch of rec["units"] units and scaled."""
    import torch
    rec = recorded_inst_mix(kernel, workload)
    if rec is None:
        return {"available": False,
                "why": "no ncu instruction counts recorded for these kernel sources and this launch"}
    if batch is not None and rec.get("batch") not in (None, batch):
        return {"available": False, "why": "instruction counts recorded for batch %s" % rec.get("batch")}
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    mhz = float(sm_mhz) if sm_mhz else 2070.0
    scale = (units / float(rec["units"])) if units else 1.0
    per = {}
    for unit, rate in PIPE_WARP_INST_PER_SM_CLOCK.items():
        count = scale * float(rec["inst"] if unit == "issue" else rec[unit])
        need_ms = count / (rate * sms * mhz * 1e6) * 1e3
        per[unit] = {"warp_inst_per_launch": count, "ms_at_peak": need_ms, "frac": need_ms / launch_ms}
    bound = max(per, key=lambda k: per[k]["frac"])
    peak = PIPE_WARP_INST_PER_SM_CLOCK[bound] * sms * mhz * 1e6 / 1e9
    return {"bound": bound, "achieved": per[bound]["warp_inst_per_launch"] / (launch_ms * 1e-3) / 1e9,
            "peak": peak, "unit": "G warp instructions/s", "frac": per[bound]["frac"],
            "per_unit": per, "thread_inst_per_pixel": rec.get("thread_inst_per_pixel"),
            "peak_basis": (f"{sms} SMs x {PIPE_WARP_INST_PER_SM_CLOCK[bound]:.0f} warp instructions per "
                           f"SM clock ({bound}; measured rates, profiles/pipe_rates_gb300.md) x {mhz:.0f} MHz"),
            "counts": "profiles/inst_mix.json (ncu, same kernel sources and launch)"}


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel sources changed since the capture."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d[kernel][workload]
        if e.get("source_hash") != kernel_source_hash():
            return None
        return int(e["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.times = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)
                self.times.append(time.time())

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float | None = None, t1: float | None = None):
        """Clocks over the samples taken in [t0, t1] (all samples by default)."""
        rows = [r for r, t in zip(self.rows, self.times)
                if (t0 is None or t >= t0) and (t1 is None or t <= t1)]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def sustained_launches(run, stream, min_seconds: float = 1.0, min_launches: int = 200,
                       max_launches: int = 100000) -> dict:
    """Repeat one unit of work (`run` enqueues it on `stream`) back to back for
    at least min_seconds and min_launches, each bracketed by CUDA events on the
    stream; returns the distribution of the per-launch device times (ms)."""
    import torch
    probe = []
    for _ in range(5):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        run()
        b.record(stream)
        probe.append((a, b))
    torch.cuda.synchronize()
    est = max(statistics.median(a.elapsed_time(b) for a, b in probe), 1e-3)
    n = int(min(max_launches, max(min_launches, min_seconds * 1e3 / est)))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    t0 = time.time()
    for a, b in ev:
        a.record(stream)
        run()
        b.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    ms = sorted(a.elapsed_time(b) for a, b in ev)
    return {"launches": n, "seconds": ev[0][0].elapsed_time(ev[-1][1]) / 1e3,
            "median_ms": statistics.median(ms), "mean_ms": statistics.mean(ms),
            "p10_ms": ms[len(ms) // 10], "p90_ms": ms[(9 * len(ms)) // 10], "t0": t0, "t1": t1}


def cpu_oracle_rate(batch, budget_s: float, min_pairs: int = 2):
    """The oracle, as it stands, on a bounded sample of the workload: motion
    SAD over consecutive reference lumas plus SSE of Y, U, V for each pair,
    single-threaded.  Returns (pairs/s, pairs, seconds)."""
    import oracle
    o = oracle.Oracle()
    t0 = time.perf_counter()
    done = 0
    while done < batch.n and (done < min_pairs or time.perf_counter() - t0 < budget_s):
        lo = max(done - 1, 0)
        o.motion_sad_sequence(batch.ref_y[lo:done + 1], batch.bpc)
        o.sse(batch.ref_y[done], batch.dist_y[done], batch.bpc)
        o.sse(batch.ref_u[done], batch.dist_u[done], batch.bpc)
        o.sse(batch.ref_v[done], batch.dist_v[done], batch.bpc)
        done += 1
    dt = time.perf_counter() - t0
    return done / dt, done, dt


def cpu_oracle_parallel_rate(batch, budget_s: float, cores: int):
    """The same per-pair oracle work (as cpu_oracle_rate) spread over `cores`
    threads for about budget_s seconds, cycling through the batch's pairs (the
    oracle's C calls release the GIL).  Returns (pairs/s, pairs, seconds)."""
    import itertools
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    o = oracle.Oracle()
    nxt = itertools.count()
    lock = threading.Lock()
    t0 = time.perf_counter()
    stop = t0 + budget_s

    def worker():
        done = 0
        while time.perf_counter() < stop:
            with lock:
                i = next(nxt) % batch.n
            lo = max(i - 1, 0)
            o.motion_sad_sequence(batch.ref_y[lo:i + 1], batch.bpc)
            o.sse(batch.ref_y[i], batch.dist_y[i], batch.bpc)
            o.sse(batch.ref_u[i], batch.dist_u[i], batch.bpc)
            o.sse(batch.ref_v[i], batch.dist_v[i], batch.bpc)
            done += 1
        return done

    with ThreadPoolExecutor(cores) as ex:
        total = sum(f.result() for f in [ex.submit(worker) for _ in range(cores)])
    dt = time.perf_counter() - t0
    return total / dt, total, dt


def run_reference(args):
    """The reference arm: the CPU oracle, as it stands, on the machine's host cores.
    Each step is a bounded sample of the workload -- 2 pairs per core -- split
    into one contiguous run of pairs per thread (each run re-blurs the frame
    before it, as a shard does); the oracle's C calls release the GIL."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    import synth
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    per_thread = 2
    pairs_per_step = per_thread * cores
    batch = synth.make(WORKLOAD, n=pairs_per_step + 1)   # reused by every step
    o = oracle.Oracle()

    def run(t):
        s = 1 + t * per_thread
        o.motion_sad_sequence(batch.ref_y[s - 1:s + per_thread], batch.bpc)
        for j in range(s, s + per_thread):
            o.sse(batch.ref_y[j], batch.dist_y[j], batch.bpc)
            o.sse(batch.ref_u[j], batch.dist_u[j], batch.bpc)
            o.sse(batch.ref_v[j], batch.dist_v[j], batch.bpc)

    with ThreadPoolExecutor(cores) as ex:
        def step():
            list(ex.map(run, range(cores)))

        for _ in range(args.warmup):
            step()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            step()
        dt = time.perf_counter() - t0
    value = pairs_per_step * args.steps / dt
    sample = (f"{pairs_per_step} pairs of 3840x2160 8-bit 4:2:0 per step over {cores} threads, "
              f"{per_thread} consecutive pairs per thread (motion SAD on the reference luma, "
              f"blurring {per_thread + 1} frames, + SSE of Y, U, V), the C oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "frames/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * dt / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": {"workload": WORKLOAD, "w": 3840, "h": 2160, "bpc": 8,
                   "pairs_per_step": pairs_per_step},
        "cpu_baseline": {"value": value, "unit": "frames/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "frames/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def _graph_of(step, dev, stream):
    """One call of step() captured as a CUDA graph (after a direct warm-up on a
    side stream); returns the replay function."""
    import torch
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step()
    stream.wait_stream(side)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize(dev)
    return graph.replay


def secondary_measurements(dev, stream, planes, n_pairs: int, w420: int, h420: int, clocks,
                           min_seconds: float = 0.4) -> dict:
    """The other configurations, each timed as back-to-back steps for at least
    min_seconds (median step time) with the clocks of its own window: the 10-bit
    4K sequence at batch 32 and swept over batch 1..32, the 1080p sequence at
    batch 16, the 576x324 sequence as one 48-frame launch (host-launched and as
    a CUDA graph), the 64x48 pair per submitted frame, and the stand-alone SSE
    and moment launches on the 4:2:0 pairs of the default step."""
    import math

    import numpy as np
    import torch

    import integer_image_filter_gb300 as iif
    import synth
    peak, peak_kind = peaks()
    out = {}

    def seq_entry(name, batches, graph=False):
        c = synth.CONFIGS[name]
        w, h, bpc = c["w"], c["h"], c["bpc"]
        frames = synth.make(name)
        n = frames.shape[0]
        s = 1 if bpc == 8 else 2
        d = torch.from_numpy(frames.view(np.int16) if bpc > 8 else frames).to(dev)
        sad = torch.zeros(n, dtype=torch.int64, device=dev)
        res = {}
        with iif.MotionContext(w, h, bpc) as ctx:
            for batch in batches:
                def step():
                    cur = torch.cuda.current_stream(dev)
                    ctx.reset()
                    for b0 in range(0, n, batch):
                        ctx.submit_batch(d[b0:b0 + batch], sad[b0:b0 + batch], stream=cur)
                for _ in range(3):
                    step()
                torch.cuda.synchronize(dev)
                run = _graph_of(step, dev, stream) if graph else step
                for _ in range(3):
                    run()
                r = sustained_launches(run, stream, min_seconds=min_seconds, min_launches=20)
                ms = r["median_ms"]
                launches = math.ceil(n / batch)
                alg = w * h * s * n
                res[batch] = {"frames_per_s": n / (ms * 1e-3), "gb_per_s": alg / (ms * 1e-3) / 1e9,
                              "hbm_frac": alg / (ms * 1e-3) / 1e9 / peak, "step_ms": ms,
                              "kernel_ms_per_launch": ms / launches, "batch": batch,
                              "frames_per_step": n, "steps_timed": r["launches"],
                              "cuda_graph": graph,
                              "clocks": clocks.summary(r["t0"], r["t1"])}
                rows = motion_tile_rows(w, h, batch)
                res[batch]["tile_rows"] = rows
                res[batch]["roofline"] = seq_roofline(alg, ms, peak, peak_kind,
                                                      motion_kernel_name(bpc, tile_rows=rows), name,
                                                      n, res[batch]["clocks"].get("sm_mhz"), batch)
        return res

    t_all = time.time()
    u10 = seq_entry("seq_3840x2160_u10", [32, 1, 2, 4, 8, 16])
    out["seq_3840x2160_u10"] = dict(u10[32], sweep={b: {"frames_per_s": v["frames_per_s"],
                                                        "hbm_frac": v["hbm_frac"],
                                                        "kernel_ms_per_launch": v["kernel_ms_per_launch"]}
                                                    for b, v in sorted(u10.items())})
    out["seq_1920x1080_u8_cuts"] = seq_entry("seq_1920x1080_u8_cuts", [16])[16]
    out["seq_576x324_u8"] = seq_entry("seq_576x324_u8", [48])[48]
    out["seq_576x324_u8_graph"] = seq_entry("seq_576x324_u8", [48], graph=True)[48]
    # the 64x48 pair: one submitted frame per call (launch + 16-byte readback)
    pair = synth.make("pair_64x48_u8")
    dp = torch.from_numpy(pair).to(dev)
    with iif.MotionContext(64, 48, 8) as ctx:
        for _ in range(20):
            ctx.submit(dp[0])
        t0 = time.perf_counter()
        k = 0
        while time.perf_counter() - t0 < min_seconds:
            ctx.reset()
            ctx.submit(dp[0])
            ctx.submit(dp[1])
            k += 2
        us = (time.perf_counter() - t0) / k * 1e6
    out["pair_64x48_u8"] = {"us_per_submitted_frame": us, "frames": k}
    # stand-alone SSE and moment sums on the default step's pairs
    sse = torch.zeros((n_pairs, 3), dtype=torch.int64, device=dev)
    mom = torch.zeros((n_pairs, 4), dtype=torch.int64, device=dev)
    for name, fn, alg in (
            ("sse_yuv420_%dx%d_u8_pairs" % (w420, h420),
             lambda: iif.psnr_sse_yuv420_batch(w420, h420, 8, *planes, sse, stream=stream),
             algorithmic_bytes_per_pair(w420, h420, 8) * n_pairs),
            ("moment_%dx%d_u8_pairs" % (w420, h420),
             lambda: iif.moment_sums_batch(planes[0], planes[3], 8, mom, stream=stream),
             2 * w420 * h420 * n_pairs)):
        for _ in range(3):
            fn()
        r = sustained_launches(fn, stream, min_seconds=min_seconds, min_launches=50)
        ms = r["median_ms"]
        out[name] = {"pairs_per_s": n_pairs / (ms * 1e-3), "gb_per_s": alg / (ms * 1e-3) / 1e9,
                     "hbm_frac": alg / (ms * 1e-3) / 1e9 / peak, "kernel_ms": ms,
                     "launches_timed": r["launches"], "clocks": clocks.summary(r["t0"], r["t1"])}
    out["seconds"] = time.time() - t_all
    return out


def run_gpu(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import integer_image_filter_gb300 as iif
    import synth

    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    iif.load_library()

    n = args.pairs
    # every rank draws its own pairs (weak scaling: a disjoint shard per rank)
    batch = synth.yuv420_pairs(4 + 1000 * rank, n, args.w, args.h, max_shift=2, dist_sigma=3.0)
    host = [torch.from_numpy(p) for p in batch.planes()]
    planes = [p.to(dev) for p in host]
    sad = torch.zeros(n, dtype=torch.int64, device=dev)
    sse = torch.zeros((n, 3), dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev)
    ctx = iif.MotionContext(args.w, args.h, 8)

    def step():
        ctx.reset()
        ctx.yuv420_batch(*planes, sad, sse, stream=stream)

    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize(dev)

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    launches0 = iif.motion_kernel_launch_count()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    all0 = torch.cuda.Event(enable_timing=True)
    all1 = torch.cuda.Event(enable_timing=True)
    all0.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    all1.record(stream)
    torch.cuda.synchronize(dev)
    launches = iif.motion_kernel_launch_count() - launches0
    total_ms = all0.elapsed_time(all1)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    if ws > 1:
        t = torch.tensor([total_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
        dist.barrier()
    # the same step repeated back to back for at least a second: the launch
    # time the roofline uses (median of >= 200 launch events), with the clocks
    # of that window
    sus = sustained_launches(step, stream, min_seconds=args.sustain_seconds, min_launches=200)
    sus["clocks"] = clocks.summary(sus["t0"], sus["t1"])
    secondary = None
    streams = None
    if ws == 1 and not args.no_secondary:
        secondary = secondary_measurements(dev, stream, planes, n, args.w, args.h, clocks)
        streams = hbm_stream_ceilings()
    clocks.stop()

    # the same metric end to end: pinned host pictures -> device -> results on the host
    pinned = [p.pin_memory() for p in host]
    for _ in range(1):
        ctx.reset()
        ctx.yuv420_batch_host(*pinned)
    e2e_steps = max(1, min(args.steps, 10))
    if ws > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        ctx.reset()
        h_sad, h_sse = ctx.yuv420_batch_host(*pinned)
    e2e_s = time.perf_counter() - t0
    if ws > 1:
        t = torch.tensor([e2e_s], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_s = float(t.item())
    h2d = sum(p.numel() * p.element_size() for p in pinned)
    numa = numa_placement(pinned[0])
    # this box's pinned host->device rate now (a plain copy of the reference luma
    # onto its own device copy, best of 3): the ceiling of the end-to-end rate
    link = 0.0
    for _ in range(3):
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        planes[0].copy_(pinned[0], non_blocking=True)
        c1.record(stream)
        torch.cuda.synchronize(dev)
        link = max(link, pinned[0].numel() * pinned[0].element_size() / (c0.elapsed_time(c1) * 1e-3) / 1e9)
    d2h = h_sad.nbytes + h_sse.nbytes
    dev_sad = sad.cpu().numpy().astype(np.uint64)
    dev_sse = sse.cpu().numpy().astype(np.uint64)
    assert np.array_equal(dev_sad, h_sad) and np.array_equal(dev_sse, h_sse), \
        "device-resident and host-buffer paths disagree"

    if rank != 0:
        ctx.close()
        if ws > 1:
            dist.destroy_process_group()
        return 0

    peak, peak_kind = peaks()
    bytes_per_launch = algorithmic_bytes_per_pair(args.w, args.h, 8) * n
    kern_ms = sus["median_ms"]
    clk = clocks.summary(None, sus["t1"])
    achieved = bytes_per_launch / (kern_ms * 1e-3) / 1e9
    value = ws * n * args.steps / (total_ms * 1e-3)
    cpu = None
    if not args.no_cpu_baseline and ws == 1:
        rate, done, secs = cpu_oracle_rate(batch, args.cpu_seconds)
        cpu = {"value": rate, "unit": "frames/s", "cores": 1, "kind": "oracle",
               "sample": (f"the first {done} of the step's {n} pairs ({args.w}x{args.h} 8-bit "
                          f"4:2:0): motion SAD + Y/U/V SSE, single-threaded C oracle, "
                          f"{secs:.1f} s")}
        cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
        if cores > 1 and args.cpu_seconds > 0:
            prate, pdone, psecs = cpu_oracle_parallel_rate(batch, args.cpu_seconds / 2, cores)
            cpu["parallel"] = {"value": prate, "unit": "frames/s", "cores": cores,
                               "sample": (f"{pdone} pairs of the step's {n} (cycled) over {cores} "
                                          f"threads of the same oracle, {psecs:.1f} s")}
    line = {
        "metric": METRIC, "value": value, "unit": "frames/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic",
        "config": {"workload": WORKLOAD if (args.w, args.h, n) == (3840, 2160, 50) else
                   f"yuv420_{args.w}x{args.h}_u8_pairs", "w": args.w, "h": args.h, "bpc": 8,
                   "pairs_per_step": n, "launches_per_step": launches / max(args.steps, 1),
                   "l2": f"inputs {bytes_per_launch / 1e9:.2f} GB per step vs 129 MB L2 (no flush)",
                   "parallelism": f"dp{ws} (disjoint pairs per rank, no collective)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": recorded_traffic("motion_tma_kernel<uint8_t, fused>", WORKLOAD),
                     "kernel": "motion_tma_kernel<uint8_t, fused>",
                     "algorithmic_bytes_per_launch": bytes_per_launch,
                     "kernel_ms": kern_ms,
                     "kernel_ms_basis": ("median of %d launch events over %.2f s of back-to-back steps "
                                         "(each step: the call's two output memsets and the fused "
                                         "kernel); the timed steps' mean is %.4f ms"
                                         % (sus["launches"], sus["seconds"], statistics.mean(step_ms))),
                     "sustained": {k: sus[k] for k in ("launches", "seconds", "median_ms", "mean_ms",
                                                        "p10_ms", "p90_ms", "clocks")},
                     "alu": instruction_co_bound("motion_tma_kernel<uint8_t, fused>", WORKLOAD, kern_ms,
                                                 (clk or {}).get("sm_mhz")),
                     # the launch reads 1.25 GB and writes 16 MB: against this box's read-only
                     # stream rate as well as the copy bandwidth of MEASURED_PEAKS.json
                     "stream_ceilings": read_only_ceiling(streams, secondary, achieved)},
        "cpu_baseline": cpu,
        "e2e": {"value": ws * n * e2e_steps / e2e_s, "unit": "frames/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "host_link_gbs": h2d * e2e_steps / e2e_s / 1e9,
                "link_h2d_ceiling_gbs": link, "frac_of_link": h2d * e2e_steps / e2e_s / 1e9 / link,
                "numa": numa},
        "gpu_launches": launches,
        "clocks": clk,
        "secondary": secondary,
    }
    print(json.dumps(line), flush=True)
    ctx.close()
    if ws > 1:
        dist.destroy_process_group()
    return 0


def seq_roofline(alg_bytes: int, ms: float, peak_gbs: float, peak_kind: str, kernel: str,
                 workload: str, frames: int, sm_mhz=None, batch: int | None = None) -> dict:
    """Roofline of a motion-only step: HBM (algorithmic bytes, every frame read
    once, at the measured copy bandwidth) is the roof; beside it the integer
    co-bound of the same time from the kernel's recorded instruction counts
    (instruction_co_bound), which is the one these launches run against: 8-bit
    motion needs about 19 instructions per byte read."""
    hbm = {"bound": "hbm", "achieved": alg_bytes / (ms * 1e-3) / 1e9, "peak": peak_gbs,
           "unit": "GB/s", "frac": alg_bytes / (ms * 1e-3) / 1e9 / peak_gbs, "peak_kind": peak_kind,
           "algorithmic_bytes_per_step": alg_bytes}
    hbm["alu"] = instruction_co_bound(kernel, workload, ms, sm_mhz, units=frames, batch=batch)
    return hbm


def run_sequence_workload(args):
    """Motion-only workloads (not the headline): frames/s and GB/s of the
    batched motion kernel on one of the sequence configurations, with the
    batch size of the configuration (or --batch), optionally swept."""
    import numpy as np
    import torch

    import integer_image_filter_gb300 as iif
    import synth

    c = synth.CONFIGS[args.workload]
    w, h, bpc = c["w"], c["h"], c["bpc"]
    frames = synth.make(args.workload)
    if args.trim:
        # drop the last columns and pack the rows tightly: rows of an odd
        # width that the TMA cannot address in place
        w -= args.trim
        frames = np.ascontiguousarray(frames[:, :, :w])
    n = frames.shape[0]
    s = 1 if bpc == 8 else 2
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    d = torch.from_numpy(frames.view(np.int16) if bpc > 8 else frames).to(dev)
    sad = torch.zeros(n, dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev)
    peak, peak_kind = peaks()
    batches = [args.batch] if args.batch else [c.get("batch", n)]
    if args.sweep:
        batches = [1, 2, 4, 8, 16, 32]
    lines = []
    for batch in batches:
        ctx = iif.MotionContext(w, h, bpc)
        if args.generic:
            ctx.set_kernel_path(iif.MOTION_PATH_GENERIC)

        submit = ctx.submit_batch_v2 if args.v2 else ctx.submit_batch

        def step():
            # the calls go to the current stream: the timing stream, or the
            # capture stream of a CUDA graph
            cur = torch.cuda.current_stream(dev)
            ctx.reset()
            for b0 in range(0, n, batch):
                submit(d[b0:b0 + batch], sad[b0:b0 + batch], stream=cur)

        for _ in range(max(args.warmup, 3)):
            step()
        torch.cuda.synchronize(dev)
        run = step
        l0 = iif.motion_kernel_launch_count()
        if args.graph:
            # one step captured as a CUDA graph (the library launches counted at
            # capture are the ones every replay runs)
            side = torch.cuda.Stream(dev)
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                step()
            stream.wait_stream(side)
            torch.cuda.synchronize(dev)
            graph = torch.cuda.CUDAGraph()
            l0 = iif.motion_kernel_launch_count()
            with torch.cuda.graph(graph):
                step()
            launches = iif.motion_kernel_launch_count() - l0
            run = graph.replay
            for _ in range(max(args.warmup, 3)):
                run()
            torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            run()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / args.steps
        if not args.graph:
            launches = (iif.motion_kernel_launch_count() - l0) / args.steps
        rows = 32 if args.generic else motion_tile_rows(w, h, batch, args.v2)
        alg = w * h * s * n
        e2e = None
        if not args.v2 and not args.graph and not args.generic:
            # end to end: the same sequence from pinned host memory through
            # motion_submit_batch_host, chunks of the batch size (uploads
            # overlap the kernels), SADs back to the host
            host = torch.from_numpy(frames.view(np.int16) if bpc > 8 else frames).pin_memory().numpy()
            ctx.reset()
            ctx.submit_batch_host(host, frames_per_chunk=batch)
            t0 = time.perf_counter()
            e2e_steps = max(1, min(args.steps, 10))
            for _ in range(e2e_steps):
                ctx.reset()
                h_sad = ctx.submit_batch_host(host, frames_per_chunk=batch)
            e2e_s = time.perf_counter() - t0
            assert np.array_equal(h_sad, sad.cpu().numpy().astype(np.uint64)), \
                "device-resident and host-buffer paths disagree"
            e2e = {"value": n * e2e_steps / e2e_s, "unit": "frames/s",
                   "h2d_bytes_per_step": int(host.nbytes), "d2h_bytes_per_step": 8 * n}
        lines.append({"metric": "frames/s (batched motion%s SAD)" % ("_v2" if args.v2 else ""),
                      "value": n / (ms * 1e-3),
                      "unit": "frames/s", "n_gpus": 1, "steps": args.steps,
                      "warmup": max(args.warmup, 3), "ms_per_step": ms, "higher_is_better": True,
                      "dtype": "u8" if bpc == 8 else "u16", "data": "synthetic",
                      "config": {"workload": args.workload + ("_v2" if args.v2 else "") +
                                             ("_trim%d" % args.trim if args.trim else ""),
                                 "w": w, "h": h, "bpc": bpc,
                                 "frames_per_step": n, "batch": batch,
                                 "launches_per_step": launches, "cuda_graph": bool(args.graph),
                                 "kernel_path": "generic" if args.generic else "auto",
                                 "tile_rows": rows},
                      "roofline": seq_roofline(alg, ms, peak, peak_kind,
                                               motion_kernel_name(bpc, args.v2, rows),
                                               args.workload, n, batch=batch), "e2e": e2e})
        ctx.close()
    for ln in lines:
        print(json.dumps(ln), flush=True)
    return 0


def run_sse_workload(args):
    """The stand-alone SSE launch (all planes of all pairs) on the 4:2:0 pairs."""
    import torch

    import integer_image_filter_gb300 as iif
    import synth

    n = args.pairs
    batch = synth.yuv420_pairs(4, n, args.w, args.h, max_shift=2, dist_sigma=3.0)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    planes = [torch.from_numpy(p).to(dev) for p in batch.planes()]
    sse = torch.zeros((n, 3), dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        iif.psnr_sse_yuv420_batch(args.w, args.h, 8, *planes, sse, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / args.steps
    peak, peak_kind = peaks()
    alg = algorithmic_bytes_per_pair(args.w, args.h, 8) * n
    print(json.dumps({"metric": "pairs/s (PSNR SSE of Y, U, V)", "value": n / (ms * 1e-3),
                      "unit": "frames/s", "ms_per_step": ms, "steps": args.steps,
                      "config": {"workload": "sse_yuv420_%dx%d_u8_pairs" % (args.w, args.h),
                                 "pairs_per_step": n},
                      "roofline": {"bound": "hbm", "achieved": alg / (ms * 1e-3) / 1e9,
                                   "peak": peak, "unit": "GB/s",
                                   "frac": alg / (ms * 1e-3) / 1e9 / peak,
                                   "peak_kind": peak_kind}}), flush=True)
    return 0


def run_moment_workload(args):
    """Moment sums (sum ref, sum dist, sum ref^2, sum dist^2) of the luma of the
    4:2:0 pairs in one launch; algorithmic bytes 2 w h per pair."""
    import torch

    import integer_image_filter_gb300 as iif
    import synth

    n = args.pairs
    batch = synth.yuv420_pairs(4, n, args.w, args.h, max_shift=2, dist_sigma=3.0)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    ref = torch.from_numpy(batch.ref_y).to(dev)
    dist = torch.from_numpy(batch.dist_y).to(dev)
    out = torch.zeros((n, 4), dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        iif.moment_sums_batch(ref, dist, 8, out, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / args.steps
    peak, peak_kind = peaks()
    alg = 2 * args.w * args.h * n
    print(json.dumps({"metric": "pairs/s (luma moment sums)", "value": n / (ms * 1e-3),
                      "unit": "frames/s", "ms_per_step": ms, "steps": args.steps,
                      "config": {"workload": "moment_%dx%d_u8_pairs" % (args.w, args.h),
                                 "pairs_per_step": n},
                      "roofline": {"bound": "hbm", "achieved": alg / (ms * 1e-3) / 1e9,
                                   "peak": peak, "unit": "GB/s",
                                   "frac": alg / (ms * 1e-3) / 1e9 / peak,
                                   "peak_kind": peak_kind}}), flush=True)
    return 0


def run_latency_workload(args):
    """Per-frame submit latency (one launch and one 8-byte readback per frame)
    on the small configurations."""
    import numpy as np
    import torch

    import integer_image_filter_gb300 as iif
    import synth

    c = synth.CONFIGS[args.workload]
    w, h, bpc = c["w"], c["h"], c["bpc"]
    frames = synth.make(args.workload)
    n = frames.shape[0]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    d = torch.from_numpy(frames).to(dev)
    ctx = iif.MotionContext(w, h, bpc)
    for _ in range(3):
        ctx.reset()
        for i in range(n):
            ctx.submit(d[i])
    t0 = time.perf_counter()
    for _ in range(args.steps):
        ctx.reset()
        for i in range(n):
            ctx.submit(d[i])
    us = (time.perf_counter() - t0) / (args.steps * n) * 1e6
    ctx.close()
    print(json.dumps({"metric": "us per submitted frame (launch + 8-byte readback)", "value": us,
                      "unit": "us/frame", "higher_is_better": False, "steps": args.steps,
                      "config": {"workload": args.workload, "w": w, "h": h, "bpc": bpc,
                                 "frames_per_step": n}}), flush=True)
    return 0


def run_host_link(args):
    """Host link ceiling by NUMA node: 1 GiB pinned buffers allocated under a
    memory policy bound to each host node (and the default policy), host->device
    and device->host copy rates (best of 5 and 3, CUDA events); one JSON line
    with the GPU's node and where the pinned pages landed."""
    import ctypes
    import glob

    import torch
    libc = ctypes.CDLL(None, use_errno=True)
    nr_set_mempolicy = 237 if os.uname().machine == "aarch64" else 238
    nodes = sorted(int(p.rsplit("node", 1)[1]) for p in glob.glob("/sys/devices/system/node/node[0-9]*"))

    def bind(node):
        if node is None:
            return libc.syscall(nr_set_mempolicy, 0, None, ctypes.c_ulong(0))
        mask = ctypes.c_ulong(1 << node)
        return libc.syscall(nr_set_mempolicy, 2, ctypes.byref(mask), ctypes.c_ulong(64))

    torch.cuda.set_device(0)
    s = torch.cuda.current_stream()
    dev = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")

    def rate(copy, reps):
        best = 0.0
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            copy()
            e1.record(s)
            torch.cuda.synchronize()
            best = max(best, (1 << 30) / (e0.elapsed_time(e1) * 1e-3) / 1e9)
        return best

    res = {}
    for node in [None] + nodes:
        if bind(node) != 0:
            res["default" if node is None else str(node)] = {"error": "set_mempolicy refused"}
            continue
        try:
            h = torch.empty(1 << 30, dtype=torch.uint8).pin_memory()
            h.fill_(1)
        finally:
            bind(None)
        dev.copy_(h, non_blocking=True)
        torch.cuda.synchronize()
        res["default" if node is None else str(node)] = {
            "h2d_gbs": rate(lambda: dev.copy_(h, non_blocking=True), 5),
            "d2h_gbs": rate(lambda: h.copy_(dev, non_blocking=True), 3),
            "placement": numa_placement(h)}
        del h
    print(json.dumps({"metric": "pinned host link GB/s by NUMA node", "by_policy": res,
                      "config": {"workload": "host_link", "bytes": 1 << 30}}), flush=True)
    return 0


def hbm_stream_ceilings() -> dict | None:
    """HBM read-only, write-only and copy stream rates measured now on this
    device (libpipe_rates_gb300.so, hbm_stream_gbs), or None when the probe
    library cannot be built or a CUDA call failed."""
    import ctypes

    from integer_image_filter_gb300 import _build
    try:
        lib = ctypes.CDLL(_build.build_pipe_rates())
    except Exception:
        return None
    out = {}
    for kind, name in ((0, "read_only_gbs"), (1, "write_only_gbs"), (2, "copy_gbs")):
        g = ctypes.c_double()
        if lib.hbm_stream_gbs(kind, ctypes.byref(g)) != 0:
            return None
        out[name] = round(g.value, 1)
    out["basis"] = ("hbm_stream_gbs (libpipe_rates_gb300.so): 16-byte streaming accesses over 4 GiB "
                    "read / 4 GiB written / 2 GiB copied (read + write counted), best of 5 launches")
    return out


def read_only_ceiling(streams: dict | None, secondary: dict | None, achieved: float) -> dict | None:
    """The stream rates of this run with the fused launch's fraction of the
    fastest read-only stream measured in it: the probe's, or the stand-alone
    SSE launch's (a read-only stream of the same pairs) when that was faster."""
    if not streams:
        return None
    best, basis = streams["read_only_gbs"], "hbm_stream_gbs read probe"
    sse = (secondary or {}).get("sse_yuv420_3840x2160_u8_pairs") or {}
    if sse.get("gb_per_s", 0) > best:
        best, basis = sse["gb_per_s"], "the stand-alone SSE launch of this run (read-only, same pairs)"
    return dict(streams, read_only_best_gbs=round(best, 1), read_only_best_basis=basis,
                frac_of_read_only=achieved / best)


def run_pipe_rates(args):
    """The instruction-throughput microbenchmark (libpipe_rates_gb300.so):
    lane-operations per SM clock per SM of each instruction class the motion
    kernels issue, measured on this device; one JSON line."""
    import ctypes

    import torch

    from integer_image_filter_gb300 import _build
    lib = ctypes.CDLL(_build.build_pipe_rates())
    lib.pipe_rates_name.restype = ctypes.c_char_p
    n = lib.pipe_rates_count()
    out = (ctypes.c_double * n)()
    torch.cuda.set_device(0)
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.3)
    rc = lib.pipe_rates_measure(out)
    time.sleep(0.3)
    clocks.stop()
    if rc != 0:
        raise RuntimeError("pipe_rates_measure failed")
    rates = {lib.pipe_rates_name(i).decode(): round(out[i], 2) for i in range(n)}
    streams = hbm_stream_ceilings()
    print(json.dumps({"metric": "lane-operations per SM clock per SM (shared loads: bytes)",
                      "rates": rates, "sms": torch.cuda.get_device_properties(0).multi_processor_count,
                      "hbm_streams": streams,
                      "clocks": clocks.summary(),
                      "config": {"workload": "pipe_rates", "threads_per_sm": 1024,
                                 "chains_per_thread": 8}}), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--pairs", type=int, default=50)
    ap.add_argument("--w", type=int, default=3840)
    ap.add_argument("--h", type=int, default=2160)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the other configurations' measurements in the default line")
    ap.add_argument("--sustain-seconds", type=float, default=1.0,
                    help="length of the back-to-back launch loop behind roofline.kernel_ms")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="the headline 4:2:0 workload (default) or one of the motion-only "
                         "configurations: seq_3840x2160_u10, seq_1920x1080_u8_cuts, "
                         "seq_576x324_u8, pair_64x48_u8; or sse_yuv420_3840x2160_u8_pairs, "
                         "moment_3840x2160_u8_pairs (stand-alone SSE / luma moment sums); "
                         "pipe_rates (instruction throughput per SM), host_link (pinned copy "
                         "rates by NUMA node)")
    ap.add_argument("--batch", type=int, default=0, help="frames per launch (sequence workloads)")
    ap.add_argument("--sweep", action="store_true", help="sweep batch sizes 1..32")
    ap.add_argument("--graph", action="store_true",
                    help="sequence workloads: time replays of one step captured as a CUDA graph")
    ap.add_argument("--trim", type=int, default=0,
                    help="sequence workloads: drop this many columns and pack the rows tightly")
    ap.add_argument("--generic", action="store_true",
                    help="sequence workloads: force the generic (non-TMA) kernel")
    ap.add_argument("--v2", action="store_true",
                    help="sequence workloads: motion_v2 (blur of prev - cur) instead of motion")
    args = ap.parse_args(argv)
    if args.workload == "pipe_rates" and args.impl == "ours":
        return run_pipe_rates(args)
    if args.workload == "host_link" and args.impl == "ours":
        return run_host_link(args)
    if args.workload == "sse_yuv420_3840x2160_u8_pairs" and args.impl == "ours":
        return run_sse_workload(args)
    if args.workload == "moment_3840x2160_u8_pairs" and args.impl == "ours":
        return run_moment_workload(args)
    if args.workload in ("seq_3840x2160_u10", "seq_1920x1080_u8_cuts") and args.impl == "ours":
        return run_sequence_workload(args)
    if args.workload in ("seq_576x324_u8", "pair_64x48_u8") and args.impl == "ours":
        return run_latency_workload(args) if not args.batch else run_sequence_workload(args)
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
