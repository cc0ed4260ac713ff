"""Child process of tests/test_gpu_threads.py (GPU side only).

Several host threads, each with its own motion context and CUDA stream, are
released together by a barrier, so that their first calls into the library
overlap -- and with them the library's one-time set-up (the tensor-map encoder
lookup, the per-device launch attributes and the resident-CTA count).  The
ctypes calls release the GIL, so the library really is entered concurrently.
Every result goes to the JSON file named on the command line; the parent
compares it with the oracle.

    python -m tests.threaded_contexts OUT.json
"""
from __future__ import annotations

import json
import sys
import threading

import numpy as np

import synth

# kind, seed, frames (pairs), w, h, bpc
JOBS = [
    ("motion", 201, 9, 640, 160, 8),
    ("motion", 202, 9, 213, 70, 10),       # 426-byte rows: the copy kernel, then the TMA kernel
    ("motion_v2", 203, 9, 384, 96, 8),
    ("motion_v2", 204, 9, 130, 34, 12),
    ("yuv420", 205, 9, 256, 96, 8),
    ("yuv420", 206, 9, 130, 66, 10),
    ("yuv420_host", 207, 5, 200, 64, 8),   # host buffers: the two-stream pipeline
    ("motion_host", 208, 7, 96, 40, 10),
    ("moments", 209, 6, 576, 324, 8),
    ("motion", 210, 6, 1920, 1080, 8),
]
BATCH = 3


def inputs(kind: str, seed: int, n: int, w: int, h: int, bpc: int):
    """The job's seeded inputs (the parent rebuilds the same ones)."""
    if kind in ("yuv420", "yuv420_host", "moments"):
        return synth.uniform_yuv420(seed, n, w, h, bpc)
    return synth.uniform_frames(seed, n, w, h, bpc)


def _dev(a: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a.view(np.int16) if a.dtype == np.uint16 else a)).cuda()


def run_job(iif, job, barrier: threading.Barrier) -> dict:
    import torch
    kind, seed, n, w, h, bpc = job
    data = inputs(*job)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        if kind in ("yuv420", "moments"):
            planes = [_dev(p) for p in data.planes()]
        elif kind in ("motion", "motion_v2"):
            d = _dev(data)
        sad = torch.zeros(n, dtype=torch.int64, device="cuda")
        sse = torch.zeros((n, 3), dtype=torch.int64, device="cuda")
        sums = torch.zeros((n, 4), dtype=torch.int64, device="cuda")
    s.synchronize()
    barrier.wait()
    out: dict = {}
    if kind == "moments":
        iif.moment_sums_batch(planes[0], planes[3], bpc, sums, stream=s)
        s.synchronize()
        return {"sums": sums.cpu().numpy().astype(np.uint64).tolist()}
    with iif.MotionContext(w, h, bpc) as ctx:
        if kind == "yuv420_host":
            got_sad, got_sse = ctx.yuv420_batch_host(*data.planes())
            out = {"sad": np.asarray(got_sad, np.uint64).tolist(), "sse": np.asarray(got_sse, np.uint64).tolist()}
        elif kind == "motion_host":
            out = {"sad": np.asarray(ctx.submit_batch_host(data), np.uint64).tolist()}
        else:
            for b0 in range(0, n, BATCH):
                e = min(b0 + BATCH, n)
                if kind == "yuv420":
                    ctx.yuv420_batch(*[p[b0:e] for p in planes], sad[b0:e], sse[b0:e], stream=s)
                elif kind == "motion_v2":
                    ctx.submit_batch_v2(d[b0:e], sad[b0:e], stream=s)
                else:
                    ctx.submit_batch(d[b0:e], sad[b0:e], stream=s)
            s.synchronize()
            out = {"sad": sad.cpu().numpy().astype(np.uint64).tolist()}
            if kind == "yuv420":
                out["sse"] = sse.cpu().numpy().astype(np.uint64).tolist()
        out["device_error"] = ctx.device_error()
    return out


def main(path: str) -> None:
    import torch
    import integer_image_filter_gb300 as iif
    torch.cuda.init()
    barrier = threading.Barrier(len(JOBS))
    results: list = [None] * len(JOBS)
    errors: list = []

    def worker(i: int) -> None:
        try:
            results[i] = run_job(iif, JOBS[i], barrier)
        except BaseException as e:   # reported by the parent
            errors.append(f"{JOBS[i]}: {type(e).__name__}: {e}")
            barrier.abort()

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(JOBS))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    with open(path, "w") as f:
        json.dump({"results": results, "errors": errors}, f)


if __name__ == "__main__":
    main(sys.argv[1])
