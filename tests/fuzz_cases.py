"""Seeded fuzz cases for the C ABI (used by tests/test_gpu_fuzz.py).

Case i draws, from one seeded generator, a kind (motion, motion_v2, fused
4:2:0, stand-alone 4:2:0 SSE, single-plane SSE, moment sums; after them the
host-buffer pipelines and the single-frame call), a frame size
from 3x3 up, a bit depth from 8 to 16, padded rows, a base offset, the cut
points that split the frames over consecutive calls and the kernel path; it
places uniform samples in that layout, calls the library through its raw
entry points and compares every result with the oracle.

Run as a child with the bounds-checked library (the kinds whose kernels are
instrumented: motion, motion_v2, fused 4:2:0), printing one JSON line
{"cases": N, "failures": [...]}:

    python -m tests.fuzz_cases checked
"""
from __future__ import annotations

import json
import sys

import numpy as np

import synth

KINDS = ("motion", "motion_v2", "yuv420", "sse420", "sse", "moments")
CHECKED_KINDS = ("motion", "motion_v2", "yuv420")
N_CASES = 120
# host-buffer pipelines and the single-frame call, after the device cases
HOST_KINDS = ("yuv420_host", "motion_host", "single")
N_HOST_CASES = 36
N_ALL = N_CASES + N_HOST_CASES


def check(cond: bool, msg) -> None:
    if not cond:
        raise AssertionError(msg)


def draw(i: int) -> dict:
    """Case i: every choice from one seeded generator."""
    rng = np.random.default_rng(9000 + i)
    kind = KINDS[i % len(KINDS)] if i < N_CASES else HOST_KINDS[(i - N_CASES) % len(HOST_KINDS)]
    bpc = int(rng.choice([8, 8, 9, 10, 12, 14, 16]))
    s = 1 if bpc == 8 else 2
    w = int(rng.integers(3, 300))
    h = int(rng.integers(3, 120))
    if rng.random() < 0.15:                       # now and then a frame near the 3x3 minimum
        w, h = int(rng.integers(3, 8)), int(rng.integers(3, 8))
    n = int(rng.integers(1, 11))
    pad = int(rng.integers(0, 40)) * s if rng.random() < 0.6 else 0     # bytes after each row
    off = int(rng.integers(0, 24)) * s if rng.random() < 0.5 else 0     # bytes before the first sample
    cuts = sorted(set(int(c) for c in rng.integers(1, n, size=int(rng.integers(0, 3))))) if n > 1 else []
    generic = bool(rng.random() < 0.3)
    d = dict(kind=kind, bpc=bpc, s=s, w=w, h=h, n=n, pad=pad, off=off, cuts=cuts,
             generic=generic, seed=int(rng.integers(0, 2**31 - 1)))
    # the TMA kernel's tile height for the motion kinds: these small launches
    # choose 128 x 16 tiles; every other case forces 128 x 32 (taken from the
    # case number, not the generator, so that the draws above stay as they were)
    d["rows32"] = (i % 4) >= 2
    if i >= N_CASES:                              # drawn last: the device cases stay as they were
        d["chunk"] = int(rng.integers(0, 4))      # frames (pairs) per host chunk, 0 = the default
    return d


def place(frames: np.ndarray, pad: int, off: int):
    """A device byte buffer holding `frames` (n, h, w) with rows w*s + pad bytes
    apart and the first sample off bytes in; returns (buffer, address, pitch,
    frame stride)."""
    import torch
    n, h, w = frames.shape
    s = frames.itemsize
    pitch = w * s + pad
    host = np.zeros((n, h, pitch), np.uint8)
    host[:, :, :w * s] = frames.view(np.uint8).reshape(n, h, w * s)
    buf = torch.zeros(off + host.size + 64, dtype=torch.uint8, device="cuda")
    buf[off:off + host.size] = torch.from_numpy(host.reshape(-1)).to("cuda")
    return buf, buf.data_ptr() + off, pitch, h * pitch


def place_host(frames: np.ndarray, pad: int, off: int):
    """As place(), in a host (pageable) byte buffer."""
    n, h, w = frames.shape
    s = frames.itemsize
    pitch = w * s + pad
    buf = np.zeros(off + n * h * pitch + 64, np.uint8)
    view = buf[off:off + n * h * pitch].reshape(n, h, pitch)
    view[:, :, :w * s] = frames.view(np.uint8).reshape(n, h, w * s)
    return buf, buf.ctypes.data + off, pitch, h * pitch


def spans(n: int, cuts):
    edges = [0] + list(cuts) + [n]
    return [(a, b) for a, b in zip(edges[:-1], edges[1:]) if b > a]


def sse420(o, b) -> np.ndarray:
    return np.array([[o.sse(b.ref_y[k], b.dist_y[k], b.bpc), o.sse(b.ref_u[k], b.dist_u[k], b.bpc),
                      o.sse(b.ref_v[k], b.dist_v[k], b.bpc)] for k in range(b.n)], dtype=np.uint64)


def run_case(iif, o, i: int) -> None:
    """Run case i; raises AssertionError naming the case on any difference."""
    import torch
    c = draw(i)
    kind, bpc, w, h, n = c["kind"], c["bpc"], c["w"], c["h"], c["n"]
    lib = iif.load_library()
    what = f"case {i}: {c}"

    def ok(rc):
        check(rc == 0, (what, iif.motion_strerror(rc)))

    if kind in HOST_KINDS:
        run_host_case(iif, o, c, what)
        return
    if kind in ("motion", "motion_v2"):
        fr = synth.uniform_frames(c["seed"], n, w, h, bpc)
        buf, addr, pitch, stride = place(fr, c["pad"], c["off"])
        out = torch.zeros(n, dtype=torch.int64, device="cuda")
        fn = lib.motion_v2_submit_batch if kind == "motion_v2" else lib.motion_submit_batch
        with iif.MotionContext(w, h, bpc) as ctx:
            if c["generic"]:
                ctx.set_kernel_path(iif.MOTION_PATH_GENERIC)
            elif c["rows32"]:
                ctx.set_kernel_path(iif.MOTION_PATH_TMA_32)
            for a, b in spans(n, c["cuts"]):
                ok(fn(ctx.handle, addr + a * stride, b - a, stride, pitch, None, out.data_ptr() + 8 * a))
            torch.cuda.synchronize()
            check(ctx.device_error() == 0, ("device error", what))
        want = (o.motion_v2_sequence if kind == "motion_v2" else o.motion_sad_sequence)(fr, bpc)
        check(out.cpu().numpy().astype(np.uint64).tolist() == [int(x) for x in want], what)
        return
    if kind == "sse":
        ref = synth.uniform_frames(c["seed"], 1, w, h, bpc)
        dist = synth.uniform_frames(c["seed"] + 1, 1, w, h, bpc)
        rb, ra, rp, _ = place(ref, c["pad"], c["off"])
        db, da, dp, _ = place(dist, c["s"] * (i % 5), 0)        # a second pitch for dist
        out = torch.zeros(1, dtype=torch.int64, device="cuda")
        ok(lib.psnr_sse(ra, da, rp, dp, w, h, bpc, None, out.data_ptr()))
        torch.cuda.synchronize()
        check(int(out.cpu().numpy().astype(np.uint64)[0]) == o.sse(ref[0], dist[0], bpc), what)
        return
    b = synth.uniform_yuv420(c["seed"], n, w, h, bpc)
    if kind == "moments":
        rb, ra, pitch, stride = place(b.ref_y, c["pad"], c["off"])
        db, da, _, _ = place(b.dist_y, c["pad"], c["off"])
        out = torch.zeros((n, 4), dtype=torch.int64, device="cuda")
        ok(lib.moment_sums_batch(w, h, bpc, n, ra, da, pitch, stride, None, out.data_ptr()))
        torch.cuda.synchronize()
        want = [[int(v) for v in o.moment_sums(b.ref_y[k], b.dist_y[k], bpc)] for k in range(n)]
        check(out.cpu().numpy().astype(np.uint64).tolist() == want, what)
        return
    keep, views = [], []
    for p in b.planes():                          # luma planes share one layout, chroma another
        pad = c["pad"] if p.shape[2] == w else c["s"] * (c["pad"] // (2 * c["s"]))
        buf, addr, pitch, stride = place(p, pad, c["off"])
        keep.append(buf)
        views.append((addr, pitch, stride))
    (py, sy), (puv, suv) = views[0][1:], views[1][1:]
    sse = torch.zeros((n, 3), dtype=torch.int64, device="cuda")
    if kind == "sse420":
        ok(lib.psnr_sse_yuv420_batch(w, h, bpc, n, *[v[0] for v in views], py, puv, sy, suv, None,
                                     sse.data_ptr()))
        torch.cuda.synchronize()
    else:
        sad = torch.zeros(n, dtype=torch.int64, device="cuda")
        with iif.MotionContext(w, h, bpc) as ctx:
            if c["generic"]:
                ctx.set_kernel_path(iif.MOTION_PATH_GENERIC)
            for a, e in spans(n, c["cuts"]):
                ptrs = [v[0] + a * (sy if k in (0, 3) else suv) for k, v in enumerate(views)]
                ok(lib.motion_psnr_yuv420_batch(ctx.handle, e - a, *ptrs, py, puv, sy, suv, None,
                                                sad.data_ptr() + 8 * a, sse.data_ptr() + 24 * a))
            torch.cuda.synchronize()
            check(ctx.device_error() == 0, ("device error", what))
        check(sad.cpu().numpy().astype(np.uint64).tolist() ==
              [int(x) for x in o.motion_sad_sequence(b.ref_y, bpc)], what)
    check(np.array_equal(sse.cpu().numpy().astype(np.uint64), sse420(o, b)), what)


def run_host_case(iif, o, c: dict, what: str) -> None:
    """Host-buffer pipelines (host pictures in, host results out, in chunks of
    c["chunk"]) and the single-frame call mixed with batches on one sequence."""
    import ctypes

    import torch
    kind, bpc, w, h, n = c["kind"], c["bpc"], c["w"], c["h"], c["n"]
    lib = iif.load_library()

    def ok(rc):
        check(rc == 0, (what, iif.motion_strerror(rc)))

    if kind == "motion_host":
        fr = synth.uniform_frames(c["seed"], n, w, h, bpc)
        buf, addr, pitch, stride = place_host(fr, c["pad"], c["off"])
        out = np.zeros(n, np.uint64)
        with iif.MotionContext(w, h, bpc) as ctx:
            for a, b in spans(n, c["cuts"]):
                ok(lib.motion_submit_batch_host(ctx.handle, addr + a * stride, b - a, stride, pitch,
                                                c["chunk"], out.ctypes.data + 8 * a))
            check(ctx.device_error() == 0, ("device error", what))
        check(out.tolist() == [int(x) for x in o.motion_sad_sequence(fr, bpc)], what)
        return
    if kind == "single":
        fr = synth.uniform_frames(c["seed"], n, w, h, bpc)
        buf, addr, pitch, stride = place(fr, c["pad"], c["off"])
        sad = np.zeros(n, np.uint64)
        score = np.zeros(n, np.float64)
        d_out = torch.zeros(n, dtype=torch.int64, device="cuda")
        with iif.MotionContext(w, h, bpc) as ctx:
            if c["generic"]:
                ctx.set_kernel_path(iif.MOTION_PATH_GENERIC)
            for j, (a, b) in enumerate(spans(n, c["cuts"])):
                if j % 2 == 0:                    # frame by frame, with the 8-byte readback
                    for k in range(a, b):
                        v, sc = ctypes.c_uint64(), ctypes.c_double()
                        ok(lib.motion_submit(ctx.handle, addr + k * stride, pitch, None,
                                             ctypes.byref(v), ctypes.byref(sc)))
                        sad[k], score[k] = v.value, sc.value
                else:                             # then a batch continuing the sequence
                    ok(lib.motion_submit_batch(ctx.handle, addr + a * stride, b - a, stride, pitch, None,
                                               d_out.data_ptr() + 8 * a))
                    torch.cuda.synchronize()
                    sad[a:b] = d_out[a:b].cpu().numpy().astype(np.uint64)
                    score[a:b] = (sad[a:b].astype(np.float64) / 256.0) / float(w * h)
            check(ctx.device_error() == 0, ("device error", what))
        want = o.motion_sad_sequence(fr, bpc)
        check(sad.tolist() == [int(x) for x in want], what)
        check(score.tolist() == o.scores(want, w, h)[0].tolist(), ("score", what))
        return
    b = synth.uniform_yuv420(c["seed"], n, w, h, bpc)
    keep, views = [], []
    for p in b.planes():
        pad = c["pad"] if p.shape[2] == w else c["s"] * (c["pad"] // (2 * c["s"]))
        buf, addr, pitch, stride = place_host(p, pad, c["off"])
        keep.append(buf)
        views.append((addr, pitch, stride))
    (py, sy), (puv, suv) = views[0][1:], views[1][1:]
    sad = np.zeros(n, np.uint64)
    sse = np.zeros((n, 3), np.uint64)
    with iif.MotionContext(w, h, bpc) as ctx:
        if c["generic"]:
            ctx.set_kernel_path(iif.MOTION_PATH_GENERIC)
        if c["chunk"]:
            ok(lib.motion_reserve_host_staging(ctx.handle, c["chunk"], sy, suv))
        for a, e in spans(n, c["cuts"]):
            ptrs = [v[0] + a * (sy if k in (0, 3) else suv) for k, v in enumerate(views)]
            ok(lib.motion_psnr_yuv420_batch_host(ctx.handle, e - a, *ptrs, py, puv, sy, suv,
                                                 sad.ctypes.data + 8 * a, sse.ctypes.data + 24 * a))
        check(ctx.device_error() == 0, ("device error", what))
    check(sad.tolist() == [int(x) for x in o.motion_sad_sequence(b.ref_y, bpc)], what)
    check(np.array_equal(sse, sse420(o, b)), what)


def main(mode: str) -> int:
    import integer_image_filter_gb300 as iif
    from integer_image_filter_gb300 import _build
    if mode != "checked":
        raise SystemExit("usage: python -m tests.fuzz_cases checked")
    iif.load_library(_build.build(checked=True))
    import oracle
    o = oracle.Oracle()
    cases, failures = 0, []
    for i in range(N_CASES):
        if draw(i)["kind"] not in CHECKED_KINDS:
            continue
        cases += 1
        try:
            run_case(iif, o, i)
        except AssertionError as e:
            failures.append(str(e)[:400])
    print(json.dumps({"cases": cases, "n_failures": len(failures), "failures": failures}))
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv[1] if len(sys.argv) > 1 else ""))
