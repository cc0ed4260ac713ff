"""Parity cases for the bounds-checked library (libmotion_gb300_checked.so,
built with MG_BOUNDS_CHECK=1), run as a child process of
tests/test_gpu_bounds_checked.py so that the binding loads that library.

Every shared- and global-memory access of the motion kernels is checked there
against its buffer; a failed check skips the access and sets bit 1 of the
context's device error word.  Each case below runs both kernel paths (TMA and
generic) on frames of odd, ragged and tile-straddling sizes, contiguous and
with padded rows, at 8, 10 and 16 bits, over two calls (the second continues
the sequence), and records a failure when a result differs from the oracle or
the error word is not 0; the motion cases also run with the tile height
forced to 128 x 32 (the small frames here otherwise take 128 x 16 tiles).
The allocation-free entry point runs the same way
(start, then continue) with its own error word read after each case.  Prints
one JSON line: {"cases": N, "failures": [...]}.
"""
from __future__ import annotations

import json
import sys

import numpy as np

SIZES = [(3, 3), (5, 7), (17, 9), (67, 35), (129, 33), (130, 34), (200, 100), (257, 70),
         (256, 70), (129, 100)]   # full right-edge tiles with mirrored halo reads
FUSED_SIZES = [(4, 4), (67, 35), (130, 70), (258, 66)]
# the allocation-free entry point: packed odd rows take the generic kernel,
# 16-byte rows the TMA kernel
NOALLOC_SIZES = [(67, 35), (256, 70), (130, 34)]
# a launch shape whose tail is split (900 tiles of 128 x 32 over 608 resident
# blocks: the last 292 tiles run in chunks of 4 frames), 8 frames per call
SPLIT_SIZES = [(2560, 1440)]


def _dev(a: np.ndarray, pad: bool):
    import torch
    n, h, w = a.shape
    s = a.itemsize
    wp = ((w * s + 15) // 16 * 16 + (16 if pad else 0)) // s if pad else w
    big = np.zeros((n, h, wp), dtype=a.dtype)
    big[:, :, :w] = a
    t = torch.from_numpy(big.view(np.int16) if a.dtype == np.uint16 else big).to("cuda")
    return t[:, :, :w]


def _frames(rng, n, h, w, bpc):
    dt = np.uint8 if bpc == 8 else np.uint16
    return rng.integers(0, 1 << bpc, size=(n, h, w)).astype(dt)


def main() -> int:
    import torch

    import integer_image_filter_gb300 as iif
    from integer_image_filter_gb300 import _build
    iif.load_library(_build.build(checked=True))
    import oracle
    o = oracle.Oracle()
    rng = np.random.default_rng(20261202)
    cases, failures = 0, []

    def u64(t):
        return t.cpu().numpy().astype(np.uint64)

    # AUTO runs these small frames in 128 x 16 tiles (they fit in one wave of
    # 128 x 32 tiles); TMA_32 runs the motion cases in 128 x 32 tiles as well
    for path in (iif.MOTION_PATH_AUTO, iif.MOTION_PATH_GENERIC, iif.MOTION_PATH_TMA_32):
        for (w, h) in SIZES:
            for bpc in (8, 10, 16):
                for pad in (False, True):
                    fr = _frames(rng, 6, h, w, bpc)
                    d = _dev(fr, pad)
                    want = o.motion_sad_sequence(fr, bpc).astype(np.uint64)
                    want_v2 = o.motion_v2_sequence(fr, bpc).astype(np.uint64)
                    for v2 in (False, True):
                        out = torch.zeros(6, dtype=torch.int64, device="cuda")
                        with iif.MotionContext(w, h, bpc) as ctx:
                            ctx.set_kernel_path(path)
                            sub = ctx.submit_batch_v2 if v2 else ctx.submit_batch
                            sub(d[:4], out[:4])
                            sub(d[4:], out[4:])
                            torch.cuda.synchronize()
                            err = ctx.device_error()
                        got = u64(out)
                        cases += 1
                        exp = want_v2 if v2 else want
                        if err != 0 or not np.array_equal(got, exp):
                            failures.append({"kind": "motion_v2" if v2 else "motion", "w": w, "h": h,
                                             "bpc": bpc, "pad": pad, "path": path, "err": err,
                                             "got": got.tolist(), "want": exp.tolist()})
        for (w, h) in (FUSED_SIZES if path != iif.MOTION_PATH_TMA_32 else ()):
            for bpc in (8, 10):
                for pad in (False, True):
                    n = 5
                    cw, ch = (w + 1) // 2, (h + 1) // 2
                    ry, dy = _frames(rng, n, h, w, bpc), _frames(rng, n, h, w, bpc)
                    ru, du, rv, dv = (_frames(rng, n, ch, cw, bpc) for _ in range(4))
                    want_sad = o.motion_sad_sequence(ry, bpc).astype(np.uint64)
                    want_sse = np.array([[o.sse(ry[i], dy[i], bpc), o.sse(ru[i], du[i], bpc),
                                          o.sse(rv[i], dv[i], bpc)] for i in range(n)], dtype=np.uint64)
                    sad = torch.zeros(n, dtype=torch.int64, device="cuda")
                    sse = torch.zeros((n, 3), dtype=torch.int64, device="cuda")
                    with iif.MotionContext(w, h, bpc) as ctx:
                        ctx.set_kernel_path(path)
                        ctx.yuv420_batch(_dev(ry, pad), _dev(ru, pad), _dev(rv, pad), _dev(dy, pad),
                                         _dev(du, pad), _dev(dv, pad), sad, sse)
                        torch.cuda.synchronize()
                        err = ctx.device_error()
                    cases += 1
                    if err != 0 or not np.array_equal(u64(sad), want_sad) or not np.array_equal(u64(sse), want_sse):
                        failures.append({"kind": "fused", "w": w, "h": h, "bpc": bpc, "pad": pad, "path": path,
                                         "err": err})
    for (w, h) in NOALLOC_SIZES:
        for bpc in (8, 10):
            for pad in (False, True):
                fr = _frames(rng, 6, h, w, bpc)
                d = _dev(fr, pad)
                want = o.motion_sad_sequence(fr, bpc).astype(np.uint64)
                out = torch.zeros(6, dtype=torch.int64, device="cuda")
                iif.motion_submit_batch_noalloc(d[:4], out[:4], bpc=bpc, continue_sequence=False)
                iif.motion_submit_batch_noalloc(d[4:], out[4:], bpc=bpc, continue_sequence=True)
                torch.cuda.synchronize()
                err = iif.motion_noalloc_device_error()
                cases += 1
                if err != 0 or not np.array_equal(u64(out), want):
                    failures.append({"kind": "noalloc", "w": w, "h": h, "bpc": bpc, "pad": pad,
                                     "err": err, "got": u64(out).tolist(), "want": want.tolist()})
    for (w, h) in SPLIT_SIZES:
        for bpc in (8, 10):
            fr = _frames(rng, 16, h, w, bpc)
            d = _dev(fr, False)
            want = o.motion_sad_sequence(fr, bpc).astype(np.uint64)
            out = torch.zeros(16, dtype=torch.int64, device="cuda")
            with iif.MotionContext(w, h, bpc) as ctx:
                ctx.submit_batch(d[:8], out[:8])
                ctx.submit_batch(d[8:], out[8:])
                torch.cuda.synchronize()
                err = ctx.device_error()
            cases += 1
            if err != 0 or not np.array_equal(u64(out), want):
                failures.append({"kind": "split", "w": w, "h": h, "bpc": bpc, "err": err})
    print(json.dumps({"cases": cases, "failures": failures[:20], "n_failures": len(failures)}))
    return 0


if __name__ == "__main__":
    sys.exit(main())
