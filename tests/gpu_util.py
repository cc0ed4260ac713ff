"""Helpers for the GPU parity tests: device upload of numpy planes and the
oracle run in threads (its C calls release the GIL)."""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np


def to_dev(a: np.ndarray):
    import torch
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


def dev_zeros(shape):
    import torch
    return torch.zeros(shape, dtype=torch.int64, device="cuda")


def to_u64(t) -> np.ndarray:
    return t.cpu().numpy().astype(np.uint64)


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def oracle_sad(o, frames: np.ndarray, bpc: int) -> np.ndarray:
    """Oracle SAD sequence, split into overlapping chunks run in parallel (chunk
    k covers frames [s-1, e) so that its first SAD is against frame s-1)."""
    n = frames.shape[0]
    if n <= 8:
        return o.motion_sad_sequence(frames, bpc)
    k = _threads()
    bounds = np.linspace(0, n, k + 1).astype(int)

    def run(i):
        s, e = int(bounds[i]), int(bounds[i + 1])
        if e <= s:
            return np.zeros(0, np.uint64)
        lo = max(s - 1, 0)
        r = o.motion_sad_sequence(frames[lo:e], bpc)
        return r if s == 0 else r[1:]

    with ThreadPoolExecutor(k) as ex:
        parts = list(ex.map(run, range(k)))
    return np.concatenate(parts).astype(np.uint64)


def oracle_sse420(o, b) -> np.ndarray:
    def run(i):
        return [o.sse(b.ref_y[i], b.dist_y[i], b.bpc), o.sse(b.ref_u[i], b.dist_u[i], b.bpc),
                o.sse(b.ref_v[i], b.dist_v[i], b.bpc)]
    with ThreadPoolExecutor(_threads()) as ex:
        rows = list(ex.map(run, range(b.n)))
    return np.array(rows, dtype=np.uint64).reshape(b.n, 3)
