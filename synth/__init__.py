"""Seeded synthetic video inputs shared by the tests, the smoke check and the
benchmark.

This module holds no part of the method's arithmetic (no blur, no SAD, no
squared error): it only draws frames.  Both the CUDA path and the CPU oracle
are fed the same arrays made here.

Recipes (each one fixed by its seed):

* ``uniform_frames`` / ``uniform_yuv420`` -- samples i.i.d. uniform over
  [0, 2^bpc - 1] (integer draws only: identical on every platform, which the
  stored expected values in tests/golden rely on).
* ``smooth_sequence`` -- a smooth luma field, 128 + sum of 8 random 2-D
  sinusoids (amplitudes a_k ~ U(0, 100/8), so the sum stays within +-100;
  spatial frequencies of 0.5 to 8 cycles per frame in each axis with random
  sign; phases ~ U(0, 2*pi)), plus per-frame Gaussian noise, rounded half to
  even and clipped to 0..255.  Frame t shows the field translated by the
  cumulative sum of per-frame integer steps (dx, dy) ~ U{-s..s}; a fraction of
  frames is replaced by a fresh field (scene cuts), from which the translation
  continues.  For bpc > 8 the noisy float field is scaled by (2^bpc-1)/255,
  rounded and clipped to 0..2^bpc-1.
* ``yuv420_pairs`` -- 4:2:0 reference pictures (luma from ``smooth_sequence``;
  each chroma plane its own smooth field at half size, translated by half the
  luma offset), and distorted pictures = reference + N(0, sigma^2) per sample,
  rounded and clipped.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

__all__ = ["uniform_frames", "smooth_sequence", "yuv420_pairs", "Yuv420Batch",
           "translation_walk", "CONFIGS", "chroma_dims"]


def chroma_dims(w: int, h: int) -> tuple[int, int]:
    """4:2:0 chroma plane size: ceil(w/2) x ceil(h/2)."""
    return (w + 1) // 2, (h + 1) // 2


def _dtype(bpc: int):
    if not 8 <= bpc <= 16:
        raise ValueError("bpc must be in [8, 16]")
    return np.uint8 if bpc == 8 else np.uint16


def uniform_frames(seed: int, n: int, w: int, h: int, bpc: int = 8) -> np.ndarray:
    rng = np.random.default_rng(seed)
    hi = (1 << bpc)
    return rng.integers(0, hi, size=(n, h, w), dtype=np.int64).astype(_dtype(bpc))


def uniform_yuv420(seed: int, n: int, w: int, h: int, bpc: int = 8) -> "Yuv420Batch":
    """4:2:0 pairs whose six planes are i.i.d. uniform over [0, 2^bpc - 1],
    drawn in the order ref Y, U, V, dist Y, U, V from one generator (integer
    draws only, so the same seed gives the same planes on every platform)."""
    rng = np.random.default_rng(seed)
    hi = 1 << bpc
    cw, ch = chroma_dims(w, h)
    dt = _dtype(bpc)
    shapes = [(n, h, w), (n, ch, cw), (n, ch, cw)] * 2
    planes = [rng.integers(0, hi, size=sh, dtype=np.int64).astype(dt) for sh in shapes]
    return Yuv420Batch(w, h, bpc, *planes)


def translation_walk(rng: np.random.Generator, n: int, max_shift: int) -> np.ndarray:
    """Cumulative integer offsets (n, 2) as (X_t, Y_t); X_0 = Y_0 = 0."""
    steps = rng.integers(-max_shift, max_shift + 1, size=(n, 2))
    steps[0] = 0
    return np.cumsum(steps, axis=0)


def _field_params(rng: np.random.Generator, n_waves: int = 8, amplitude: float = 100.0):
    a = rng.uniform(0.0, amplitude / n_waves, size=n_waves)
    u = rng.uniform(0.5, 8.0, size=n_waves) * rng.choice([-1.0, 1.0], size=n_waves)
    v = rng.uniform(0.5, 8.0, size=n_waves) * rng.choice([-1.0, 1.0], size=n_waves)
    phi = rng.uniform(0.0, 2.0 * np.pi, size=n_waves)
    return a, u, v, phi


def _render_canvas(params, w: int, h: int, u0: int, v0: int, cw: int, ch: int) -> np.ndarray:
    """Field value at field coordinates (u0 + j, v0 + i) for a canvas of ch x cw,
    with frequencies in cycles per w (resp. h) samples.  Separable rendering:
    sin(A + B) = sin A cos B + cos A sin B."""
    a, fu, fv, phi = params
    xs = (u0 + np.arange(cw, dtype=np.float64)) / w
    ys = (v0 + np.arange(ch, dtype=np.float64)) / h
    out = np.full((ch, cw), 128.0, dtype=np.float64)
    for k in range(len(a)):
        A = 2.0 * np.pi * fu[k] * xs
        B = 2.0 * np.pi * fv[k] * ys + phi[k]
        out += a[k] * (np.outer(np.cos(B), np.sin(A)) + np.outer(np.sin(B), np.cos(A)))
    return out.astype(np.float32)


def _workers() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _parallel(fn, items):
    """Run fn over items on a thread pool (numpy's generators and ufuncs release
    the GIL).  Every item carries its own generator, so results do not depend on
    the number of threads."""
    items = list(items)
    if len(items) <= 1:
        return [fn(it) for it in items]
    with ThreadPoolExecutor(_workers()) as ex:
        return list(ex.map(fn, items))


def _children(seed_seq: np.random.SeedSequence, n: int):
    return [np.random.default_rng(c) for c in seed_seq.spawn(n)]


def _quantise(field: np.ndarray, bpc: int) -> np.ndarray:
    if bpc == 8:
        return np.clip(np.rint(field), 0, 255).astype(np.uint8)
    scaled = field * np.float32(((1 << bpc) - 1) / 255.0)
    return np.clip(np.rint(scaled), 0, (1 << bpc) - 1).astype(np.uint16)


def smooth_sequence(seed: int, n: int, w: int, h: int, max_shift: int,
                    noise_sigma: float = 4.0, cut_frac: float = 0.0,
                    bpc: int = 8, return_offsets: bool = False):
    """(n, h, w) frames of a translating smooth field with noise and cuts."""
    rng = np.random.default_rng(seed)
    offs = translation_walk(rng, n, max_shift)
    n_cuts = int(round(cut_frac * n))
    cuts = set()
    if n_cuts > 0 and n > 1:
        cuts = set(int(c) for c in rng.choice(np.arange(1, n), size=n_cuts, replace=False))
    out = np.empty((n, h, w), dtype=_dtype(bpc))
    # segment boundaries: each segment has its own field and its own canvas
    starts = [0] + sorted(cuts)
    ends = starts[1:] + [n]
    for s, e in zip(starts, ends):
        params = _field_params(rng)
        seg = offs[s:e]
        min_x, max_x = int(seg[:, 0].min()), int(seg[:, 0].max())
        min_y, max_y = int(seg[:, 1].min()), int(seg[:, 1].max())
        # frame pixel (x, y) at offset (X, Y) shows field(x - X, y - Y)
        canvas = _render_canvas(params, w, h, -max_x, -max_y,
                                w + max_x - min_x, h + max_y - min_y)
        gens = _children(np.random.SeedSequence(int(rng.integers(0, 2**63 - 1))), e - s)

        def frame(job, canvas=canvas, max_x=max_x, max_y=max_y):
            t, g = job
            X, Y = int(offs[t, 0]), int(offs[t, 1])
            c0, r0 = max_x - X, max_y - Y
            f = canvas[r0:r0 + h, c0:c0 + w].copy()
            if noise_sigma > 0:
                f += g.standard_normal(size=(h, w), dtype=np.float32) * np.float32(noise_sigma)
            out[t] = _quantise(f, bpc)

        _parallel(frame, zip(range(s, e), gens))
    if return_offsets:
        return out, offs
    return out


@dataclass
class Yuv420Batch:
    w: int
    h: int
    bpc: int
    ref_y: np.ndarray
    ref_u: np.ndarray
    ref_v: np.ndarray
    dist_y: np.ndarray
    dist_u: np.ndarray
    dist_v: np.ndarray

    @property
    def n(self) -> int:
        return self.ref_y.shape[0]

    def planes(self):
        return (self.ref_y, self.ref_u, self.ref_v, self.dist_y, self.dist_u, self.dist_v)

    def nbytes(self) -> int:
        return sum(p.nbytes for p in self.planes())


def _distort(rng: np.random.Generator, plane: np.ndarray, sigma: float, bpc: int) -> np.ndarray:
    hi = (1 << bpc) - 1
    noise = rng.standard_normal(size=plane.shape, dtype=np.float32) * np.float32(sigma)
    d = np.rint(plane.astype(np.float32) + noise)
    np.clip(d, 0, hi, out=d)
    return d.astype(plane.dtype)


def yuv420_pairs(seed: int, n: int, w: int, h: int, max_shift: int = 2,
                 dist_sigma: float = 3.0, noise_sigma: float = 4.0,
                 bpc: int = 8) -> Yuv420Batch:
    rng = np.random.default_rng(seed)
    sub = [int(s) for s in rng.integers(0, 2**31 - 1, size=4)]
    ref_y, offs = smooth_sequence(sub[0], n, w, h, max_shift, noise_sigma=noise_sigma,
                                  bpc=bpc, return_offsets=True)
    cw, ch = chroma_dims(w, h)
    dt = _dtype(bpc)
    chroma = []
    for i in (1, 2):
        crng = np.random.default_rng(sub[i])
        params = _field_params(crng)
        cx = offs[:, 0] // 2
        cy = offs[:, 1] // 2
        min_x, max_x = int(cx.min()), int(cx.max())
        min_y, max_y = int(cy.min()), int(cy.max())
        canvas = _render_canvas(params, cw, ch, -max_x, -max_y,
                                cw + max_x - min_x, ch + max_y - min_y)
        plane = np.empty((n, ch, cw), dtype=dt)
        gens = _children(np.random.SeedSequence(int(crng.integers(0, 2**63 - 1))), n)

        def cframe(job, canvas=canvas, plane=plane, cx=cx, cy=cy, max_x=max_x, max_y=max_y):
            t, g = job
            c0, r0 = max_x - int(cx[t]), max_y - int(cy[t])
            f = canvas[r0:r0 + ch, c0:c0 + cw].copy()
            if noise_sigma > 0:
                f += g.standard_normal(size=(ch, cw), dtype=np.float32) * np.float32(noise_sigma)
            plane[t] = _quantise(f, bpc)

        _parallel(cframe, zip(range(n), gens))
        chroma.append(plane)
    dist_y = np.empty_like(ref_y)
    dist_u = np.empty_like(chroma[0])
    dist_v = np.empty_like(chroma[1])
    gens = _children(np.random.SeedSequence(sub[3]), n)

    def dframe(job):
        t, g = job
        dist_y[t] = _distort(g, ref_y[t], dist_sigma, bpc)
        dist_u[t] = _distort(g, chroma[0][t], dist_sigma, bpc)
        dist_v[t] = _distort(g, chroma[1][t], dist_sigma, bpc)

    _parallel(dframe, zip(range(n), gens))
    return Yuv420Batch(w, h, bpc, ref_y, chroma[0], chroma[1], dist_y, dist_u, dist_v)


# The five workloads, by what they are.  "batch" is frames (or pairs) per launch.
CONFIGS = {
    "pair_64x48_u8": dict(kind="uniform_pair", w=64, h=48, bpc=8, n=2, seed=1),
    "seq_576x324_u8": dict(kind="smooth", w=576, h=324, bpc=8, n=48, max_shift=2, seed=2),
    "seq_1920x1080_u8_cuts": dict(kind="smooth", w=1920, h=1080, bpc=8, n=300, max_shift=4,
                                  cut_frac=0.02, seed=3, batch=16),
    "yuv420_3840x2160_u8_pairs": dict(kind="yuv420", w=3840, h=2160, bpc=8, n=50, max_shift=2,
                                      dist_sigma=3.0, seed=4),
    "seq_3840x2160_u10": dict(kind="smooth", w=3840, h=2160, bpc=10, n=120, max_shift=3,
                              seed=5, batch=32),
}


def make(name: str, n: int | None = None):
    """Build the named workload (optionally with fewer frames / pairs)."""
    c = dict(CONFIGS[name])
    if n is not None:
        c["n"] = n
    kind = c["kind"]
    if kind == "uniform_pair":
        return uniform_frames(c["seed"], c["n"], c["w"], c["h"], c["bpc"])
    if kind == "smooth":
        return smooth_sequence(c["seed"], c["n"], c["w"], c["h"], c["max_shift"],
                               cut_frac=c.get("cut_frac", 0.0), bpc=c["bpc"])
    if kind == "yuv420":
        return yuv420_pairs(c["seed"], c["n"], c["w"], c["h"], max_shift=c["max_shift"],
                            dist_sigma=c["dist_sigma"], bpc=c["bpc"])
    raise KeyError(name)
