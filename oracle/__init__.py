"""CPU oracle for the integer motion feature and the PSNR squared-error sum.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package.  The product
path (the CUDA library and its Python binding) never imports it, and this
package imports nothing from the product.

The arithmetic lives in ``oracle.c`` (plain single-threaded C, compiled here with
gcc); this module only builds it and marshals numpy arrays into it.

Sources, by page title and section:
  ADR-1392 ("CUDA motion, PSNR and moment kernels add one atomic per block, the
  motion SAD filters separably, ..."), Context and Decision 4 -- separable blur,
  vertical pass rounded >> bpc then horizontal >> 16; exact 64-bit sums equal to
  the CPU's.  Taps {3571, 16004, 26386, 16004, 3571}, mirror boundaries and the
  score / motion2 formulas are this library's definition of the motion feature.

Pins (checked by ``tests/test_oracle_pins.py`` against the mathematics, not
against this code): constant-frame and two-constant closed forms, impulse closed
form, row- and column-constant frames against numpy/scipy mirror-padded
convolution, the hand-worked 6x6 example, brute-force 25-MAC per-output loop on
tiny frames, SAD/SSE invariants and planted-mistake builds; moment sums against
closed forms and numpy sums; the motion_v2 difference blur against the pinned
reading-A blur (non-negative differences), closed forms, a floor-rounding impulse
worked by hand and the brute-force per-output loop.  The PSNR dB helper
``psnr_db`` is "parity unpinned" (no page gives its formula; it is not graded).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_LIB = None


def build(defines: tuple[str, ...] = (), out_path: str | None = None) -> str:
    """Compile oracle.c into a shared object (gcc, -O2, no fast-math, no FMA
    contraction concerns: integer only).  ``defines`` are extra -D flags used by
    the planted-mistake tests.  Returns the .so path."""
    os.makedirs(_BUILD, exist_ok=True)
    if out_path is None:
        out_path = os.path.join(_BUILD, "liboracle.so")
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", "-Wextra",
           "-fvisibility=hidden", _SRC, "-o", out_path]
    cmd[1:1] = ["-D" + d for d in defines]
    subprocess.run(cmd, check=True)
    return out_path


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    P = ctypes.c_void_p
    lib.oracle_mirror.argtypes = [ctypes.c_int, ctypes.c_int]
    lib.oracle_mirror.restype = ctypes.c_int
    lib.oracle_blur.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_size_t,
                                ctypes.c_int, P]
    lib.oracle_blur.restype = ctypes.c_int
    lib.oracle_sad.argtypes = [P, P, ctypes.c_size_t]
    lib.oracle_sad.restype = ctypes.c_uint64
    lib.oracle_motion_sad_sequence.argtypes = [P, ctypes.c_int, ctypes.c_size_t,
                                               ctypes.c_int, ctypes.c_int,
                                               ctypes.c_size_t, ctypes.c_int, P]
    lib.oracle_motion_sad_sequence.restype = ctypes.c_int
    lib.oracle_sse.argtypes = [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_size_t,
                               ctypes.c_size_t, ctypes.c_int]
    lib.oracle_sse.restype = ctypes.c_uint64
    lib.oracle_scores.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P,
                                  P, P]
    lib.oracle_scores.restype = ctypes.c_int
    lib.oracle_moment_sums.argtypes = [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_size_t,
                                       ctypes.c_size_t, ctypes.c_int, P]
    lib.oracle_moment_sums.restype = ctypes.c_int
    lib.oracle_moments.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P]
    lib.oracle_moments.restype = ctypes.c_int
    lib.oracle_blur_diff.argtypes = [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_size_t,
                                     ctypes.c_int, P]
    lib.oracle_blur_diff.restype = ctypes.c_int
    lib.oracle_motion_v2_sequence.argtypes = [P, ctypes.c_int, ctypes.c_size_t, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_size_t, ctypes.c_int, P]
    lib.oracle_motion_v2_sequence.restype = ctypes.c_int
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle library."""
    global _LIB
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _LOCK:
        if _LIB is None:
            so = os.path.join(_BUILD, "liboracle.so")
            if (not os.path.exists(so)
                    or os.path.getmtime(so) < os.path.getmtime(_SRC)):
                build()
            _LIB = _bind(ctypes.CDLL(so))
    return _LIB


class Oracle:
    """numpy front end over one oracle build (the default, or a planted one)."""

    def __init__(self, lib: ctypes.CDLL | None = None):
        self.lib = lib if lib is not None else load()

    @staticmethod
    def _frames(a: np.ndarray, bpc: int) -> np.ndarray:
        want = np.uint8 if bpc == 8 else np.uint16
        if a.dtype != want:
            raise TypeError(f"bpc={bpc} needs {np.dtype(want).name} samples, got {a.dtype}")
        if a.dtype == np.uint16 and a.dtype.byteorder not in ("=", "<", "|"):
            raise TypeError("uint16 samples must be little-endian")
        return a

    def mirror(self, i: int, n: int) -> int:
        return int(self.lib.oracle_mirror(i, n))

    def blur(self, frame: np.ndarray, bpc: int) -> np.ndarray:
        """B plane (h x w uint16) of one frame (h x w, uint8 or uint16)."""
        f = self._frames(frame, bpc)
        if f.ndim != 2 or f.strides[1] != f.itemsize:
            f = np.ascontiguousarray(f)
        h, w = f.shape
        out = np.empty((h, w), dtype=np.uint16)
        rc = self.lib.oracle_blur(f.ctypes.data, w, h, f.strides[0], bpc, out.ctypes.data)
        if rc != 0:
            raise ValueError(f"oracle_blur rejected w={w} h={h} bpc={bpc}")
        return out

    def sad(self, a: np.ndarray, b: np.ndarray) -> int:
        a = np.ascontiguousarray(a, dtype=np.uint16)
        b = np.ascontiguousarray(b, dtype=np.uint16)
        if a.shape != b.shape:
            raise ValueError("shape mismatch")
        return int(self.lib.oracle_sad(a.ctypes.data, b.ctypes.data, a.size))

    def motion_sad_sequence(self, frames: np.ndarray, bpc: int) -> np.ndarray:
        """frames: (n, h, w).  Returns uint64[n], SAD[0] = 0."""
        f = self._frames(frames, bpc)
        if f.ndim != 3:
            raise ValueError("frames must be (n, h, w)")
        if f.strides[2] != f.itemsize:
            f = np.ascontiguousarray(f)
        n, h, w = f.shape
        out = np.zeros(n, dtype=np.uint64)
        if n == 0:
            return out
        rc = self.lib.oracle_motion_sad_sequence(f.ctypes.data, n, f.strides[0], w, h,
                                                 f.strides[1], bpc, out.ctypes.data)
        if rc != 0:
            raise ValueError(f"oracle_motion_sad_sequence rejected w={w} h={h} bpc={bpc}")
        return out

    def sse(self, ref: np.ndarray, dist: np.ndarray, bpc: int) -> int:
        r = self._frames(ref, bpc)
        d = self._frames(dist, bpc)
        if r.shape != d.shape or r.ndim != 2:
            raise ValueError("ref and dist must be equal-shape 2-D planes")
        if r.strides[1] != r.itemsize:
            r = np.ascontiguousarray(r)
        if d.strides[1] != d.itemsize:
            d = np.ascontiguousarray(d)
        h, w = r.shape
        return int(self.lib.oracle_sse(r.ctypes.data, d.ctypes.data, w, h,
                                       r.strides[0], d.strides[0], bpc))

    def scores(self, sad: np.ndarray, w: int, h: int,
               next_score: float | None = None) -> tuple[np.ndarray, np.ndarray]:
        s = np.ascontiguousarray(sad, dtype=np.uint64)
        n = s.size
        score = np.zeros(n, dtype=np.float64)
        motion2 = np.zeros(n, dtype=np.float64)
        nxt = None
        if next_score is not None:
            nxt = ctypes.c_double(next_score)
        rc = self.lib.oracle_scores(s.ctypes.data, n, w, h,
                                    ctypes.addressof(nxt) if nxt is not None else None,
                                    score.ctypes.data, motion2.ctypes.data)
        if rc != 0:
            raise ValueError("oracle_scores rejected its arguments")
        return score, motion2


def _pair(ref: np.ndarray, dist: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    if ref.shape != dist.shape or ref.ndim != 2:
        raise ValueError("ref and dist must be equal-shape 2-D planes")
    if ref.strides[1] != ref.itemsize:
        ref = np.ascontiguousarray(ref)
    if dist.strides[1] != dist.itemsize:
        dist = np.ascontiguousarray(dist)
    return ref, dist


def _moment_sums(self, ref: np.ndarray, dist: np.ndarray, bpc: int) -> np.ndarray:
    """uint64[4]: sum ref, sum dist, sum ref^2, sum dist^2 of one luma pair."""
    r, d = _pair(self._frames(ref, bpc), self._frames(dist, bpc))
    h, w = r.shape
    out = np.zeros(4, dtype=np.uint64)
    rc = self.lib.oracle_moment_sums(r.ctypes.data, d.ctypes.data, w, h, r.strides[0],
                                     d.strides[0], bpc, out.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_moment_sums rejected its arguments")
    return out


def _moments(self, sums: np.ndarray, w: int, h: int) -> np.ndarray:
    """float64[n][4] moments (sums over w*h) from uint64[n][4] moment sums."""
    s = np.ascontiguousarray(sums, dtype=np.uint64).reshape(-1, 4)
    out = np.zeros(s.shape, dtype=np.float64)
    rc = self.lib.oracle_moments(s.ctypes.data, s.shape[0], w, h, out.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_moments rejected its arguments")
    return out


def _blur_diff(self, prev: np.ndarray, cur: np.ndarray, bpc: int) -> np.ndarray:
    """motion_v2 blur (h x w int32) of prev - cur."""
    p = np.ascontiguousarray(self._frames(prev, bpc))
    c = np.ascontiguousarray(self._frames(cur, bpc))
    if p.shape != c.shape or p.ndim != 2:
        raise ValueError("prev and cur must be equal-shape 2-D frames")
    h, w = p.shape
    out = np.empty((h, w), dtype=np.int32)
    rc = self.lib.oracle_blur_diff(p.ctypes.data, c.ctypes.data, w, h, p.strides[0], bpc,
                                   out.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle_blur_diff rejected w={w} h={h} bpc={bpc}")
    return out


def _motion_v2_sequence(self, frames: np.ndarray, bpc: int) -> np.ndarray:
    """frames: (n, h, w).  Returns uint64[n] motion_v2 SADs, SAD[0] = 0."""
    f = self._frames(frames, bpc)
    if f.ndim != 3:
        raise ValueError("frames must be (n, h, w)")
    f = np.ascontiguousarray(f)
    n, h, w = f.shape
    out = np.zeros(n, dtype=np.uint64)
    if n == 0:
        return out
    rc = self.lib.oracle_motion_v2_sequence(f.ctypes.data, n, f.strides[0], w, h, f.strides[1],
                                            bpc, out.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle_motion_v2_sequence rejected w={w} h={h} bpc={bpc}")
    return out


Oracle.moment_sums = _moment_sums
Oracle.moments = _moments
Oracle.blur_diff = _blur_diff
Oracle.motion_v2_sequence = _motion_v2_sequence


def psnr_db(sse: int, n_samples: int, bpc: int) -> float:
    """PSNR in dB from an SSE: 10*log10((2^bpc - 1)^2 * N / SSE); +inf when
    SSE == 0.  Parity unpinned: the pages name psnr_* outputs without a formula."""
    if sse == 0:
        return math.inf
    peak = float((1 << bpc) - 1)
    return 10.0 * math.log10(peak * peak * n_samples / float(sse))


def default() -> Oracle:
    return Oracle()
