"""Python binding of libmotion_gb300 (the GB300 integer motion / PSNR-SSE
library).  Argument marshalling only: every step of the computation runs in
the library's CUDA kernels; there is no CPU fallback.  If the shared library
has not been built this module raises on first use.

The functions carry the names of the C ABI in ``include/motion.h``.  Device
arguments may be PyTorch CUDA tensors (uint8, or int16/uint16 holding uint16
samples) or raw device addresses (int); streams may be ``torch.cuda.Stream``
objects, raw ``cudaStream_t`` values (int) or None (the current PyTorch stream
when torch is loaded, else the legacy default stream).
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import numpy as np

from . import _build

__all__ = [
    "MotionError", "load_library", "motion_init", "motion_destroy", "motion_reset",
    "motion_submit", "motion_submit_batch", "motion_psnr_yuv420_batch",
    "motion_psnr_yuv420_batch_host", "motion_reserve_host_staging", "psnr_sse",
    "psnr_sse_yuv420_batch", "motion_scores_from_sad", "psnr_from_sse",
    "motion_kernel_launch_count", "motion_strerror", "MotionContext", "EXPORTED_SYMBOLS",
    "motion_set_kernel_path", "motion_device_error", "MOTION_PATH_AUTO", "MOTION_PATH_GENERIC",
    "MOTION_PATH_TMA_32", "MOTION_PATH_TMA_16",
    "motion_submit_batch_noalloc", "motion_set_stall_injection", "moment_sums_batch",
    "moments_from_sums", "motion_v2_submit_batch", "motion_plan_chunks", "motion_tile_order",
    "motion_inject_alloc_failure", "motion_submit_batch_host", "motion_set_copy_limit",
    "motion_noalloc_device_error", "motion_noalloc_set_stall_injection", "MOTION_ERR_DEVICE",
    "motion_launch_blocks", "motion_launch_shape",
]

EXPORTED_SYMBOLS = (
    "motion_init", "motion_destroy", "motion_reset", "motion_submit", "motion_submit_batch",
    "motion_psnr_yuv420_batch", "motion_psnr_yuv420_batch_host", "motion_reserve_host_staging",
    "psnr_sse", "psnr_sse_yuv420_batch", "motion_scores_from_sad", "psnr_from_sse",
    "motion_kernel_launch_count", "motion_strerror", "motion_last_cuda_error",
    "motion_set_kernel_path", "motion_device_error", "motion_submit_batch_noalloc",
    "motion_set_stall_injection", "moment_sums_batch", "moments_from_sums",
    "motion_v2_submit_batch", "motion_plan_chunks", "motion_tile_order", "motion_inject_alloc_failure",
    "motion_submit_batch_host", "motion_set_copy_limit", "motion_noalloc_device_error",
    "motion_noalloc_set_stall_injection", "motion_launch_blocks", "motion_launch_shape",
)

# Status of a call whose kernel set the device error word (include/motion.h).
MOTION_ERR_DEVICE = 10

_LIB: ctypes.CDLL | None = None
_LIB_LOCK = threading.Lock()


class MotionError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        msg = _LIB.motion_strerror(code).decode() if _LIB is not None else str(code)
        extra = ""
        if _LIB is not None and code == 6:
            extra = f" (cudaError {_LIB.motion_last_cuda_error()})"
        super().__init__(f"{what}: {msg}{extra} [status {code}]")


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    U64P = ctypes.POINTER(ctypes.c_uint64)
    DP = ctypes.POINTER(ctypes.c_double)
    sig = {
        "motion_init": ([I, I, I, ctypes.POINTER(P)], I),
        "motion_destroy": ([P], I),
        "motion_reset": ([P], I),
        "motion_submit": ([P, P, Z, P, U64P, DP], I),
        "motion_submit_batch": ([P, P, I, Z, Z, P, P], I),
        "motion_psnr_yuv420_batch": ([P, I, P, P, P, P, P, P, Z, Z, Z, Z, P, P, P], I),
        "motion_psnr_yuv420_batch_host": ([P, I, P, P, P, P, P, P, Z, Z, Z, Z, P, P], I),
        "motion_reserve_host_staging": ([P, I, Z, Z], I),
        "psnr_sse": ([P, P, Z, Z, I, I, I, P, P], I),
        "psnr_sse_yuv420_batch": ([I, I, I, I, P, P, P, P, P, P, Z, Z, Z, Z, P, P], I),
        "motion_scores_from_sad": ([P, I, I, I, P, P, P], I),
        "psnr_from_sse": ([ctypes.c_uint64, ctypes.c_uint64, I, DP, DP], I),
        "motion_kernel_launch_count": ([], ctypes.c_uint64),
        "motion_strerror": ([I], ctypes.c_char_p),
        "motion_last_cuda_error": ([], I),
        "motion_set_kernel_path": ([P, I], I),
        "motion_device_error": ([P, ctypes.POINTER(I)], I),
        "motion_submit_batch_noalloc": ([P, I, I, I, I, Z, Z, I, P, P], I),
        "motion_set_stall_injection": ([P, I], I),
        "moment_sums_batch": ([I, I, I, I, P, P, Z, Z, P, P], I),
        "moments_from_sums": ([P, I, I, I, P], I),
        "motion_v2_submit_batch": ([P, P, I, Z, Z, P, P], I),
        "motion_plan_chunks": ([I, I, I, I, ctypes.POINTER(I)], I),
        "motion_tile_order": ([I, I, I, ctypes.c_longlong, ctypes.POINTER(I)], I),
        "motion_inject_alloc_failure": ([I], I),
        "motion_submit_batch_host": ([P, P, I, Z, Z, I, P], I),
        "motion_set_copy_limit": ([P, Z], I),
        "motion_noalloc_device_error": ([P, ctypes.POINTER(I)], I),
        "motion_noalloc_set_stall_injection": ([I], I),
        "motion_launch_blocks": ([I, I, I, I, I, ctypes.c_longlong, ctypes.POINTER(I),
                                  ctypes.POINTER(ctypes.c_longlong)], I),
        "motion_launch_shape": ([I, I, I, I, I, ctypes.POINTER(I)], I),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libmotion_gb300.so (built in-tree by ``__graft_entry__.build()``)."""
    global _LIB
    with _LIB_LOCK:   # threads that get here first together load it once
        if _LIB is None:
            p = path or _build.lib_path()
            if not os.path.exists(p):
                raise RuntimeError(
                    f"{p} is missing: build the CUDA library first (python -c 'import "
                    "__graft_entry__ as g; g.build()'); there is no CPU fallback")
            _LIB = _declare(ctypes.CDLL(p))
        return _LIB


def _check(code: int, what: str) -> None:
    if code != 0:
        raise MotionError(code, what)


# ----------------------------------------------------------------- marshalling
def _addr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if hasattr(x, "is_cuda") and not x.is_cuda:
            raise ValueError("expected a CUDA tensor")
        return int(x.data_ptr())
    raise TypeError(f"cannot take the device address of {type(x).__name__}")


def _host_addr(x) -> int:
    if isinstance(x, int):
        return x
    if isinstance(x, np.ndarray):
        return int(x.ctypes.data)
    if hasattr(x, "data_ptr"):
        if getattr(x, "is_cuda", False):
            raise ValueError("expected a host tensor")
        return int(x.data_ptr())
    raise TypeError(f"cannot take the host address of {type(x).__name__}")


def _stream(s) -> int:
    if s is None:
        try:
            import torch
            if torch.cuda.is_available() and torch.cuda.is_initialized():
                return int(torch.cuda.current_stream().cuda_stream)
        except Exception:
            pass
        return 0
    if isinstance(s, int):
        return s
    if hasattr(s, "cuda_stream"):
        return int(s.cuda_stream)
    raise TypeError("stream must be a torch.cuda.Stream, an int handle or None")


def _itemsize(t) -> int:
    return int(t.element_size()) if hasattr(t, "element_size") else int(t.itemsize)


# The C ABI takes plain pointers and cannot see how much memory is behind them;
# these checks keep a short array from turning into an out-of-bounds access.
def _span(t):
    """Bytes from t's first element to the end of what it may address (the
    tensor's storage, or a contiguous array's own data), or None if unknown."""
    if t is None or isinstance(t, int):
        return None
    if hasattr(t, "untyped_storage"):
        return int(t.untyped_storage().nbytes()) - int(t.storage_offset()) * _itemsize(t)
    if isinstance(t, np.ndarray) and t.flags["C_CONTIGUOUS"]:
        return int(t.nbytes)
    return None


def _need(t, nbytes: int, what: str) -> None:
    span = _span(t)
    if span is not None and nbytes > 0 and span < nbytes:
        raise ValueError(f"{what} holds {span} bytes from its first element; {nbytes} are needed")


def _need_out(t, count: int, what: str) -> None:
    """An output the library writes as `count` contiguous 64-bit integers."""
    if t is None or isinstance(t, int) or count <= 0:
        return
    if _itemsize(t) != 8:
        raise TypeError(f"{what} must hold 64-bit integers")
    contiguous = t.is_contiguous() if hasattr(t, "is_contiguous") else bool(t.flags["C_CONTIGUOUS"])
    if not contiguous:
        raise ValueError(f"{what} must be contiguous")
    _need(t, 8 * count, what)


def _plane_bytes(n: int, w: int, h: int, bpc: int, pitch: int, stride: int) -> int:
    """Bytes a batch of n planes of w x h samples addresses from its first
    sample (0, i.e. no check, for arguments the library itself rejects)."""
    if n <= 0 or w <= 0 or h <= 0 or not 8 <= bpc <= 16 or pitch < w * (1 if bpc == 8 else 2):
        return 0
    return (n - 1) * stride + (h - 1) * pitch + w * (1 if bpc == 8 else 2)


def _layout(t):
    """(pitch_bytes, frame_stride_bytes) of a (h, w) or (n, h, w) array/tensor
    whose last dimension is contiguous."""
    st = t.stride() if callable(getattr(t, "stride", None)) else tuple(s // t.itemsize for s in t.strides)
    if st[-1] != 1:
        raise ValueError("samples within a row must be contiguous")
    isz = _itemsize(t)
    pitch = st[-2] * isz
    stride = st[0] * isz if len(st) == 3 else 0
    return pitch, stride


# ----------------------------------------------------------------- C-ABI names
def motion_init(w: int, h: int, bpc: int) -> int:
    lib = load_library()
    h_ = ctypes.c_void_p()
    _check(lib.motion_init(w, h, bpc, ctypes.byref(h_)), "motion_init")
    return int(h_.value)


def motion_destroy(ctx: int) -> None:
    _check(load_library().motion_destroy(ctx), "motion_destroy")


def motion_reset(ctx: int) -> None:
    _check(load_library().motion_reset(ctx), "motion_reset")


def motion_submit(ctx: int, frame, pitch_bytes: int | None = None, stream=None):
    """One frame; returns (SAD, score) after the stream has been synchronised."""
    if pitch_bytes is None:
        pitch_bytes, _ = _layout(frame)
    sad = ctypes.c_uint64()
    score = ctypes.c_double()
    _check(load_library().motion_submit(ctx, _addr(frame), pitch_bytes, _stream(stream),
                                        ctypes.byref(sad), ctypes.byref(score)), "motion_submit")
    return int(sad.value), float(score.value)


def motion_submit_batch(ctx: int, frames, sad_out, n: int | None = None,
                        frame_stride: int | None = None, pitch_bytes: int | None = None,
                        stream=None) -> None:
    if n is None:
        n = int(frames.shape[0])
    if pitch_bytes is None or frame_stride is None:
        p, s = _layout(frames)
        pitch_bytes = p if pitch_bytes is None else pitch_bytes
        frame_stride = s if frame_stride is None else frame_stride
    _need_out(sad_out, n, "sad_out")
    _check(load_library().motion_submit_batch(ctx, _addr(frames), n, frame_stride, pitch_bytes,
                                              _stream(stream), _addr(sad_out)),
           "motion_submit_batch")


def motion_submit_batch_host(ctx: int, frames, sad_out: np.ndarray | None = None,
                             n: int | None = None, frame_stride: int | None = None,
                             pitch_bytes: int | None = None, frames_per_chunk: int = 0) -> np.ndarray:
    """Host frames in, host SADs out (uint64[n]); uploads overlap the kernels."""
    if n is None:
        n = int(frames.shape[0])
    if pitch_bytes is None or frame_stride is None:
        p, s = _layout(frames)
        pitch_bytes = p if pitch_bytes is None else pitch_bytes
        frame_stride = s if frame_stride is None else frame_stride
    if sad_out is None:
        sad_out = np.zeros(n, np.uint64)
    _need_out(sad_out, n, "sad_out")
    _check(load_library().motion_submit_batch_host(ctx, _host_addr(frames), n, frame_stride, pitch_bytes,
                                                   frames_per_chunk, _host_addr(sad_out)),
           "motion_submit_batch_host")
    return sad_out


def motion_v2_submit_batch(ctx: int, frames, sad_out, n: int | None = None,
                           frame_stride: int | None = None, pitch_bytes: int | None = None,
                           stream=None) -> None:
    if n is None:
        n = int(frames.shape[0])
    if pitch_bytes is None or frame_stride is None:
        p, s = _layout(frames)
        pitch_bytes = p if pitch_bytes is None else pitch_bytes
        frame_stride = s if frame_stride is None else frame_stride
    _need_out(sad_out, n, "sad_out")
    _check(load_library().motion_v2_submit_batch(ctx, _addr(frames), n, frame_stride,
                                                 pitch_bytes, _stream(stream), _addr(sad_out)),
           "motion_v2_submit_batch")


@dataclass
class Yuv420Layout:
    pitch_y: int
    pitch_uv: int
    stride_y: int
    stride_uv: int


def _yuv_layout(ref_y, ref_u) -> Yuv420Layout:
    py, sy = _layout(ref_y)
    pu, su = _layout(ref_u)
    return Yuv420Layout(py, pu, sy, su)


def motion_psnr_yuv420_batch(ctx: int, ref_y, ref_u, ref_v, dist_y, dist_u, dist_v,
                             sad_out, sse_out, n: int | None = None,
                             layout: Yuv420Layout | None = None, stream=None) -> None:
    if n is None:
        n = int(ref_y.shape[0])
    lay = layout or _yuv_layout(ref_y, ref_u)
    _need_out(sad_out, n, "sad_out")
    _need_out(sse_out, 3 * n, "sse_out")
    _check(load_library().motion_psnr_yuv420_batch(
        ctx, n, _addr(ref_y), _addr(ref_u), _addr(ref_v), _addr(dist_y), _addr(dist_u),
        _addr(dist_v), lay.pitch_y, lay.pitch_uv, lay.stride_y, lay.stride_uv, _stream(stream),
        _addr(sad_out), _addr(sse_out)), "motion_psnr_yuv420_batch")


def motion_psnr_yuv420_batch_host(ctx: int, ref_y, ref_u, ref_v, dist_y, dist_u, dist_v,
                                  sad_out: np.ndarray | None = None,
                                  sse_out: np.ndarray | None = None,
                                  n: int | None = None, layout: Yuv420Layout | None = None):
    """Host pictures in, host results out (uint64[n], uint64[n][3])."""
    if n is None:
        n = int(ref_y.shape[0])
    lay = layout or _yuv_layout(ref_y, ref_u)
    if sad_out is None:
        sad_out = np.zeros(n, np.uint64)
    if sse_out is None:
        sse_out = np.zeros((n, 3), np.uint64)
    _need_out(sad_out, n, "sad_out")
    _need_out(sse_out, 3 * n, "sse_out")
    _check(load_library().motion_psnr_yuv420_batch_host(
        ctx, n, _host_addr(ref_y), _host_addr(ref_u), _host_addr(ref_v), _host_addr(dist_y),
        _host_addr(dist_u), _host_addr(dist_v), lay.pitch_y, lay.pitch_uv, lay.stride_y,
        lay.stride_uv, _host_addr(sad_out), _host_addr(sse_out)), "motion_psnr_yuv420_batch_host")
    return sad_out, sse_out


def motion_reserve_host_staging(ctx: int, pairs_per_chunk: int = 0, stride_y: int = 0,
                                stride_uv: int = 0) -> None:
    _check(load_library().motion_reserve_host_staging(ctx, pairs_per_chunk, stride_y, stride_uv),
           "motion_reserve_host_staging")


def psnr_sse(ref, dist, bpc: int, sse_out, w: int | None = None, h: int | None = None,
             ref_pitch: int | None = None, dist_pitch: int | None = None, stream=None) -> None:
    if h is None or w is None:
        h, w = int(ref.shape[-2]), int(ref.shape[-1])
    if ref_pitch is None:
        ref_pitch, _ = _layout(ref)
    if dist_pitch is None:
        dist_pitch, _ = _layout(dist)
    _need(ref, _plane_bytes(1, w, h, bpc, ref_pitch, 0), "ref")
    _need(dist, _plane_bytes(1, w, h, bpc, dist_pitch, 0), "dist")
    _need_out(sse_out, 1, "sse_out")
    _check(load_library().psnr_sse(_addr(ref), _addr(dist), ref_pitch, dist_pitch, w, h, bpc,
                                   _stream(stream), _addr(sse_out)), "psnr_sse")


def psnr_sse_yuv420_batch(w: int, h: int, bpc: int, ref_y, ref_u, ref_v, dist_y, dist_u, dist_v,
                          sse_out, n: int | None = None, layout: Yuv420Layout | None = None,
                          stream=None) -> None:
    if n is None:
        n = int(ref_y.shape[0])
    lay = layout or _yuv_layout(ref_y, ref_u)
    cw, ch = (w + 1) // 2, (h + 1) // 2
    for t, what in ((ref_y, "ref_y"), (dist_y, "dist_y")):
        _need(t, _plane_bytes(n, w, h, bpc, lay.pitch_y, lay.stride_y), what)
    for t, what in ((ref_u, "ref_u"), (ref_v, "ref_v"), (dist_u, "dist_u"), (dist_v, "dist_v")):
        _need(t, _plane_bytes(n, cw, ch, bpc, lay.pitch_uv, lay.stride_uv), what)
    _need_out(sse_out, 3 * n, "sse_out")
    _check(load_library().psnr_sse_yuv420_batch(
        w, h, bpc, n, _addr(ref_y), _addr(ref_u), _addr(ref_v), _addr(dist_y), _addr(dist_u),
        _addr(dist_v), lay.pitch_y, lay.pitch_uv, lay.stride_y, lay.stride_uv, _stream(stream),
        _addr(sse_out)), "psnr_sse_yuv420_batch")


def motion_scores_from_sad(sad, w: int, h: int, next_score: float | None = None):
    s = np.ascontiguousarray(np.asarray(sad, dtype=np.uint64))
    n = s.size
    score = np.zeros(n, np.float64)
    motion2 = np.zeros(n, np.float64)
    nxt = ctypes.c_double(next_score) if next_score is not None else None
    _check(load_library().motion_scores_from_sad(
        s.ctypes.data, n, w, h, ctypes.addressof(nxt) if nxt is not None else None,
        score.ctypes.data, motion2.ctypes.data), "motion_scores_from_sad")
    return score, motion2


def moment_sums_batch(ref, dist, bpc: int, out, w: int | None = None, h: int | None = None,
                      n: int | None = None, pitch: int | None = None, stride: int | None = None,
                      stream=None) -> None:
    """Moment sums of n luma pairs ((n, h, w) or (h, w) device tensors sharing one
    layout) into the device uint64/int64 tensor out[n][4]."""
    if h is None or w is None:
        h, w = int(ref.shape[-2]), int(ref.shape[-1])
    if n is None:
        n = int(ref.shape[0]) if len(ref.shape) == 3 else 1
    if pitch is None or stride is None:
        p, st = _layout(ref)
        pitch = p if pitch is None else pitch
        stride = st if stride is None else stride
    _need(ref, _plane_bytes(n, w, h, bpc, pitch, stride), "ref")
    _need(dist, _plane_bytes(n, w, h, bpc, pitch, stride), "dist")
    _need_out(out, 4 * n, "out")
    _check(load_library().moment_sums_batch(w, h, bpc, n, _addr(ref), _addr(dist), pitch, stride,
                                            _stream(stream), _addr(out)), "moment_sums_batch")


def moments_from_sums(sums, w: int, h: int) -> np.ndarray:
    """float64[n][4] moments (each sum over w*h) from uint64[n][4] moment sums."""
    s = np.ascontiguousarray(np.asarray(sums, dtype=np.uint64)).reshape(-1, 4)
    out = np.zeros(s.shape, np.float64)
    _check(load_library().moments_from_sums(s.ctypes.data, s.shape[0], w, h, out.ctypes.data),
           "moments_from_sums")
    return out


def motion_tile_order(w: int, h: int, chunks: int, block: int) -> tuple[int, int, int]:
    """(tile column, tile row, chunk) of one block of a batched launch (host only)."""
    t = (ctypes.c_int * 3)()
    _check(load_library().motion_tile_order(w, h, chunks, block, t), "motion_tile_order")
    return int(t[0]), int(t[1]), int(t[2])


def motion_launch_blocks(w: int, h: int, n: int, resident_ctas: int, block: int = -1, tile_rows: int = 32):
    """Diagnostic: the block count of a batched motion launch in 128 x
    tile_rows tiles and, for block >= 0, that block's (tile column, tile row,
    first frame, end frame)."""
    out = (ctypes.c_int * 4)()
    cnt = ctypes.c_longlong()
    _check(load_library().motion_launch_blocks(w, h, n, tile_rows, resident_ctas, block, out,
                                               ctypes.byref(cnt)),
           "motion_launch_blocks")
    return int(cnt.value), (tuple(out) if block >= 0 else None)


def motion_launch_shape(w: int, h: int, n: int, resident_ctas: int, v2: bool = False) -> int:
    """Diagnostic: the tile height (16 or 32) of a batched motion-only launch."""
    rows = ctypes.c_int()
    _check(load_library().motion_launch_shape(w, h, n, int(bool(v2)), resident_ctas, ctypes.byref(rows)),
           "motion_launch_shape")
    return int(rows.value)


def motion_plan_chunks(w: int, h: int, n: int, resident_ctas: int) -> int:
    """Frame chunks of a batched launch (host only; see include/motion.h)."""
    c = ctypes.c_int()
    _check(load_library().motion_plan_chunks(w, h, n, resident_ctas, ctypes.byref(c)),
           "motion_plan_chunks")
    return int(c.value)


def psnr_from_sse(sse: int, n_samples: int, bpc: int):
    mse = ctypes.c_double()
    db = ctypes.c_double()
    _check(load_library().psnr_from_sse(sse, n_samples, bpc, ctypes.byref(mse), ctypes.byref(db)),
           "psnr_from_sse")
    return float(mse.value), float(db.value)


def motion_submit_batch_noalloc(frames, sad_out, w: int | None = None, h: int | None = None,
                                bpc: int = 8, n: int | None = None,
                                frame_stride: int | None = None, pitch_bytes: int | None = None,
                                continue_sequence: bool = False, stream=None) -> None:
    """Batched motion SAD without a context and without any allocation: the
    previous frame's blurred plane lives in a fixed array inside the library
    (for callers that may not allocate device memory)."""
    if n is None:
        n = int(frames.shape[0])
    if h is None or w is None:
        h, w = int(frames.shape[-2]), int(frames.shape[-1])
    if pitch_bytes is None or frame_stride is None:
        p, s = _layout(frames)
        pitch_bytes = p if pitch_bytes is None else pitch_bytes
        frame_stride = s if frame_stride is None else frame_stride
    _need(frames, _plane_bytes(n, w, h, bpc, pitch_bytes, frame_stride), "frames")
    _need_out(sad_out, n, "sad_out")
    _check(load_library().motion_submit_batch_noalloc(
        _addr(frames), n, w, h, bpc, frame_stride, pitch_bytes, 1 if continue_sequence else 0,
        _stream(stream), _addr(sad_out)), "motion_submit_batch_noalloc")


def motion_noalloc_device_error(stream=None) -> int:
    """The collect step of the allocation-free calls: waits for `stream`, reads
    and clears this device's error word (a set word also makes the next
    continuing call refuse until a sequence is started)."""
    v = ctypes.c_int()
    _check(load_library().motion_noalloc_device_error(_stream(stream), ctypes.byref(v)),
           "motion_noalloc_device_error")
    return int(v.value)


def motion_noalloc_set_stall_injection(on: bool) -> None:
    """Test hook: the allocation-free calls' stage waits can never complete."""
    _check(load_library().motion_noalloc_set_stall_injection(1 if on else 0),
           "motion_noalloc_set_stall_injection")


MOTION_PATH_AUTO = 0
MOTION_PATH_GENERIC = 1
MOTION_PATH_TMA_32 = 2      # the TMA kernel with 128 x 32 tiles for motion-only launches
MOTION_PATH_TMA_16 = 3      # ... with 128 x 16 tiles


def motion_set_kernel_path(ctx: int, path: int) -> None:
    _check(load_library().motion_set_kernel_path(ctx, path), "motion_set_kernel_path")


def motion_inject_alloc_failure(nth: int) -> None:
    """Test hook: the nth allocation of the library from now on fails (0: off)."""
    _check(load_library().motion_inject_alloc_failure(nth), "motion_inject_alloc_failure")


def motion_set_copy_limit(ctx: int, nbytes: int) -> None:
    _check(load_library().motion_set_copy_limit(ctx, nbytes), "motion_set_copy_limit")


def motion_set_stall_injection(ctx: int, on: bool) -> None:
    _check(load_library().motion_set_stall_injection(ctx, 1 if on else 0),
           "motion_set_stall_injection")


def motion_device_error(ctx: int) -> int:
    v = ctypes.c_int()
    _check(load_library().motion_device_error(ctx, ctypes.byref(v)), "motion_device_error")
    return int(v.value)


def motion_kernel_launch_count() -> int:
    return int(load_library().motion_kernel_launch_count())


def motion_strerror(code: int) -> str:
    return load_library().motion_strerror(code).decode()


class MotionContext:
    """Owning wrapper over a motion_ctx handle."""

    def __init__(self, w: int, h: int, bpc: int = 8):
        self.w, self.h, self.bpc = w, h, bpc
        self.handle = motion_init(w, h, bpc)

    def close(self) -> None:
        if self.handle:
            motion_destroy(self.handle)
            self.handle = 0

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def reset(self) -> None:
        motion_reset(self.handle)

    def set_copy_limit(self, nbytes: int) -> None:
        motion_set_copy_limit(self.handle, nbytes)

    def set_kernel_path(self, path: int) -> None:
        motion_set_kernel_path(self.handle, path)

    def device_error(self) -> int:
        return motion_device_error(self.handle)

    def _frames_fit(self, frames, n: int) -> None:
        if hasattr(frames, "shape") and len(frames.shape) in (2, 3):
            pitch, stride = _layout(frames)
            _need(frames, _plane_bytes(n, self.w, self.h, self.bpc, pitch, stride), "frames")

    def _yuv_fit(self, planes, n: int) -> None:
        if all(hasattr(t, "shape") for t in planes):
            lay = _yuv_layout(planes[0], planes[1])
            cw, ch = (self.w + 1) // 2, (self.h + 1) // 2
            for i, t in enumerate(planes):
                luma = i in (0, 3)
                _need(t, _plane_bytes(n, self.w if luma else cw, self.h if luma else ch, self.bpc,
                                      lay.pitch_y if luma else lay.pitch_uv,
                                      lay.stride_y if luma else lay.stride_uv), "picture plane")

    def submit(self, frame, stream=None):
        self._frames_fit(frame, 1)
        return motion_submit(self.handle, frame, stream=stream)

    def submit_batch(self, frames, sad_out, stream=None) -> None:
        self._frames_fit(frames, int(frames.shape[0]))
        motion_submit_batch(self.handle, frames, sad_out, stream=stream)

    def submit_batch_host(self, frames, sad_out=None, frames_per_chunk: int = 0) -> np.ndarray:
        """motion_submit_batch_host: host frames (numpy or a CPU tensor), host SADs."""
        self._frames_fit(frames, int(frames.shape[0]))
        return motion_submit_batch_host(self.handle, frames, sad_out, frames_per_chunk=frames_per_chunk)

    def submit_batch_v2(self, frames, sad_out, stream=None) -> None:
        self._frames_fit(frames, int(frames.shape[0]))
        motion_v2_submit_batch(self.handle, frames, sad_out, stream=stream)

    def yuv420_batch(self, ref_y, ref_u, ref_v, dist_y, dist_u, dist_v, sad_out, sse_out,
                     stream=None) -> None:
        self._yuv_fit((ref_y, ref_u, ref_v, dist_y, dist_u, dist_v), int(ref_y.shape[0]))
        motion_psnr_yuv420_batch(self.handle, ref_y, ref_u, ref_v, dist_y, dist_u, dist_v,
                                 sad_out, sse_out, stream=stream)

    def yuv420_batch_host(self, ref_y, ref_u, ref_v, dist_y, dist_u, dist_v, sad_out=None,
                          sse_out=None):
        self._yuv_fit((ref_y, ref_u, ref_v, dist_y, dist_u, dist_v), int(ref_y.shape[0]))
        return motion_psnr_yuv420_batch_host(self.handle, ref_y, ref_u, ref_v, dist_y, dist_u,
                                             dist_v, sad_out, sse_out)
