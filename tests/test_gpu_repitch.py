"""Layouts the TMA cannot address -- a plane base, row pitch or frame stride that
is not a multiple of 16 bytes -- are copied into 16-byte-aligned rows first and
then take the TMA kernel (two launches per call: the copy and the motion
kernel).  Bit-exact against the oracle for every source alignment granule
(1, 2, 4 and 8 bytes), odd widths, motion, motion_v2 over two calls and the
fused 4:2:0 pass, and equal to the generic kernel on the same inputs."""
import numpy as np
import pytest

from tests.gpu_util import oracle_sse420
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def iif():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import integer_image_filter_gb300 as m
    from integer_image_filter_gb300 import _build
    _build.build()
    m.load_library()
    return m


def _layout(frames: np.ndarray, extra_pitch: int, offset: int):
    """A device view of `frames` with rows `w*s + extra_pitch` bytes apart and
    the first sample `offset` bytes into its buffer."""
    import torch
    n, h, w = frames.shape
    s = frames.itemsize
    pitch = w * s + extra_pitch
    buf = torch.zeros(offset + n * h * pitch + 64, dtype=torch.uint8, device="cuda")
    host = np.zeros((n, h, pitch), np.uint8)
    host[:, :, :w * s] = frames.view(np.uint8).reshape(n, h, w * s)
    buf[offset:offset + n * h * pitch] = torch.from_numpy(host.reshape(-1)).to("cuda")
    return buf, offset, pitch


def _submit(iif, ctx, kind, buf, offset, pitch, n, h, out):
    lib = iif.load_library()
    fn = lib.motion_v2_submit_batch if kind == "motion_v2" else lib.motion_submit_batch
    rc = fn(ctx.handle, buf.data_ptr() + offset, n, h * pitch, pitch, None, out.data_ptr())
    assert rc == 0, iif.motion_strerror(rc)


# (w, h, bpc, extra pitch bytes, base offset bytes): source granules 1, 2, 4, 8
LAYOUTS = [(854 // 4, 48, 8, 0, 0),     # 213-byte rows: granule 1
           (107, 37, 8, 3, 1),          # odd pitch and an odd base
           (130, 34, 8, 2, 0),          # 132-byte pitch: granule 4
           (127, 35, 10, 2, 2),         # 256-byte pitch, 2 bytes into the buffer: granule 2
           (203, 67, 10, 0, 2),         # 406-byte rows at a 2-byte offset: granule 2
           (300, 40, 16, 8, 8),         # 608-byte pitch, 8-byte offset: granule 8
           (1918 // 2, 540, 8, 0, 0)]   # a 959-byte row at 540 rows


@pytest.mark.parametrize("w,h,bpc,extra,off", LAYOUTS)
@pytest.mark.parametrize("kind", ["motion", "motion_v2"])
def test_unaligned_layouts_take_the_tma_kernel(iif, oracle, w, h, bpc, extra, off, kind):
    import torch
    n = 5
    fr = synth.uniform_frames(31 + w + bpc, 2 * n, w, h, bpc)
    want = (oracle.motion_v2_sequence if kind == "motion_v2" else oracle.motion_sad_sequence)(fr, bpc)
    buf, offset, pitch = _layout(fr, extra, off)
    got = {}
    for path in (iif.MOTION_PATH_AUTO, iif.MOTION_PATH_GENERIC):
        out = torch.zeros(2 * n, dtype=torch.int64, device="cuda")
        with iif.MotionContext(w, h, bpc) as ctx:
            ctx.set_kernel_path(path)
            l0 = iif.motion_kernel_launch_count()
            _submit(iif, ctx, kind, buf, offset, pitch, n, h, out[:n])
            launches = iif.motion_kernel_launch_count() - l0
            _submit(iif, ctx, kind, buf, offset + n * h * pitch, pitch, n, h, out[n:])
            torch.cuda.synchronize()
            assert ctx.device_error() == 0
        if path == iif.MOTION_PATH_AUTO:
            assert launches == 2          # the copy into aligned rows, then the TMA kernel
        got[path] = out.cpu().numpy().astype(np.uint64)
        assert got[path].tolist() == [int(x) for x in want], (path, w, h, bpc)
    assert np.array_equal(got[iif.MOTION_PATH_AUTO], got[iif.MOTION_PATH_GENERIC])


@pytest.mark.parametrize("w,h,bpc", [(213, 48, 8), (203, 67, 10)])
def test_unaligned_fused_pairs(iif, oracle, w, h, bpc):
    """Fused 4:2:0 pass on planes at an odd base offset (granule 1 for 8-bit,
    2 for 10-bit): motion SAD and the three SSEs."""
    import torch
    b = synth.uniform_yuv420(77 + bpc, 4, w, h, bpc)
    off = 1 if bpc == 8 else 2
    views = []
    keep = []
    for p in b.planes():
        n, ph, pw = p.shape
        buf, o, pitch = _layout(p, 0, off)
        keep.append(buf)
        views.append((buf.data_ptr() + o, pitch, ph * pitch))
    sad = torch.zeros(b.n, dtype=torch.int64, device="cuda")
    sse = torch.zeros((b.n, 3), dtype=torch.int64, device="cuda")
    lib = iif.load_library()
    with iif.MotionContext(w, h, bpc) as ctx:
        rc = lib.motion_psnr_yuv420_batch(ctx.handle, b.n, views[0][0], views[1][0], views[2][0],
                                          views[3][0], views[4][0], views[5][0], views[0][1],
                                          views[1][1], views[0][2], views[1][2], None,
                                          sad.data_ptr(), sse.data_ptr())
        assert rc == 0, iif.motion_strerror(rc)
        torch.cuda.synchronize()
        assert ctx.device_error() == 0
    assert sad.cpu().numpy().astype(np.uint64).tolist() == [int(x) for x in oracle.motion_sad_sequence(b.ref_y, bpc)]
    assert np.array_equal(sse.cpu().numpy().astype(np.uint64), oracle_sse420(oracle, b))


@pytest.mark.parametrize("kind", ["motion", "motion_v2", "fused"])
def test_copy_limit_splits_a_call_into_parts(iif, oracle, kind):
    """A copy limit of about 3 frames' (pairs') scratch turns a 10-frame call on
    unaligned planes into 4 parts (4 copies and 4 motion launches), each
    continuing the sequence; the results are the oracle's."""
    import torch
    w, h, bpc, n = 213, 48, 8, 10
    lib = iif.load_library()
    if kind == "fused":
        b = synth.uniform_yuv420(91, n, w, h, bpc)
        keep, views = [], []
        for p in b.planes():
            buf, o, pitch = _layout(p, 0, 1)
            keep.append(buf)
            views.append((buf.data_ptr() + o, pitch, p.shape[1] * pitch))
        py, puv = (w + 15) // 16 * 16, ((w + 1) // 2 + 15) // 16 * 16
        per = 2 * py * h + 4 * puv * ((h + 1) // 2)
        sad = torch.zeros(n, dtype=torch.int64, device="cuda")
        sse = torch.zeros((n, 3), dtype=torch.int64, device="cuda")
        with iif.MotionContext(w, h, bpc) as ctx:
            ctx.set_copy_limit(3 * per)
            l0 = iif.motion_kernel_launch_count()
            rc = lib.motion_psnr_yuv420_batch(ctx.handle, n, views[0][0], views[1][0], views[2][0],
                                              views[3][0], views[4][0], views[5][0], views[0][1],
                                              views[1][1], views[0][2], views[1][2], None,
                                              sad.data_ptr(), sse.data_ptr())
            assert rc == 0, iif.motion_strerror(rc)
            torch.cuda.synchronize()
            assert iif.motion_kernel_launch_count() - l0 == 8
            assert ctx.device_error() == 0
        assert sad.cpu().numpy().astype(np.uint64).tolist() == [int(x) for x in oracle.motion_sad_sequence(b.ref_y, bpc)]
        assert np.array_equal(sse.cpu().numpy().astype(np.uint64), oracle_sse420(oracle, b))
        return
    fr = synth.uniform_frames(92, n, w, h, bpc)
    want = (oracle.motion_v2_sequence if kind == "motion_v2" else oracle.motion_sad_sequence)(fr, bpc)
    buf, offset, pitch = _layout(fr, 0, 0)
    out = torch.zeros(n, dtype=torch.int64, device="cuda")
    with iif.MotionContext(w, h, bpc) as ctx:
        ctx.set_copy_limit(3 * ((w + 15) // 16 * 16) * h)
        l0 = iif.motion_kernel_launch_count()
        _submit(iif, ctx, kind, buf, offset, pitch, n, h, out)
        torch.cuda.synchronize()
        assert iif.motion_kernel_launch_count() - l0 == 8
        assert ctx.device_error() == 0
    assert out.cpu().numpy().astype(np.uint64).tolist() == [int(x) for x in want]
