"""The largest frame sides (32768 samples wide or high) on the GPU, for the
motion SAD, motion_v2 and the moment sums.  Frames that are constant along
one axis blur to the 1-D blur along the other (the mirror along the constant
axis changes nothing), so the oracle run on a 3-sample-thick frame with the
same profile gives every row (or column) of the expected result."""
import numpy as np
import pytest

from tests.gpu_util import dev_zeros, to_dev, to_u64

pytestmark = pytest.mark.gpu

MAX = 32768


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


def _profiles(bpc, n, length, seed):
    rng = np.random.default_rng(seed)
    dt = np.uint8 if bpc == 8 else np.uint16
    return rng.integers(0, 1 << bpc, size=(n, length)).astype(dt)


def _frames(prof, w, h, wide):
    """(n, h, w) frames constant along y (wide) or along x (tall)."""
    if wide:
        return np.ascontiguousarray(np.broadcast_to(prof[:, None, :], (prof.shape[0], h, w)))
    return np.ascontiguousarray(np.broadcast_to(prof[:, :, None], (prof.shape[0], h, w)))


def _thin(prof_row, wide):
    # the same profile, 3 samples thick along the constant axis
    return np.repeat(prof_row[None, :], 3, axis=0) if wide else np.repeat(prof_row[:, None], 3, axis=1)


@pytest.mark.parametrize("path", ["auto", "tma32", "tma16"])
@pytest.mark.parametrize("bpc", [8, 10])
@pytest.mark.parametrize("wide", [True, False])
def test_motion_and_v2_at_the_largest_side(iif, oracle, bpc, wide, path):
    """Both tile heights (the wide frame chooses 128 x 16 tiles, the tall one
    128 x 32; each is also forced to the other)."""
    import torch
    w, h = (MAX, 64) if wide else (64, MAX)
    n = 3
    prof = _profiles(bpc, n, w if wide else h, seed=bpc * 7 + wide)
    frames = _frames(prof, w, h, wide)
    other = h if wide else w           # the constant axis' length

    def line(b):                       # the 1-D result every row (column) repeats
        return b[0] if wide else b[:, 0]

    blur = [line(oracle.blur(_thin(prof[i], wide), bpc).astype(np.int64)) for i in range(n)]
    want = [0] + [other * int(np.abs(blur[i] - blur[i - 1]).sum()) for i in range(1, n)]
    want_v2 = [0] + [other * int(np.abs(line(oracle.blur_diff(_thin(prof[i - 1], wide),
                                                              _thin(prof[i], wide), bpc))
                                         .astype(np.int64)).sum()) for i in range(1, n)]
    d = to_dev(frames)
    out, out2 = dev_zeros(n), dev_zeros(n)
    with iif.MotionContext(w, h, bpc) as ctx:
        ctx.set_kernel_path({"auto": iif.MOTION_PATH_AUTO, "tma32": iif.MOTION_PATH_TMA_32,
                             "tma16": iif.MOTION_PATH_TMA_16}[path])
        ctx.submit_batch(d, out)
        ctx.submit_batch_v2(d, out2)
        torch.cuda.synchronize()
        assert ctx.device_error() == 0
    assert to_u64(out).tolist() == want
    assert to_u64(out2).tolist() == want_v2


@pytest.mark.parametrize("wide", [True, False])
def test_moments_at_the_largest_side(iif, wide):
    import torch
    w, h = (MAX, 48) if wide else (48, MAX)
    prof = _profiles(10, 2, w if wide else h, seed=5 + wide)
    frames = _frames(prof, w, h, wide)
    other = h if wide else w
    out = dev_zeros((1, 4))
    d = to_dev(frames)
    iif.moment_sums_batch(d[0:1], d[1:2], 10, out)
    torch.cuda.synchronize()
    r, s = prof[0].astype(np.uint64), prof[1].astype(np.uint64)
    want = [other * int(r.sum()), other * int(s.sum()), other * int((r * r).sum()),
            other * int((s * s).sum())]
    assert to_u64(out)[0].tolist() == want


def test_sides_beyond_the_largest_are_rejected(iif):
    import torch
    with pytest.raises(iif.MotionError):
        iif.MotionContext(MAX + 1, 16, 8)
    # straight through the C ABI (the binding would refuse the short buffer
    # itself): the library rejects the size before it reads anything
    a = torch.zeros((1, 4, 4), dtype=torch.uint8, device="cuda")
    out = dev_zeros((1, 4))
    rc = iif.load_library().moment_sums_batch(MAX + 1, 4, 8, 1, a.data_ptr(), a.data_ptr(),
                                              MAX + 1, 0, None, out.data_ptr())
    assert rc == 5                     # MOTION_ERR_TOO_LARGE
