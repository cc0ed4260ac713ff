"""Allocation failures, injected on the host (motion_inject_alloc_failure makes
the nth allocation of the library fail without reaching the driver): every
entry point that allocates returns MOTION_ERR_OUT_OF_MEMORY, keeps nothing
half-made, and the same context (or a new one) computes the oracle's results
afterwards.  No GPU fault is involved."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

OOM = 7   # MOTION_ERR_OUT_OF_MEMORY


@pytest.fixture(scope="module")
def iif():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import integer_image_filter_gb300 as m
    from integer_image_filter_gb300 import _build
    _build.build()
    m.load_library()
    yield m
    m.motion_inject_alloc_failure(0)


def _frames(w, h, n, bpc=8, seed=3):
    import torch
    fr = synth.uniform_frames(seed, n, w, h, bpc)
    return fr, torch.from_numpy(fr.view(np.int16) if bpc > 8 else fr).cuda()


def test_init_fails_cleanly_at_each_allocation(iif, oracle):
    import torch
    # motion_init allocates two resident planes, the result slot (which also
    # holds the device error word) and the pinned readback slot
    for k in range(1, 5):
        iif.motion_inject_alloc_failure(k)
        with pytest.raises(iif.MotionError) as e:
            iif.MotionContext(64, 48, 8)
        assert e.value.code == OOM, k
    iif.motion_inject_alloc_failure(0)
    fr, d = _frames(64, 48, 3)
    out = torch.zeros(3, dtype=torch.int64, device="cuda")
    with iif.MotionContext(64, 48, 8) as ctx:
        ctx.submit_batch(d, out)
        torch.cuda.synchronize()
    assert out.cpu().numpy().astype(np.uint64).tolist() == [int(x) for x in oracle.motion_sad_sequence(fr, 8)]


@pytest.mark.parametrize("k", [1, 2])
def test_motion_v2_planes_fail_cleanly(iif, oracle, k):
    import torch
    fr, d = _frames(96, 40, 4, bpc=10, seed=4)
    out = torch.zeros(4, dtype=torch.int64, device="cuda")
    with iif.MotionContext(96, 40, 10) as ctx:
        iif.motion_inject_alloc_failure(k)      # the first or the second raw plane
        with pytest.raises(iif.MotionError) as e:
            ctx.submit_batch_v2(d, out)
        assert e.value.code == OOM
        iif.motion_inject_alloc_failure(0)
        ctx.submit_batch_v2(d, out)
        torch.cuda.synchronize()
        assert ctx.device_error() == 0
    assert out.cpu().numpy().astype(np.uint64).tolist() == [int(x) for x in oracle.motion_v2_sequence(fr, 10)]


def test_copy_scratch_failure_leaves_the_sequence_unchanged(iif, oracle):
    import torch
    w, h = 213, 40                              # rows 213 bytes apart: the copy kernel's scratch
    fr, d = _frames(w, h, 6, seed=5)
    out = torch.zeros(6, dtype=torch.int64, device="cuda")
    with iif.MotionContext(w, h, 8) as ctx:
        ctx.submit_batch(d[:2], out[:2])        # allocates a scratch for 2 frames
        iif.motion_inject_alloc_failure(1)      # growing it for 4 fails
        with pytest.raises(iif.MotionError) as e:
            ctx.submit_batch(d[2:], out[2:])
        assert e.value.code == OOM
        iif.motion_inject_alloc_failure(0)
        ctx.submit_batch(d[2:], out[2:])      # continues from frame 1, as if the failed call never ran
        torch.cuda.synchronize()
        assert ctx.device_error() == 0
    assert out.cpu().numpy().astype(np.uint64).tolist() == [int(x) for x in oracle.motion_sad_sequence(fr, 8)]


@pytest.mark.parametrize("k", [1, 2, 5])
def test_host_pipeline_staging_failure(iif, oracle, k):
    """The host-buffer call allocates two staging sets and result buffers, then
    a pinned result buffer; a failure at any of them returns the error and the
    next call runs."""
    b = synth.yuv420_pairs(6, 3, 128, 64, max_shift=2, dist_sigma=3.0)
    with iif.MotionContext(128, 64, 8) as ctx:
        iif.motion_inject_alloc_failure(k)
        with pytest.raises(iif.MotionError) as e:
            ctx.yuv420_batch_host(*b.planes())
        assert e.value.code == OOM
        iif.motion_inject_alloc_failure(0)
        sad, sse = ctx.yuv420_batch_host(*b.planes())
    assert np.asarray(sad, np.uint64).tolist() == [int(x) for x in oracle.motion_sad_sequence(b.ref_y, 8)]
    want = [[oracle.sse(b.ref_y[i], b.dist_y[i], 8), oracle.sse(b.ref_u[i], b.dist_u[i], 8),
             oracle.sse(b.ref_v[i], b.dist_v[i], 8)] for i in range(b.n)]
    assert np.asarray(sse, np.uint64).tolist() == want
