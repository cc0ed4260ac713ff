"""Failure detection on the GPU without faulting it: a stage wait that can
never complete (the stage expects more bytes than its copies deliver) runs
into the kernel's time bound; the kernel sets the context's device error word
and leaves, the host reads the status, and the context computes correctly
afterwards."""
import numpy as np
import pytest

import synth
from tests.gpu_util import dev_zeros, oracle_sse420, to_dev, to_u64

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


@pytest.mark.parametrize("mode", ["motion", "fused", "motion_v2"])
def test_stage_wait_times_out_and_context_recovers(iif, oracle, mode):
    import torch
    w, h, n = 640, 160, 3                     # 16-byte rows: the TMA kernel; interior and border tiles
    b = synth.yuv420_pairs(31, n, w, h)
    planes = [torch.from_numpy(p).cuda() for p in b.planes()]
    sad, sse = dev_zeros(n), dev_zeros((n, 3))
    with iif.MotionContext(w, h, 8) as ctx:
        assert ctx.device_error() == 0
        iif.motion_set_stall_injection(ctx.handle, True)
        run(ctx, mode, planes, sad, sse)
        torch.cuda.synchronize()               # the launch ends: the waits are bounded
        flags = ctx.device_error()
        assert flags & 1, flags
        assert ctx.device_error() == 0          # read and cleared
        iif.motion_set_stall_injection(ctx.handle, False)
        ctx.reset()
        run(ctx, mode, planes, sad, sse)
        torch.cuda.synchronize()
        assert ctx.device_error() == 0
    seq = oracle.motion_v2_sequence if mode == "motion_v2" else oracle.motion_sad_sequence
    assert np.array_equal(to_u64(sad), seq(b.ref_y, 8))


def run(ctx, mode, planes, sad, sse):
    if mode == "fused":
        ctx.yuv420_batch(*planes, sad, sse)
    elif mode == "motion_v2":
        ctx.submit_batch_v2(planes[0], sad)
    else:
        ctx.submit_batch(planes[0], sad)


def test_submit_returns_device_error_and_restarts(iif, oracle):
    """motion_submit reads the error word in the same readback as the SAD: a
    wait that ran out gives MOTION_ERR_DEVICE (no SAD written), the word is
    cleared, and the sequence restarts with the next frame."""
    w, h, n = 640, 160, 4
    frames = synth.uniform_frames(32, n, w, h)
    d = to_dev(frames)
    with iif.MotionContext(w, h, 8) as ctx:
        ctx.submit(d[0])
        ctx.submit(d[1])                          # a sequence is running
        iif.motion_set_stall_injection(ctx.handle, True)
        with pytest.raises(iif.MotionError) as e:
            ctx.submit(d[2])
        assert e.value.code == iif.MOTION_ERR_DEVICE
        assert ctx.device_error() == 0            # the call read and cleared the word
        iif.motion_set_stall_injection(ctx.handle, False)
        got = [ctx.submit(d[i])[0] for i in range(n)]
    assert got == [int(x) for x in oracle.motion_sad_sequence(frames, 8)]
    assert got[0] == 0                            # restarted


@pytest.mark.parametrize("kind", ["yuv420_host", "frames_host"])
def test_host_calls_return_device_error_outputs_untouched(iif, oracle, kind):
    w, h, n = 640, 160, 3
    b = synth.yuv420_pairs(33, n, w, h)
    host = [np.ascontiguousarray(p) for p in b.planes()]
    sad = np.full(n, 7, np.uint64)
    sse = np.full((n, 3), 7, np.uint64)
    with iif.MotionContext(w, h, 8) as ctx:
        ctx.submit_batch_host(host[0])            # a sequence is running
        iif.motion_set_stall_injection(ctx.handle, True)
        with pytest.raises(iif.MotionError) as e:
            if kind == "yuv420_host":
                ctx.yuv420_batch_host(*host, sad_out=sad, sse_out=sse)
            else:
                ctx.submit_batch_host(host[0], sad_out=sad)
        assert e.value.code == iif.MOTION_ERR_DEVICE
        assert (sad == 7).all() and (sse == 7).all()   # nothing written on error
        assert ctx.device_error() == 0
        iif.motion_set_stall_injection(ctx.handle, False)
        if kind == "yuv420_host":
            got_sad, got_sse = ctx.yuv420_batch_host(*host)
            assert np.array_equal(got_sse, oracle_sse420(oracle, b))
        else:
            got_sad = ctx.submit_batch_host(host[0])
    assert np.array_equal(got_sad, oracle.motion_sad_sequence(b.ref_y, 8))   # restarted


def test_async_call_error_is_collected_and_restarts(iif, oracle):
    """The asynchronous batch call cannot see the word; motion_device_error is
    its collect step, and a set word restarts the sequence."""
    import torch
    w, h, n = 640, 160, 3
    frames = synth.uniform_frames(34, n, w, h)
    d = to_dev(frames)
    sad = dev_zeros(n)
    with iif.MotionContext(w, h, 8) as ctx:
        ctx.submit_batch(d, sad)
        iif.motion_set_stall_injection(ctx.handle, True)
        ctx.submit_batch(d, sad)                  # incomplete: the waits run out
        assert ctx.device_error() & 1
        iif.motion_set_stall_injection(ctx.handle, False)
        ctx.submit_batch(d, sad)                  # the context restarted the sequence
        torch.cuda.synchronize()
        assert ctx.device_error() == 0
    assert np.array_equal(to_u64(sad), oracle.motion_sad_sequence(frames, 8))


def test_noalloc_error_word_is_collected(iif, oracle):
    """The allocation-free calls report a wait that ran out through
    motion_noalloc_device_error; a continuing call is then refused until a
    sequence is started, and that one matches the oracle."""
    import torch
    w, h, n = 640, 160, 4
    frames = synth.uniform_frames(35, n, w, h)
    d = to_dev(frames)
    sad = dev_zeros(n)
    assert iif.motion_noalloc_device_error() == 0
    iif.motion_noalloc_set_stall_injection(True)
    try:
        iif.motion_submit_batch_noalloc(d[:2], sad[:2])
        flags = iif.motion_noalloc_device_error()
    finally:
        iif.motion_noalloc_set_stall_injection(False)
    assert flags & 1, flags
    assert iif.motion_noalloc_device_error() == 0          # read and cleared
    with pytest.raises(iif.MotionError) as e:
        iif.motion_submit_batch_noalloc(d[2:], sad[2:], continue_sequence=True)
    assert e.value.code == 1
    iif.motion_submit_batch_noalloc(d[:2], sad[:2], continue_sequence=False)
    iif.motion_submit_batch_noalloc(d[2:], sad[2:], continue_sequence=True)
    torch.cuda.synchronize()
    assert iif.motion_noalloc_device_error() == 0
    assert np.array_equal(to_u64(sad), oracle.motion_sad_sequence(frames, 8))
