"""Failure detection on the GPU without faulting it: a stage wait that can
never complete (the stage expects more bytes than its copies deliver) runs
into the kernel's time bound; the kernel sets the context's device error word
and leaves, the host reads the status, and the context computes correctly
afterwards."""
import numpy as np
import pytest

import synth
from tests.gpu_util import dev_zeros, to_u64

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
