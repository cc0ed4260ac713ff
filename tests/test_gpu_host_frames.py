"""motion_submit_batch_host: host frames in chunks, uploads on one stream
overlapping the motion kernel of the previous chunk on another, host SADs
out.  Bit-exact against the oracle for several chunk sizes, at 8 and 10 bits,
on rows the TMA takes in place and on odd widths (the copy kernel), continuing
a sequence started by a device-buffer call, and sharing its staging with the
fused host-buffer pass on the same context."""
import numpy as np
import pytest

import synth
from tests.gpu_util import oracle_sad, oracle_sse420

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


@pytest.mark.parametrize("w,h,bpc", [(320, 180, 8), (203, 67, 10), (256, 96, 16)])
@pytest.mark.parametrize("chunk", [0, 1, 3])
def test_host_frames_match_the_oracle(iif, oracle, w, h, bpc, chunk):
    fr = synth.uniform_frames(40 + w + chunk, 11, w, h, bpc)
    with iif.MotionContext(w, h, bpc) as ctx:
        got = ctx.submit_batch_host(fr, frames_per_chunk=chunk)
        assert ctx.device_error() == 0
    assert got.tolist() == [int(x) for x in oracle_sad(oracle, fr, bpc)]


def test_host_call_continues_a_device_sequence(iif, oracle):
    import torch
    w, h = 640, 160
    fr = synth.uniform_frames(9, 12, w, h, 8)
    d = torch.from_numpy(fr[:5]).cuda()
    first = torch.zeros(5, dtype=torch.int64, device="cuda")
    with iif.MotionContext(w, h, 8) as ctx:
        ctx.submit_batch(d, first)
        rest = ctx.submit_batch_host(fr[5:], frames_per_chunk=2)
        got = first.cpu().numpy().astype(np.uint64).tolist() + rest.tolist()
    assert got == [int(x) for x in oracle_sad(oracle, fr, 8)]


def test_frames_and_pairs_share_the_staging(iif, oracle):
    w, h = 256, 96
    b = synth.yuv420_pairs(13, 5, w, h, max_shift=2, dist_sigma=3.0)
    fr = synth.uniform_frames(14, 7, w, h, 8)
    with iif.MotionContext(w, h, 8) as ctx:
        got = ctx.submit_batch_host(fr, frames_per_chunk=2)
        assert got.tolist() == [int(x) for x in oracle_sad(oracle, fr, 8)]
        ctx.reset()
        sad, sse = ctx.yuv420_batch_host(*b.planes())
        assert np.asarray(sad, np.uint64).tolist() == [int(x) for x in oracle_sad(oracle, b.ref_y, 8)]
        assert np.array_equal(np.asarray(sse, np.uint64), oracle_sse420(oracle, b))
        ctx.reset()
        got = ctx.submit_batch_host(fr)                 # all frames in one chunk
        assert got.tolist() == [int(x) for x in oracle_sad(oracle, fr, 8)]
        assert ctx.device_error() == 0
