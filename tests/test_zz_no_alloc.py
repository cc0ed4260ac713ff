"""The allocation-free motion entry point against the oracle.

motion_submit_batch_noalloc serves callers that may not allocate device
memory (a host program that owns all device memory through its own pool, or
a loop where an allocation, which can synchronise the device, is not
acceptable): it keeps the previous frame's blurred plane in a fixed array
inside the library instead of in a context.  Two calls in a row (start a
sequence, then continue it) must give exactly the oracle's SAD sequence of
the frames, on both kernel paths, with the device error word read back as 0;
the context-based entry point on the same two batches must agree too.  This
file sorts last so that a run stopping at the first failure has run every
other test before it; it also passes alone."""
import numpy as np
import pytest

import synth
from tests.gpu_util import dev_zeros, oracle_sad, to_dev, to_u64

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


def context_sads(iif, d, split, w, h, bpc):
    out = dev_zeros(d.shape[0])
    with iif.MotionContext(w, h, bpc) as ctx:
        ctx.submit_batch(d[:split], out[:split])
        ctx.submit_batch(d[split:], out[split:])
    return out


@pytest.mark.parametrize("w,h,bpc,n,split", [
    (1920, 1080, 8, 12, 5),     # 16-byte-aligned rows: the TMA kernel
    (576, 324, 10, 9, 4),
    (333, 201, 8, 7, 3),        # odd pitch: the generic kernel
    (333, 201, 10, 6, 2),
])
def test_noalloc_two_calls_match_oracle(iif, oracle, w, h, bpc, n, split):
    import torch
    frames = synth.smooth_sequence(w + h + bpc, n, w, h, 3, bpc=bpc)
    d = to_dev(frames)
    want = oracle_sad(oracle, frames, bpc)
    got = dev_zeros(n)
    iif.motion_submit_batch_noalloc(d[:split], got[:split], bpc=bpc, continue_sequence=False)
    iif.motion_submit_batch_noalloc(d[split:], got[split:], bpc=bpc, continue_sequence=True)
    torch.cuda.synchronize()
    assert iif.motion_noalloc_device_error() == 0
    assert np.array_equal(to_u64(got), want)
    assert want[0] == 0 and want[split] > 0
    # the context-based entry point gives the same two batches the same SADs
    assert np.array_equal(to_u64(context_sads(iif, d, split, w, h, bpc)), want)


def test_noalloc_restart_and_limits(iif, oracle):
    import torch
    frames = synth.smooth_sequence(5, 4, 640, 360, 2)
    d = to_dev(frames)
    # a fresh start ignores whatever the array holds from earlier calls
    got = dev_zeros(4)
    iif.motion_submit_batch_noalloc(d, got, continue_sequence=False)
    torch.cuda.synchronize()
    assert iif.motion_noalloc_device_error() == 0
    assert np.array_equal(to_u64(got), oracle.motion_sad_sequence(frames, 8))
    # continuing with another frame size is refused
    small = to_dev(synth.smooth_sequence(6, 2, 320, 180, 2))
    with pytest.raises(iif.MotionError) as e:
        iif.motion_submit_batch_noalloc(small, dev_zeros(2), continue_sequence=True)
    assert e.value.code == 1
    # frames larger than the built-in array are refused before any launch
    big = torch.zeros((1, 2112, 4096), dtype=torch.uint8, device="cuda")
    with pytest.raises(iif.MotionError) as e:
        iif.motion_submit_batch_noalloc(big, dev_zeros(1))
    assert e.value.code == 5
