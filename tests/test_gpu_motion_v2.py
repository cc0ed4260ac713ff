"""motion_v2 (the blur of prev - cur with floor rounding, SAD of |blur|) on the
GPU against the CPU oracle, bit for bit, through the C ABI: the three sequence
workloads at full size in their batch sizes, continuity across batches and
after a reset, the TMA and generic kernels on aligned and unaligned layouts,
tiny and ragged frames at 8, 10 and 16 bits, independence from the
motion_submit_batch state, and a closed form at a large size."""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import synth
from tests.gpu_util import dev_zeros, to_dev, to_u64

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


def oracle_v2(o, frames, bpc):
    """Oracle motion_v2 SADs, split into overlapping chunks run in threads (chunk
    [s, e) runs frames [s-1, e) so that its first SAD is against frame s-1)."""
    n = frames.shape[0]
    if n <= 8:
        return o.motion_v2_sequence(frames, bpc)
    k = 16
    bounds = np.linspace(0, n, k + 1).astype(int)

    def run(i):
        s, e = int(bounds[i]), int(bounds[i + 1])
        if e <= s:
            return np.zeros(0, np.uint64)
        lo = max(s - 1, 0)
        r = o.motion_v2_sequence(frames[lo:e], bpc)
        return r if s == 0 else r[1:]

    with ThreadPoolExecutor(k) as ex:
        parts = list(ex.map(run, range(k)))
    return np.concatenate(parts).astype(np.uint64)


def padded_dev(frames, align_bytes=16):
    n, h, w = frames.shape
    s = frames.itemsize
    wp = ((w * s + align_bytes - 1) // align_bytes * align_bytes) // s
    big = np.zeros((n, h, wp), dtype=frames.dtype)
    big[:, :, :w] = frames
    return to_dev(big)[:, :, :w]


def run_v2(iif, d, w, h, bpc, batch, path=None):
    import torch
    n = d.shape[0]
    out = dev_zeros(n)
    with iif.MotionContext(w, h, bpc) as ctx:
        if path is not None:
            ctx.set_kernel_path(path)
        for s in range(0, n, batch):
            ctx.submit_batch_v2(d[s:s + batch], out[s:s + batch])
        torch.cuda.synchronize()
        assert ctx.device_error() == 0
    return to_u64(out)


@pytest.mark.parametrize("name", ["seq_576x324_u8", "seq_1920x1080_u8_cuts", "seq_3840x2160_u10"])
def test_workloads_full_size(iif, oracle, name):
    c = synth.CONFIGS[name]
    frames = synth.make(name)
    want = oracle_v2(oracle, frames, c["bpc"])
    got = run_v2(iif, to_dev(frames), c["w"], c["h"], c["bpc"], c.get("batch", frames.shape[0]))
    assert np.array_equal(got, want)


def test_batch_sizes_continuity(iif, oracle):
    frames = synth.make("seq_576x324_u8")
    want = oracle.motion_v2_sequence(frames, 8)
    d = to_dev(frames)
    for batch in (1, 2, 7, 16, 48):
        assert np.array_equal(run_v2(iif, d, 576, 324, 8, batch), want), batch


@pytest.mark.parametrize("bpc", [8, 10, 16])
def test_paths_and_layouts(iif, oracle, bpc):
    from integer_image_filter_gb300 import MOTION_PATH_GENERIC
    rng = np.random.default_rng(bpc + 100)
    w, h, n = 389, 131, 9
    dt = np.uint8 if bpc == 8 else np.uint16
    base = rng.integers(0, 1 << bpc, size=(h + 8, w + 8)).astype(np.int64)
    frames = np.stack([np.roll(base, (i, 2 * i), axis=(0, 1))[:h, :w] for i in range(n)]).astype(dt)
    want = oracle.motion_v2_sequence(frames, bpc)
    padded = padded_dev(frames)
    assert np.array_equal(run_v2(iif, padded, w, h, bpc, 4), want)          # TMA kernel
    assert np.array_equal(run_v2(iif, padded, w, h, bpc, 4, MOTION_PATH_GENERIC), want)
    assert np.array_equal(run_v2(iif, to_dev(frames), w, h, bpc, 3), want)   # unaligned: generic


@pytest.mark.parametrize("bpc", [8, 10, 16])
@pytest.mark.parametrize("wh", [(3, 3), (5, 7), (127, 33), (130, 36), (257, 131), (1283, 723),
                                (128, 100), (256, 70), (385, 98)])
def test_tiny_and_ragged(iif, oracle, bpc, wh):
    w, h = wh
    rng = np.random.default_rng(w * 3 + h + bpc)
    dt = np.uint8 if bpc == 8 else np.uint16
    frames = rng.integers(0, 1 << bpc, size=(5, h, w)).astype(dt)
    want = oracle.motion_v2_sequence(frames, bpc)
    assert np.array_equal(run_v2(iif, padded_dev(frames), w, h, bpc, 2), want), (bpc, w, h)
    assert np.array_equal(run_v2(iif, to_dev(frames), w, h, bpc, 5), want), (bpc, w, h)


def test_reset_and_independent_of_motion_state(iif, oracle):
    import torch
    frames = synth.make("seq_576x324_u8")[:10]
    want_v2 = oracle.motion_v2_sequence(frames, 8)
    want_a = oracle.motion_sad_sequence(frames, 8)
    d = to_dev(frames)
    with iif.MotionContext(576, 324, 8) as ctx:
        v2, a = dev_zeros(10), dev_zeros(10)
        for s in range(0, 10, 3):      # interleave the two sequences on one context
            ctx.submit_batch_v2(d[s:s + 3], v2[s:s + 3])
            ctx.submit_batch(d[s:s + 3], a[s:s + 3])
        torch.cuda.synchronize()
        assert np.array_equal(to_u64(v2), want_v2)
        assert np.array_equal(to_u64(a), want_a)
        ctx.reset()
        again = dev_zeros(4)
        ctx.submit_batch_v2(d[6:10], again)
        torch.cuda.synchronize()
        assert np.array_equal(to_u64(again), oracle.motion_v2_sequence(frames[6:10], 8))


def test_constant_frames_closed_form_large(iif):
    """Alternating constant frames c1, c2: SAD = |c1 - c2| 2^(16-bpc) w h (the
    floor rounding leaves a constant difference exact, of either sign)."""
    import torch
    w, h = 8192, 4320
    for bpc, (c1, c2) in ((8, (200, 13)), (10, (3, 1000)), (16, (65535, 0))):
        dt = torch.uint8 if bpc == 8 else torch.int16
        v1 = c1 if bpc == 8 or c1 < 32768 else c1 - 65536
        v2 = c2 if bpc == 8 or c2 < 32768 else c2 - 65536
        d = torch.empty((4, h, w), dtype=dt, device="cuda")
        d[0::2] = v1
        d[1::2] = v2
        out = dev_zeros(4)
        with iif.MotionContext(w, h, bpc) as ctx:
            ctx.submit_batch_v2(d, out)
            torch.cuda.synchronize()
        exp = abs(c1 - c2) * (1 << (16 - bpc)) * w * h
        assert [int(x) for x in out.cpu()] == [0, exp, exp, exp], bpc


@pytest.mark.parametrize("bpc", [9, 12, 15])
def test_other_depths(iif, oracle, bpc):
    rng = np.random.default_rng(bpc)
    w, h = 200, 70
    frames = rng.integers(0, 1 << bpc, size=(6, h, w)).astype(np.uint16)
    want = oracle.motion_v2_sequence(frames, bpc)
    assert np.array_equal(run_v2(iif, padded_dev(frames), w, h, bpc, 4), want)
    assert np.array_equal(run_v2(iif, to_dev(frames), w, h, bpc, 6), want)


def test_long_batch_many_chunks(iif, oracle):
    """200 frames of a small frame in one launch: few tiles, so the launch is
    split into frame chunks, each re-deriving its warm-up frame's sums."""
    frames = synth.smooth_sequence(77, 200, 130, 36, 2)
    want = oracle.motion_v2_sequence(frames, 8)
    assert np.array_equal(run_v2(iif, padded_dev(frames), 130, 36, 8, 200), want)
    assert np.array_equal(run_v2(iif, padded_dev(frames), 130, 36, 8, 37), want)
