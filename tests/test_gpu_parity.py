"""GPU path against the CPU oracle, bit for bit (integer SAD / SSE) and
exactly equal double scores, through the C ABI.  Covers the five workloads at
their full sizes, tiny and ragged frames, pitches and alignments, batch
continuity and error returns."""
import numpy as np
import pytest

import synth
from tests.gpu_util import dev_zeros, oracle_sad, oracle_sse420, to_dev, to_u64

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


def padded_dev(frames, align_bytes=16):
    """Device copy whose row pitch is rounded up to align_bytes (a view of the
    first w samples of each row), so that 16-byte-aligned layouts reach the
    TMA kernel whatever the width."""
    n, h, w = frames.shape
    s = frames.itemsize
    wp = ((w * s + align_bytes - 1) // align_bytes * align_bytes) // s
    big = np.zeros((n, h, wp), dtype=frames.dtype)
    big[:, :, :w] = frames
    return to_dev(big)[:, :, :w]


def run_batches(iif, frames, bpc, batch, path=None, padded=False):
    import torch
    n, h, w = frames.shape
    d = padded_dev(frames) if padded else to_dev(frames)
    out = dev_zeros(n)
    with iif.MotionContext(w, h, bpc) as ctx:
        if path is not None:
            ctx.set_kernel_path(path)
        for s in range(0, n, batch):
            e = min(n, s + batch)
            ctx.submit_batch(d[s:e], out[s:e])
        torch.cuda.synchronize()
        assert ctx.device_error() == 0
    return to_u64(out)


# --------------------------------------------------------------- the workloads
def test_pair_64x48_u8(iif, oracle):
    frames = synth.make("pair_64x48_u8")
    want = oracle.motion_sad_sequence(frames, 8)
    d = to_dev(frames)
    with iif.MotionContext(64, 48, 8) as ctx:
        sad0, s0 = ctx.submit(d[0])
        sad1, s1 = ctx.submit(d[1])
    assert (sad0, sad1) == (0, int(want[1]))
    score, _ = oracle.scores(want, 64, 48)
    assert s0 == 0.0 and s1 == score[1]
    assert np.array_equal(run_batches(iif, frames, 8, 2), want)


def test_seq_576x324_single_submits_and_scores(iif, oracle):
    frames = synth.make("seq_576x324_u8")
    want = oracle_sad(oracle, frames, 8)
    d = to_dev(frames)
    got, scores = [], []
    with iif.MotionContext(576, 324, 8) as ctx:
        for i in range(frames.shape[0]):
            s, sc = ctx.submit(d[i])
            got.append(s)
            scores.append(sc)
    assert np.array_equal(np.array(got, np.uint64), want)
    ws, wm2 = oracle.scores(want, 576, 324)
    assert np.array_equal(np.array(scores), ws)
    gs, gm2 = iif.motion_scores_from_sad(np.array(got, np.uint64), 576, 324)
    assert np.array_equal(gs, ws) and np.array_equal(gm2, wm2)
    assert np.array_equal(run_batches(iif, frames, 8, 48), want)


def test_seq_1920x1080_cuts_batch16(iif, oracle):
    frames = synth.make("seq_1920x1080_u8_cuts")
    want = oracle_sad(oracle, frames, 8)
    assert np.array_equal(run_batches(iif, frames, 8, 16), want)
    assert np.array_equal(run_batches(iif, frames[:40], 8, 16, path=iif.MOTION_PATH_GENERIC),
                          want[:40])


def test_yuv420_4k_fused_full(iif, oracle):
    import torch
    b = synth.make("yuv420_3840x2160_u8_pairs")
    want_sad = oracle_sad(oracle, b.ref_y, 8)
    want_sse = oracle_sse420(oracle, b)
    planes = [to_dev(p) for p in b.planes()]
    sad, sse = dev_zeros(b.n), dev_zeros((b.n, 3))
    with iif.MotionContext(b.w, b.h, 8) as ctx:
        ctx.yuv420_batch(*planes, sad, sse)
        torch.cuda.synchronize()
    assert np.array_equal(to_u64(sad), want_sad)
    assert np.array_equal(to_u64(sse), want_sse)
    # the stand-alone SSE launch over all planes and pairs
    sse2 = dev_zeros((b.n, 3))
    iif.psnr_sse_yuv420_batch(b.w, b.h, 8, *planes, sse2)
    torch.cuda.synchronize()
    assert np.array_equal(to_u64(sse2), want_sse)


def test_yuv420_4k_host_pipeline(iif, oracle):
    import torch
    b = synth.make("yuv420_3840x2160_u8_pairs", n=12)
    want_sad = oracle_sad(oracle, b.ref_y, 8)
    want_sse = oracle_sse420(oracle, b)
    pinned = [torch.from_numpy(p).pin_memory() for p in b.planes()]
    with iif.MotionContext(b.w, b.h, 8) as ctx:
        iif.motion_reserve_host_staging(ctx.handle, 5)        # 3 chunks, ragged last
        sad, sse = ctx.yuv420_batch_host(*pinned)
        assert np.array_equal(sad, want_sad) and np.array_equal(sse, want_sse)
        ctx.reset()
        sad, sse = ctx.yuv420_batch_host(*b.planes())          # pageable host memory
        assert np.array_equal(sad, want_sad) and np.array_equal(sse, want_sse)


def test_seq_4k_u10_batch32(iif, oracle):
    frames = synth.make("seq_3840x2160_u10")
    assert frames.max() <= 1023
    want = oracle_sad(oracle, frames, 10)
    assert np.array_equal(run_batches(iif, frames, 10, 32), want)


@pytest.mark.parametrize("batch", [1, 3, 7, 32])
def test_u10_batch_sizes_agree(iif, oracle, batch):
    frames = synth.make("seq_3840x2160_u10", n=9)
    want = oracle_sad(oracle, frames, 10)
    assert np.array_equal(run_batches(iif, frames, 10, batch), want)


@pytest.mark.parametrize("bpc", [8, 10])
def test_split_tail_launch(iif, oracle, bpc):
    """A launch shape that splits its tail: 2560x1440 frames in batches of 8
    are 900 tiles, one full wave of 4 blocks per SM plus 292 tiles, which run
    in chunks of 4 frames after the whole tiles (the plan checked through
    motion_launch_blocks on this device's SM count); two calls of the sequence
    against the oracle, motion and motion_v2."""
    import torch
    w, h, n, batch = 2560, 1440, 16, 8
    slots = 4 * torch.cuda.get_device_properties(0).multi_processor_count
    tiles = (w // 128) * (h // 32)
    count, _ = iif.motion_launch_blocks(w, h, batch, slots)
    if iif.motion_plan_chunks(w, h, batch, slots) == 1 and tiles > slots and 0 < 2 * (tiles % slots) <= slots:
        assert count > tiles, "the launch splits its tail"
    frames = synth.uniform_frames(77 + bpc, n, w, h, bpc)
    want = oracle_sad(oracle, frames, bpc)
    assert np.array_equal(run_batches(iif, frames, bpc, batch), want)
    d = to_dev(frames)
    out = dev_zeros(n)
    with iif.MotionContext(w, h, bpc) as ctx:
        for s0 in range(0, n, batch):
            ctx.submit_batch_v2(d[s0:s0 + batch], out[s0:s0 + batch])
        torch.cuda.synchronize()
        assert ctx.device_error() == 0
    assert np.array_equal(to_u64(out), oracle.motion_v2_sequence(frames, bpc))


@pytest.mark.parametrize("bpc", [8, 10])
def test_short_and_full_tiles_agree(iif, oracle, bpc):
    """1080p frames in batches of 16 fit in one wave of 128 x 32 tiles, so
    they run 128 x 16 tiles; batches of 32 (three chunks) run 128 x 32.  The
    shape chosen is checked through motion_launch_shape on this device's SM
    count, and both tile heights, chosen or forced, equal the oracle, for
    motion and motion_v2 (ragged last tile row: 1080 = 67.5 x 16)."""
    import torch
    w, h, n = 1920, 1080, 32
    slots = 4 * torch.cuda.get_device_properties(0).multi_processor_count
    assert iif.motion_launch_shape(w, h, 16, slots) == 16
    assert iif.motion_launch_shape(w, h, 32, slots) == 32
    frames = synth.smooth_sequence(31 + bpc, n, w, h, 5, bpc=bpc)
    want = oracle_sad(oracle, frames, bpc)
    for batch, path in ((16, None), (32, None), (16, iif.MOTION_PATH_TMA_32), (32, iif.MOTION_PATH_TMA_16)):
        assert np.array_equal(run_batches(iif, frames, bpc, batch, path=path), want), (batch, path)
    want_v2 = oracle.motion_v2_sequence(frames, bpc)
    d = to_dev(frames)
    for path in (iif.MOTION_PATH_TMA_32, iif.MOTION_PATH_TMA_16):
        out = dev_zeros(n)
        with iif.MotionContext(w, h, bpc) as ctx:
            ctx.set_kernel_path(path)
            for s0 in range(0, n, 16):
                ctx.submit_batch_v2(d[s0:s0 + 16], out[s0:s0 + 16])
            torch.cuda.synchronize()
            assert ctx.device_error() == 0
        assert np.array_equal(to_u64(out), want_v2), path


@pytest.mark.parametrize("bpc", [8, 10])
def test_short_tiles_with_split_tail(iif, oracle, bpc):
    """1920x1280 in batches of 16: its 600 tiles of 128 x 32 fit in one wave,
    so it runs 1200 tiles of 128 x 16, more than the 1064 that are resident at
    once on GB300: the launch splits its tail (the 16-row plan checked through
    motion_launch_shape and motion_launch_blocks on this device's SM count).
    Two calls against the oracle, motion and motion_v2."""
    import torch
    w, h, n, batch = 1920, 1280, 32, 16
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert iif.motion_launch_shape(w, h, batch, 4 * sms) == 16
    tiles16 = (w // 128) * (h // 16)
    count, _ = iif.motion_launch_blocks(w, h, batch, 7 * sms, tile_rows=16)
    if tiles16 > 7 * sms and 0 < 2 * (tiles16 % (7 * sms)) <= 7 * sms:
        assert count > tiles16, "the 16-row launch splits its tail"
    frames = synth.uniform_frames(91 + bpc, n, w, h, bpc)
    want = oracle_sad(oracle, frames, bpc)
    assert np.array_equal(run_batches(iif, frames, bpc, batch), want)
    d = to_dev(frames)
    out = dev_zeros(n)
    with iif.MotionContext(w, h, bpc) as ctx:
        ctx.set_kernel_path(iif.MOTION_PATH_TMA_16)
        for s0 in range(0, n, batch):
            ctx.submit_batch_v2(d[s0:s0 + batch], out[s0:s0 + batch])
        torch.cuda.synchronize()
        assert ctx.device_error() == 0
    assert np.array_equal(to_u64(out), oracle.motion_v2_sequence(frames, bpc))


# --------------------------------------------------------------- shapes, layouts
SIZES = [(w, h) for w in (3, 4, 5, 7, 9) for h in (3, 4, 6, 9)] + [
    (16, 16), (17, 33), (67, 35), (127, 31), (128, 32), (129, 33), (131, 70), (160, 36),
    (255, 97), (300, 65), (513, 129),
    # full tiles on the left and right edges with all rows inside the frame: their
    # halo lanes read the mirrored columns (w - x0 = 128 and 129, one and several columns)
    (128, 100), (129, 100), (256, 70), (385, 98)]


@pytest.mark.parametrize("bpc", [8, 10, 16])
def test_tiny_and_ragged_frames(iif, oracle, bpc):
    rng = np.random.default_rng(bpc)
    for (w, h) in SIZES:
        frames = synth.uniform_frames(int(rng.integers(1 << 30)), 3, w, h, bpc)
        want = oracle.motion_sad_sequence(frames, bpc)
        got = run_batches(iif, frames, bpc, 3)
        assert np.array_equal(got, want), (w, h, bpc)


@pytest.mark.parametrize("bpc", [8, 10, 16])
def test_tma_and_generic_paths_on_aligned_layouts(iif, oracle, bpc):
    """16-byte-aligned pitches: the TMA kernel (mirrored reads on border tiles)
    with 128 x 32 and with 128 x 16 tiles, and the generic kernel (mirror
    applied at load), all equal the oracle."""
    rng = np.random.default_rng(100 + bpc)
    for (w, h) in SIZES:
        frames = synth.uniform_frames(int(rng.integers(1 << 30)), 4, w, h, bpc)
        want = oracle.motion_sad_sequence(frames, bpc)
        for path in (iif.MOTION_PATH_AUTO, iif.MOTION_PATH_GENERIC, iif.MOTION_PATH_TMA_32,
                     iif.MOTION_PATH_TMA_16):
            got = run_batches(iif, frames, bpc, 3, path=path, padded=True)
            assert np.array_equal(got, want), (w, h, bpc, path)


@pytest.mark.parametrize("bpc", [8, 10])
def test_fused_paths_on_aligned_layouts(iif, oracle, bpc):
    import torch
    for (w, h) in ((3, 3), (64, 48), (130, 66), (257, 131), (300, 97)):
        b = synth.yuv420_pairs(w * 3 + h, 5, w, h, bpc=bpc)
        want_sad = oracle.motion_sad_sequence(b.ref_y, bpc)
        want_sse = oracle_sse420(oracle, b)
        planes = [padded_dev(p) for p in b.planes()]
        for path in (iif.MOTION_PATH_AUTO, iif.MOTION_PATH_GENERIC):
            sad, sse = dev_zeros(5), dev_zeros((5, 3))
            with iif.MotionContext(w, h, bpc) as ctx:
                ctx.set_kernel_path(path)
                ctx.yuv420_batch(*planes, sad, sse)
                torch.cuda.synchronize()
                assert ctx.device_error() == 0
            assert np.array_equal(to_u64(sad), want_sad), (w, h, path)
            assert np.array_equal(to_u64(sse), want_sse), (w, h, path)


@pytest.mark.parametrize("bpc", [8, 10])
def test_pitch_and_misaligned_base(iif, oracle, bpc):
    import torch
    rng = np.random.default_rng(99)
    w, h, n = 301, 77, 4
    frames = synth.uniform_frames(7, n, w, h, bpc)
    want = oracle.motion_sad_sequence(frames, bpc)
    s = 1 if bpc == 8 else 2
    for off, extra in ((1, 3), (3, 16), (0, 5), (8, 0)):
        big = np.zeros((n, h, w + off + extra), dtype=frames.dtype)
        big[:, :, off:off + w] = frames
        d = to_dev(big)[:, :, off:off + w]                 # row pitch (w+off+extra)*s bytes
        out = dev_zeros(n)
        with iif.MotionContext(w, h, bpc) as ctx:
            ctx.submit_batch(d, out)
            torch.cuda.synchronize()
        assert np.array_equal(to_u64(out), want), (off, extra)
    # the fused pass on a layout that is not 16-byte aligned
    b = synth.yuv420_pairs(3, 3, 130, 66, bpc=bpc)
    off = 2 if bpc > 8 else 1
    views = []
    for p in b.planes():
        big = np.zeros((p.shape[0], p.shape[1], p.shape[2] + off + 1), dtype=p.dtype)
        big[:, :, off:off + p.shape[2]] = p
        views.append(to_dev(big)[:, :, off:off + p.shape[2]])
    sad, sse = dev_zeros(3), dev_zeros((3, 3))
    with iif.MotionContext(130, 66, bpc) as ctx:
        ctx.yuv420_batch(*views, sad, sse)
        torch.cuda.synchronize()
    assert np.array_equal(to_u64(sad), oracle.motion_sad_sequence(b.ref_y, bpc))
    assert np.array_equal(to_u64(sse), oracle_sse420(oracle, b))


@pytest.mark.parametrize("bpc", [8, 10, 12, 16])
@pytest.mark.parametrize("wh", [(1, 1), (3, 3), (17, 5), (64, 48), (1000, 3), (1921, 1081)])
def test_psnr_sse_single_plane(iif, oracle, bpc, wh):
    import torch
    w, h = wh
    rng = np.random.default_rng(w * 7 + h + bpc)
    hi = 1 << bpc
    dt = np.uint8 if bpc == 8 else np.uint16
    ref = rng.integers(0, hi, size=(h, w)).astype(dt)
    dist = rng.integers(0, hi, size=(h, w)).astype(dt)
    out = dev_zeros(1)
    iif.psnr_sse(to_dev(ref), to_dev(dist), bpc, out)
    torch.cuda.synchronize()
    assert int(out.cpu()[0]) == oracle.sse(ref, dist, bpc)


def test_yuv420_odd_sizes_all_depths(iif, oracle):
    import torch
    for (w, h, bpc) in ((3, 3, 8), (5, 7, 10), (127, 33, 8), (257, 131, 10), (66, 40, 16)):
        b = synth.yuv420_pairs(w + h, 4, w, h, bpc=bpc)
        planes = [to_dev(p) for p in b.planes()]
        sad, sse = dev_zeros(4), dev_zeros((4, 3))
        with iif.MotionContext(w, h, bpc) as ctx:
            ctx.yuv420_batch(*planes, sad, sse)
            torch.cuda.synchronize()
        assert np.array_equal(to_u64(sad), oracle.motion_sad_sequence(b.ref_y, bpc)), (w, h)
        assert np.array_equal(to_u64(sse), oracle_sse420(oracle, b)), (w, h)
        sse2 = dev_zeros((4, 3))
        iif.psnr_sse_yuv420_batch(w, h, bpc, *planes, sse2)
        torch.cuda.synchronize()
        assert np.array_equal(to_u64(sse2), oracle_sse420(oracle, b)), (w, h)


# --------------------------------------------------------------- properties at any size
def test_constant_frames_closed_form_max_size(iif):
    """Two constant frames: SAD = |c1 - c2| 2^(16-bpc) w h at the largest size."""
    import torch
    w, h = 8192, 4320
    for bpc, c1, c2 in ((8, 17, 250), (10, 1023, 0)):
        dt = torch.uint8 if bpc == 8 else torch.int16
        d = torch.empty((2, h, w), dtype=dt, device="cuda")
        d[0].fill_(c1)
        d[1].fill_(c2)
        out = dev_zeros(2)
        with iif.MotionContext(w, h, bpc) as ctx:
            ctx.submit_batch(d, out)
            torch.cuda.synchronize()
        assert to_u64(out).tolist() == [0, abs(c1 - c2) * (1 << (16 - bpc)) * w * h]


def test_large_frame_against_oracle(iif, oracle):
    frames = synth.smooth_sequence(11, 2, 8192, 4320, 4)
    assert np.array_equal(run_batches(iif, frames, 8, 2), oracle.motion_sad_sequence(frames, 8))


def test_symmetry_and_identity_on_gpu(iif):
    """SAD(a, b) == SAD(b, a) and SAD(a, a) == 0 for a 4K pair (no oracle)."""
    frames = synth.make("yuv420_3840x2160_u8_pairs", n=2).ref_y
    seq = np.stack([frames[0], frames[1], frames[0], frames[0]])
    got = run_batches(iif, seq, 8, 4)
    assert got[1] == got[2] and got[3] == 0 and got[1] > 0


# --------------------------------------------------------------- sequence state
def test_long_batches_many_chunks(iif, oracle):
    """200 frames of a small frame per launch: the launch splits the frames
    into chunks (each after the first re-blurs a warm-up frame), continuing
    the sequence across launches of 37 frames as well."""
    frames = synth.smooth_sequence(78, 200, 130, 36, 2)
    want = oracle.motion_sad_sequence(frames, 8)
    for batch in (200, 37):
        assert np.array_equal(run_batches(iif, frames, 8, batch, padded=True), want), batch


def test_batch_continuity_and_reset(iif, oracle):
    import torch
    frames = synth.make("seq_576x324_u8", n=16)
    want = oracle.motion_sad_sequence(frames, 8)
    d = to_dev(frames)
    out = dev_zeros(16)
    with iif.MotionContext(576, 324, 8) as ctx:
        for s, e in ((0, 1), (1, 4), (4, 11), (11, 16)):
            ctx.submit_batch(d[s:e], out[s:e])
        torch.cuda.synchronize()
        assert np.array_equal(to_u64(out), want)
        ctx.reset()
        out2 = dev_zeros(8)
        ctx.submit_batch(d[8:16], out2)
        torch.cuda.synchronize()
        w2 = oracle.motion_sad_sequence(frames[8:16], 8)
        assert np.array_equal(to_u64(out2), w2)
        # an empty batch is a no-op and keeps the sequence
        ctx.submit_batch(d[0:0], out2[0:0])
        s, _ = ctx.submit(d[0])
        assert s == oracle.motion_sad_sequence(np.stack([frames[15], frames[0]]), 8)[1]


def test_error_returns(iif):
    import torch
    d = torch.zeros((2, 48, 64), dtype=torch.uint8, device="cuda")
    out = dev_zeros(2)
    with iif.MotionContext(64, 48, 8) as ctx:
        with pytest.raises(iif.MotionError) as e:
            iif.motion_submit_batch(ctx.handle, d, out, pitch_bytes=32)
        assert e.value.code == 4
        with pytest.raises(iif.MotionError) as e:
            iif.motion_submit_batch(ctx.handle, d, out, n=-1)
        assert e.value.code == 1
        with pytest.raises(iif.MotionError):
            iif.motion_submit_batch(ctx.handle, 0, out, n=2, frame_stride=3072, pitch_bytes=64)
    with iif.MotionContext(64, 48, 10) as ctx:
        d16 = torch.zeros((2, 48, 65), dtype=torch.int16, device="cuda")
        with pytest.raises(iif.MotionError) as e:   # odd byte offset for uint16 samples
            iif.motion_submit_batch(ctx.handle, d16.data_ptr() + 1, out, n=2,
                                    frame_stride=48 * 130, pitch_bytes=130)
        assert e.value.code == 4
