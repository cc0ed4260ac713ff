"""CUDA graph capture of the batched entry points: a step made of a reset and
several batched calls (motion, motion_v2, the fused 4:2:0 form, the
stand-alone SSE and the moment sums) is captured once and replayed; every
replay gives the oracle's results bit for bit, and a direct call after a
replay continues the sequence from the replay's last frame.  The calls
enqueue only stream work, so the graph holds all of it."""
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


def _capture(step):
    """Capture step() into a CUDA graph (after one direct run on a side stream,
    as CUDA graph capture wants)."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("bpc", [8, 10])
def test_motion_and_v2_steps_replay(iif, oracle, bpc):
    import torch
    w, h, n, batch = 200, 100, 14, 4
    rng = np.random.default_rng(77 + bpc)
    dt = np.uint8 if bpc == 8 else np.uint16
    fr = rng.integers(0, 1 << bpc, size=(n + 1, h, w)).astype(dt)
    d = torch.from_numpy(fr.view(np.int16) if bpc > 8 else fr).cuda()
    sad = torch.zeros(n, dtype=torch.int64, device="cuda")
    sad2 = torch.zeros(n, dtype=torch.int64, device="cuda")
    want = oracle_sad(oracle, fr[:n], bpc)
    want2 = oracle.motion_v2_sequence(fr[:n], bpc).astype(np.uint64)
    with iif.MotionContext(w, h, bpc) as ctx:
        def step():
            s = torch.cuda.current_stream()
            ctx.reset()
            for b in range(0, n, batch):
                e = min(b + batch, n)
                ctx.submit_batch(d[b:e], sad[b:e], stream=s)
                ctx.submit_batch_v2(d[b:e], sad2[b:e], stream=s)
        g = _capture(step)
        for _ in range(3):
            sad.zero_()
            sad2.zero_()
            g.replay()
            torch.cuda.synchronize()
            assert sad.cpu().numpy().astype(np.uint64).tolist() == want.tolist()
            assert sad2.cpu().numpy().astype(np.uint64).tolist() == want2.tolist()
        # a direct call after the replay continues from its last frame
        one = torch.zeros(1, dtype=torch.int64, device="cuda")
        ctx.submit_batch(d[n:n + 1], one)
        torch.cuda.synchronize()
        assert int(one.item()) == int(oracle.motion_sad_sequence(fr[n - 1:n + 1], bpc)[1])
        assert ctx.device_error() == 0


def test_unaligned_step_replays(iif, oracle):
    """Frames of an odd width packed row after row take the copy kernel and
    then the TMA kernel; after one direct step (which allocates the copy's
    scratch) the captured step replays bit-exact."""
    import torch
    w, h, n = 213, 40, 6
    fr = synth.uniform_frames(5, n, w, h, 8)
    d = torch.from_numpy(fr).cuda()          # rows 213 bytes apart
    sad = torch.zeros(n, dtype=torch.int64, device="cuda")
    want = oracle.motion_sad_sequence(fr, 8).astype(np.uint64)
    with iif.MotionContext(w, h, 8) as ctx:
        def step():
            ctx.reset()
            ctx.submit_batch(d, sad, stream=torch.cuda.current_stream())
        g = _capture(step)
        for _ in range(2):
            sad.zero_()
            g.replay()
            torch.cuda.synchronize()
            assert sad.cpu().numpy().astype(np.uint64).tolist() == want.tolist()
        assert ctx.device_error() == 0


def test_sse_and_moment_steps_replay(iif, oracle):
    import torch
    b = synth.yuv420_pairs(12, 4, 192, 80, max_shift=2, dist_sigma=3.0)
    planes = [torch.from_numpy(p).cuda() for p in b.planes()]
    sse = torch.zeros((b.n, 3), dtype=torch.int64, device="cuda")
    mom = torch.zeros((b.n, 4), dtype=torch.int64, device="cuda")
    ry, dy = planes[0], planes[3]

    def step():
        s = torch.cuda.current_stream()
        iif.psnr_sse_yuv420_batch(192, 80, 8, *planes, sse, stream=s)
        iif.moment_sums_batch(ry, dy, 8, mom, stream=s)

    g = _capture(step)
    want_sse = oracle_sse420(oracle, b)
    want_mom = np.array([oracle.moment_sums(b.ref_y[i], b.dist_y[i], 8) for i in range(b.n)],
                        dtype=np.uint64)
    for _ in range(2):
        sse.zero_()
        mom.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(sse.cpu().numpy().astype(np.uint64), want_sse)
        assert np.array_equal(mom.cpu().numpy().astype(np.uint64), want_mom)


def test_fused_step_replays(iif, oracle):
    import torch
    b = synth.yuv420_pairs(9, 6, 256, 96, max_shift=2, dist_sigma=3.0)
    planes = [torch.from_numpy(p).cuda() for p in b.planes()]
    sad = torch.zeros(b.n, dtype=torch.int64, device="cuda")
    sse = torch.zeros((b.n, 3), dtype=torch.int64, device="cuda")
    want_sad = oracle_sad(oracle, b.ref_y, 8)
    want_sse = oracle_sse420(oracle, b)
    with iif.MotionContext(256, 96, 8) as ctx:
        def step():
            ctx.reset()
            ctx.yuv420_batch(*planes, sad, sse, stream=torch.cuda.current_stream())
        g = _capture(step)
        for _ in range(2):
            sad.zero_()
            sse.zero_()
            g.replay()
            torch.cuda.synchronize()
            assert np.array_equal(sad.cpu().numpy().astype(np.uint64), want_sad)
            assert np.array_equal(sse.cpu().numpy().astype(np.uint64), want_sse)
        assert ctx.device_error() == 0
