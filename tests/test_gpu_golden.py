"""The stored expected values (tests/golden) on the GPU, through the C ABI:
the hand-worked 6x6 example (SAD and score) on both kernel paths, and the
oracle's stored results on seeded inputs in the shapes of the five workloads
-- motion, motion_v2, the fused 4:2:0 pass and the moment sums."""
import numpy as np
import pytest

from tests.golden import case_inputs, hand_worked_cases, impulse_frames, oracle_cases
from tests.gpu_util import to_dev

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


def _padded(a):
    """The same frames with 16-byte row pitch (the TMA path takes them)."""
    n, h, w = a.shape
    wp = (w * a.itemsize + 15) // 16 * 16 // a.itemsize
    big = np.zeros((n, h, wp), a.dtype)
    big[:, :, :w] = a
    return to_dev(big)[:, :, :w]


@pytest.mark.parametrize("case", hand_worked_cases(), ids=lambda c: c["name"])
@pytest.mark.parametrize("padded", [False, True])
@pytest.mark.parametrize("rows", [16, 32])
def test_hand_worked_on_gpu(iif, case, padded, rows):
    """The hand-worked values on the TMA kernel with 128 x 16 and 128 x 32
    tiles, from padded rows and from packed 6-sample rows (copied into aligned
    rows first)."""
    import torch
    fr = impulse_frames(case)
    d = _padded(fr) if padded else to_dev(fr)
    out = torch.zeros(2, dtype=torch.int64, device="cuda")
    with iif.MotionContext(6, 6, 8) as ctx:
        ctx.set_kernel_path(iif.MOTION_PATH_TMA_16 if rows == 16 else iif.MOTION_PATH_TMA_32)
        ctx.submit_batch(d, out)
        torch.cuda.synchronize()
        assert ctx.device_error() == 0
    sad = out.cpu().numpy().astype(np.uint64)
    assert sad.tolist() == [0, case["sad"]]
    score, _ = iif.motion_scores_from_sad(sad, 6, 6)
    assert score[1] == case["score"]


@pytest.mark.parametrize("case", oracle_cases(),
                         ids=lambda c: "%s-%dx%d-%dbit" % (c["kind"], c["w"], c["h"], c["bpc"]))
def test_library_reproduces_stored_values(iif, case):
    import torch
    kind, n, w, h, bpc = case["kind"], case["n"], case["w"], case["h"], case["bpc"]
    data = case_inputs(kind, case["seed"], n, w, h, bpc)
    if kind in ("motion", "motion_v2"):
        out = torch.zeros(n, dtype=torch.int64, device="cuda")
        with iif.MotionContext(w, h, bpc) as ctx:
            (ctx.submit_batch_v2 if kind == "motion_v2" else ctx.submit_batch)(to_dev(data), out)
            torch.cuda.synchronize()
            assert ctx.device_error() == 0
        assert out.cpu().numpy().astype(np.uint64).tolist() == case["sad"]
    elif kind == "yuv420":
        sad = torch.zeros(n, dtype=torch.int64, device="cuda")
        sse = torch.zeros((n, 3), dtype=torch.int64, device="cuda")
        with iif.MotionContext(w, h, bpc) as ctx:
            ctx.yuv420_batch(*[to_dev(p) for p in data.planes()], sad, sse)
            torch.cuda.synchronize()
            assert ctx.device_error() == 0
        assert sad.cpu().numpy().astype(np.uint64).tolist() == case["sad"]
        assert sse.cpu().numpy().astype(np.uint64).tolist() == case["sse"]
    else:
        out = torch.zeros((n, 4), dtype=torch.int64, device="cuda")
        iif.moment_sums_batch(to_dev(data.ref_y), to_dev(data.dist_y), bpc, out)
        torch.cuda.synchronize()
        assert out.cpu().numpy().astype(np.uint64).tolist() == case["sums"]
