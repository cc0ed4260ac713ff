"""Independent contexts on independent CUDA streams: several sequences (motion,
motion_v2 and fused 4:2:0, aligned and odd layouts) submitted batch by batch
in interleaved order, each context on its own stream, all in flight at once;
every sequence equals the oracle's."""
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


def test_interleaved_contexts_on_their_own_streams(iif, oracle):
    import torch
    jobs = []
    specs = [("motion", 640, 160, 8), ("motion", 213, 70, 10), ("motion_v2", 384, 96, 8),
             ("motion_v2", 203, 67, 16), ("motion", 1920, 1080, 8)]
    for i, (kind, w, h, bpc) in enumerate(specs):
        fr = synth.uniform_frames(100 + i, 12, w, h, bpc)
        d = torch.from_numpy(fr.view(np.int16) if bpc > 8 else fr).cuda()
        want = (oracle.motion_v2_sequence(fr, bpc).astype(np.uint64) if kind == "motion_v2"
                else oracle_sad(oracle, fr, bpc))
        jobs.append({"kind": kind, "ctx": iif.MotionContext(w, h, bpc), "d": d, "want": want,
                     "out": torch.zeros(12, dtype=torch.int64, device="cuda"), "s": torch.cuda.Stream()})
    b = synth.yuv420_pairs(7, 8, 256, 96, max_shift=2, dist_sigma=3.0)
    planes = [torch.from_numpy(p).cuda() for p in b.planes()]
    fused = {"ctx": iif.MotionContext(256, 96, 8), "s": torch.cuda.Stream(),
             "sad": torch.zeros(8, dtype=torch.int64, device="cuda"),
             "sse": torch.zeros((8, 3), dtype=torch.int64, device="cuda")}
    torch.cuda.synchronize()
    for b0 in range(0, 12, 3):                   # batches of 3, interleaved across contexts
        for j in jobs:
            sub = j["ctx"].submit_batch_v2 if j["kind"] == "motion_v2" else j["ctx"].submit_batch
            sub(j["d"][b0:b0 + 3], j["out"][b0:b0 + 3], stream=j["s"])
        if b0 < 8:
            e = min(b0 + 3, 8)
            fused["ctx"].yuv420_batch(*[p[b0:e] for p in planes], fused["sad"][b0:e],
                                      fused["sse"][b0:e], stream=fused["s"])
    torch.cuda.synchronize()
    for j in jobs:
        assert j["ctx"].device_error() == 0
        assert j["out"].cpu().numpy().astype(np.uint64).tolist() == j["want"].tolist(), (j["kind"],)
        j["ctx"].close()
    assert fused["sad"].cpu().numpy().astype(np.uint64).tolist() == oracle_sad(oracle, b.ref_y, 8).tolist()
    assert np.array_equal(fused["sse"].cpu().numpy().astype(np.uint64), oracle_sse420(oracle, b))
    fused["ctx"].close()
