"""Contexts driven from several host threads at once, from the first library
call of a fresh process on: ten threads (motion, motion_v2 and fused 4:2:0 on
device buffers, both host-buffer pipelines, the moment sums; 8 to 12 bits;
aligned and odd layouts), each with its own context and CUDA stream, start
together behind a barrier (tests/threaded_contexts.py runs them in a child
interpreter).  Every result equals the oracle's and no context records a
device error."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

from tests import threaded_contexts as tc
from tests.gpu_util import oracle_sad

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from integer_image_filter_gb300 import _build
    _build.build()


def expected(o, job) -> dict:
    kind, seed, n, w, h, bpc = job
    data = tc.inputs(*job)
    if kind == "moments":
        return {"sums": [[int(v) for v in o.moment_sums(data.ref_y[i], data.dist_y[i], bpc)]
                         for i in range(n)]}
    if kind == "motion_v2":
        return {"sad": [int(v) for v in o.motion_v2_sequence(data, bpc)]}
    if kind in ("yuv420", "yuv420_host"):
        sse = [[int(o.sse(data.ref_y[i], data.dist_y[i], bpc)), int(o.sse(data.ref_u[i], data.dist_u[i], bpc)),
                int(o.sse(data.ref_v[i], data.dist_v[i], bpc))] for i in range(n)]
        return {"sad": [int(v) for v in oracle_sad(o, data.ref_y, bpc)], "sse": sse}
    return {"sad": [int(v) for v in oracle_sad(o, data, bpc)]}


def test_contexts_on_concurrent_host_threads(built, oracle, tmp_path):
    path = tmp_path / "threads.json"
    r = subprocess.run([sys.executable, "-m", "tests.threaded_contexts", str(path)], cwd=ROOT,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    with open(path) as f:
        got = json.load(f)
    assert got["errors"] == []
    for job, res in zip(tc.JOBS, got["results"]):
        want = expected(oracle, job)
        assert res.get("device_error", 0) == 0, job
        for key, v in want.items():
            assert res[key] == v, (job, key)
