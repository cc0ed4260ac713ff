"""The bounds-checked build on the GPU: the motion kernels compiled with
MG_BOUNDS_CHECK=1 check every shared- and global-memory access against its
buffer (a failed check skips the access and sets bit 1 of the device error
word).  A child process loads that library and runs the cases of
tests/bounds_checked_cases.py -- both kernel paths, odd, ragged and padded
frames, 8/10/16 bits, motion, motion_v2 and the fused 4:2:0 form, each over
two calls, the allocation-free entry point and a launch whose tail is split --
and every result must match the oracle with the error word 0.
This is the memory checker the tests use in place of a sanitizer."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bounds_checked_kernels_match_the_oracle():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from integer_image_filter_gb300 import _build
    _build.build(checked=True)
    r = subprocess.run([sys.executable, "-m", "tests.bounds_checked_cases"], cwd=ROOT,
                       capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stderr[-3000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    from tests import bounds_checked_cases as bc
    assert res["cases"] == (3 * len(bc.SIZES) * 3 * 2 * 2 + 2 * len(bc.FUSED_SIZES) * 2 * 2 +
                            len(bc.NOALLOC_SIZES) * 2 * 2 + len(bc.SPLIT_SIZES) * 2), res["cases"]
    assert res["n_failures"] == 0, res["failures"]
