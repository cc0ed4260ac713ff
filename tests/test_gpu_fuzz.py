"""Seeded fuzz parity through the raw C ABI (cases in tests/fuzz_cases.py):
kind, frame size from 3x3 up, bit depth 8..16, padded rows, base offset, the
cut points that split the frames over consecutive calls and the kernel path
are drawn per case; every result equals the oracle's.  The same cases of the
instrumented kernels also run against the bounds-checked library, where every
shared- and global-memory access is checked against its buffer."""
import json
import os
import subprocess
import sys

import pytest

from tests import fuzz_cases as fc

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


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


def test_fuzz_cases_on_the_bounds_checked_library(iif):
    from integer_image_filter_gb300 import _build
    _build.build(checked=True)
    r = subprocess.run([sys.executable, "-m", "tests.fuzz_cases", "checked"], cwd=ROOT,
                       capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stderr[-3000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["cases"] == sum(fc.draw(i)["kind"] in fc.CHECKED_KINDS for i in range(fc.N_CASES))
    assert res["n_failures"] == 0, res["failures"]


@pytest.mark.parametrize("i", range(fc.N_ALL))
def test_fuzz_case(iif, oracle, i):
    fc.run_case(iif, oracle, i)
