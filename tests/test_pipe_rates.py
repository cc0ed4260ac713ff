"""The machine-measurement library (libpipe_rates_gb300.so) behind the integer
co-bound and the HBM stream ceilings of the benchmark line: it builds for
sm_103a and exports its entry points (CPU); on a GPU the instruction classes
measure near their pipes' rates and the HBM streams at plausible rates."""
import ctypes

import pytest


@pytest.fixture(scope="module")
def plib():
    from integer_image_filter_gb300 import _build
    lib = ctypes.CDLL(_build.build_pipe_rates())
    lib.pipe_rates_name.restype = ctypes.c_char_p
    lib.hbm_stream_gbs.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_double)]
    return lib


def test_exports(plib):
    n = plib.pipe_rates_count()
    assert n == 13
    names = [plib.pipe_rates_name(i).decode() for i in range(n)]
    assert names[0].startswith("IMAD") and "dp2a" in names[1] and names[-1] == "LDS.128"
    assert plib.pipe_rates_name(n) == b"" and plib.pipe_rates_name(-1) == b""
    g = ctypes.c_double()
    assert plib.hbm_stream_gbs(3, ctypes.byref(g)) == 1      # no such stream kind
    assert plib.hbm_stream_gbs(-1, ctypes.byref(g)) == 1


@pytest.mark.gpu
def test_rates_on_the_device(plib):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    n = plib.pipe_rates_count()
    out = (ctypes.c_double * n)()
    assert plib.pipe_rates_measure(out) == 0
    rates = {plib.pipe_rates_name(i).decode(): out[i] for i in range(n)}
    # integer classes: 64 lane-operations per SM clock on GB300; a loose band
    for k in ("IMAD", "IDP.2A (dp2a)", "IADD3", "PRMT", "VABSDIFF (sad)"):
        assert 16.0 < rates[k] < 160.0, (k, rates[k])
    for kind in (0, 1, 2):
        g = ctypes.c_double()
        assert plib.hbm_stream_gbs(kind, ctypes.byref(g)) == 0
        assert 500.0 < g.value < 20000.0, (kind, g.value)
