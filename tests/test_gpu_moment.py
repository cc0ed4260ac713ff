"""Moment sums (sum ref, sum dist, sum ref^2, sum dist^2 of each pair's luma) on
the GPU against the CPU oracle, bit for bit, through the C ABI: the 4K 4:2:0
workload's luma pairs and the 10-bit sequence at full size, every depth,
ragged and tiny planes, unaligned layouts (the sample-by-sample path), the
16-bit closed form at a large size, and error returns."""
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


def oracle_moments(o, ref, dist, bpc):
    def run(i):
        return o.moment_sums(ref[i], dist[i], bpc)
    with ThreadPoolExecutor(16) as ex:
        rows = list(ex.map(run, range(ref.shape[0])))
    return np.array(rows, dtype=np.uint64).reshape(-1, 4)


def gpu_moments(iif, ref_dev, dist_dev, bpc, **kw):
    import torch
    n = ref_dev.shape[0]
    out = dev_zeros((n, 4))
    iif.moment_sums_batch(ref_dev, dist_dev, bpc, out, **kw)
    torch.cuda.synchronize()
    return to_u64(out)


def test_yuv420_4k_luma_pairs(iif, oracle):
    b = synth.make("yuv420_3840x2160_u8_pairs")
    got = gpu_moments(iif, to_dev(b.ref_y), to_dev(b.dist_y), 8)
    want = oracle_moments(oracle, b.ref_y, b.dist_y, 8)
    assert np.array_equal(got, want)
    m = iif.moments_from_sums(got, 3840, 2160)
    assert np.array_equal(m, oracle.moments(want, 3840, 2160))


def test_10bit_4k_consecutive_frames(iif, oracle):
    f = synth.make("seq_3840x2160_u10", n=33)
    got = gpu_moments(iif, to_dev(f[:-1]), to_dev(f[1:]), 10)
    assert np.array_equal(got, oracle_moments(oracle, f[:-1], f[1:], 10))


@pytest.mark.parametrize("bpc", [8, 9, 10, 12, 15, 16])
@pytest.mark.parametrize("wh", [(1, 1), (3, 3), (17, 5), (64, 48), (1000, 3), (1921, 1081)])
def test_depths_and_sizes(iif, oracle, bpc, wh):
    w, h = wh
    rng = np.random.default_rng(w * 5 + h + bpc)
    dt = np.uint8 if bpc == 8 else np.uint16
    ref = rng.integers(0, 1 << bpc, size=(3, h, w)).astype(dt)
    dist = rng.integers(0, 1 << bpc, size=(3, h, w)).astype(dt)
    got = gpu_moments(iif, to_dev(ref), to_dev(dist), bpc)
    assert np.array_equal(got, oracle_moments(oracle, ref, dist, bpc)), (bpc, w, h)


@pytest.mark.parametrize("bpc", [8, 10])
def test_unaligned_layouts(iif, oracle, bpc):
    """Odd offsets and pitches take the sample-by-sample path; the result is the same."""
    w, h, n = 301, 47, 4
    rng = np.random.default_rng(bpc)
    dt = np.uint8 if bpc == 8 else np.uint16
    big = rng.integers(0, 1 << bpc, size=(2, n, h, w + 7)).astype(dt)
    dev = to_dev(big)
    ref, dist = dev[0][:, :, 1:1 + w], dev[1][:, :, 3:3 + w]
    pitch, stride = (w + 7) * big.itemsize, h * (w + 7) * big.itemsize
    got = gpu_moments(iif, ref, dist, bpc, pitch=pitch, stride=stride)
    want = oracle_moments(oracle, np.ascontiguousarray(big[0][:, :, 1:1 + w]),
                          np.ascontiguousarray(big[1][:, :, 3:3 + w]), bpc)
    assert np.array_equal(got, want)


def test_16bit_closed_form_large(iif):
    """All samples 65535 (ref) and 1 (dist) at 8192 x 4320: sums c N and c^2 N."""
    import torch
    w, h = 8192, 4320
    ref = torch.full((1, h, w), -1, dtype=torch.int16, device="cuda")   # 0xffff
    dist = torch.full((1, h, w), 1, dtype=torch.int16, device="cuda")
    got = gpu_moments(iif, ref, dist, 16)
    n = w * h
    assert [int(x) for x in got[0]] == [65535 * n, n, 65535 * 65535 * n, n]


def test_errors_and_empty(iif):
    import torch
    a = torch.zeros((2, 8, 8), dtype=torch.uint8, device="cuda")
    out = dev_zeros((2, 4))
    with pytest.raises(iif.MotionError):
        iif.moment_sums_batch(a, a, 7, out)
    with pytest.raises(iif.MotionError):
        iif.moment_sums_batch(a, a, 8, out, w=0, h=8)
    with pytest.raises(iif.MotionError):
        iif.moment_sums_batch(a, a, 8, out, pitch=4)     # pitch < w
    iif.moment_sums_batch(a, a, 8, out, n=0)             # no-op
    torch.cuda.synchronize()
    assert int(out.abs().sum()) == 0
