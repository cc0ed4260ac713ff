"""The stored expected values (tests/golden) on the CPU: the hand-worked 6x6
example against its closed form and against the oracle, and the oracle
against the values it wrote earlier (a regression pin: a change to the
oracle's arithmetic shows here first)."""
import numpy as np
import pytest

from tests.golden import case_inputs, hand_worked_cases, impulse_frames, oracle_cases

TAPS = (3571, 16004, 26386, 16004, 3571)


def _folded(n, at):
    # the taps of each output index that land on input index `at` through the mirror
    def m(i):
        return -i if i < 0 else (2 * n - i - 2 if i >= n else i)
    return np.array([sum(t for k, t in enumerate(TAPS) if m(i + k - 2) == at) for i in range(n)],
                    dtype=np.int64)


@pytest.mark.parametrize("case", hand_worked_cases(), ids=lambda c: c["name"])
def test_hand_worked_closed_form(case):
    r, c, v = case["impulse"]
    b = (np.outer((v * _folded(6, r) + 128) >> 8, _folded(6, c)) + 32768) >> 16
    if case["B"] is not None:
        assert np.array_equal(b, case["B"])
    assert int(b.sum()) == case["sad"]                 # the previous frame is zero
    assert (case["sad"] / 256.0) / 36.0 == case["score"]


@pytest.mark.parametrize("case", hand_worked_cases(), ids=lambda c: c["name"])
def test_hand_worked_oracle(oracle, case):
    fr = impulse_frames(case)
    if case["B"] is not None:
        assert np.array_equal(oracle.blur(fr[1], 8).astype(np.int64), case["B"])
    sad = oracle.motion_sad_sequence(fr, 8)
    assert [int(x) for x in sad] == [0, case["sad"]]
    score, _ = oracle.scores(np.asarray(sad, np.uint64), 6, 6)
    assert score[1] == case["score"]


@pytest.mark.parametrize("case", oracle_cases(),
                         ids=lambda c: "%s-%dx%d-%dbit" % (c["kind"], c["w"], c["h"], c["bpc"]))
def test_oracle_reproduces_its_stored_values(oracle, case):
    data = case_inputs(case["kind"], case["seed"], case["n"], case["w"], case["h"], case["bpc"])
    bpc = case["bpc"]
    if case["kind"] == "motion":
        assert [int(x) for x in oracle.motion_sad_sequence(data, bpc)] == case["sad"]
    elif case["kind"] == "motion_v2":
        assert [int(x) for x in oracle.motion_v2_sequence(data, bpc)] == case["sad"]
    elif case["kind"] == "yuv420":
        assert [int(x) for x in oracle.motion_sad_sequence(data.ref_y, bpc)] == case["sad"]
        sse = [[oracle.sse(data.ref_y[i], data.dist_y[i], bpc), oracle.sse(data.ref_u[i], data.dist_u[i], bpc),
                oracle.sse(data.ref_v[i], data.dist_v[i], bpc)] for i in range(data.n)]
        assert sse == case["sse"]
    else:
        sums = [[int(x) for x in oracle.moment_sums(data.ref_y[i], data.dist_y[i], bpc)] for i in range(data.n)]
        assert sums == case["sums"]
