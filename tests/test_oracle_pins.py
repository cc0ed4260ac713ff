"""The CPU oracle checked against closed forms, library routines, a hand-worked
example, brute force and invariants (no GPU).  Every planted mistake in the
oracle must be caught by at least one pin."""
import os

import numpy as np
import pytest

import oracle as oracle_pkg
from tests import pins

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin_holds(oracle, pin):
    pin(oracle)


PLANTS = ["ORACLE_PLANT_MIRROR_REPEAT", "ORACLE_PLANT_NO_VROUND", "ORACLE_PLANT_VSHIFT8",
          "ORACLE_PLANT_SWAP_MIRROR_N", "ORACLE_PLANT_NO_HROUND", "ORACLE_PLANT_HFIRST",
          "ORACLE_PLANT_MOMENT_SKIP_LAST_ROW", "ORACLE_PLANT_MOMENT_SQUARE_OF_REF",
          "ORACLE_PLANT_V2_TRUNCATE", "ORACLE_PLANT_V2_CUR_MINUS_PREV"]


@pytest.mark.parametrize("plant", PLANTS)
def test_planted_mistake_is_caught(tmp_path, plant):
    so = oracle_pkg.build(defines=(plant,), out_path=str(tmp_path / f"lib_{plant}.so"))
    planted = oracle_pkg.Oracle(oracle_pkg.load(so))
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(planted)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin catches {plant}"


def test_oracle_rejects_bad_sizes(oracle):
    with pytest.raises(ValueError):
        oracle.blur(np.zeros((2, 5), np.uint8), 8)
    with pytest.raises(ValueError):
        oracle.blur(np.zeros((5, 2), np.uint8), 8)
    with pytest.raises(TypeError):
        oracle.blur(np.zeros((5, 5), np.uint16), 8)
    assert oracle.motion_sad_sequence(np.zeros((0, 4, 4), np.uint8), 8).size == 0


def test_oracle_respects_pitch(oracle):
    rng = np.random.default_rng(3)
    big = rng.integers(0, 1024, size=(9, 40)).astype(np.uint16)
    view = big[:, 5:26]          # non-contiguous rows, contiguous samples
    assert np.array_equal(oracle.blur(view, 10), oracle.blur(np.ascontiguousarray(view), 10))


def test_psnr_db_helper():
    assert oracle_pkg.psnr_db(0, 100, 8) == float("inf")
    # MSE 1 at 8 bits: 10 log10(255^2) = 48.1308...
    assert abs(oracle_pkg.psnr_db(100, 100, 8) - 20 * np.log10(255.0)) < 1e-12
