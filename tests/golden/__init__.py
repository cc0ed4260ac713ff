"""Stored expected values for the tests, each file with its source:

* hand_worked_6x6.txt -- a worked example of the blur, SAD and score on 6x6
  frames, derived by hand from the definition (the derivation is in the file).
* oracle_cases.json -- results of the CPU oracle on seeded uniform inputs in
  the shapes of the five workloads, written by make_oracle_golden.py (which
  calls only oracle/).

This module only reads the files and rebuilds the seeded inputs; it holds no
arithmetic of the method."""
from __future__ import annotations

import json
import os

import numpy as np

import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def hand_worked_cases() -> list[dict]:
    """The cases of hand_worked_6x6.txt: name, impulse (row, col, value),
    B (6x6 int array or None), sad, score."""
    cases, cur, rows = [], None, None
    with open(os.path.join(HERE, "hand_worked_6x6.txt")) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            if rows is not None and len(rows) < 6 and line[0].isdigit():
                rows.append([int(v) for v in line.split()])
                if len(rows) == 6:
                    cur["B"] = np.array(rows, dtype=np.int64)
                    rows = None
                continue
            key, *vals = line.split()
            if key == "case":
                cur = {"name": vals[0], "B": None}
                cases.append(cur)
            elif key == "impulse":
                cur["impulse"] = tuple(int(v) for v in vals)
            elif key == "B":
                rows = []
            elif key == "sad":
                cur["sad"] = int(vals[0])
            elif key == "score":
                cur["score"] = float(vals[0])
    return cases


def impulse_frames(case: dict) -> np.ndarray:
    """(2, 6, 6) uint8: an all-zero frame, then the case's impulse frame."""
    r, c, v = case["impulse"]
    fr = np.zeros((2, 6, 6), np.uint8)
    fr[1, r, c] = v
    return fr


def oracle_cases() -> list[dict]:
    with open(os.path.join(HERE, "oracle_cases.json")) as f:
        return json.load(f)["cases"]


def case_inputs(kind: str, seed: int, n: int, w: int, h: int, bpc: int):
    """A stored case's inputs: frames (n, h, w) for motion / motion_v2, a
    synth.Yuv420Batch for yuv420 and moments (moments use its two lumas)."""
    if kind in ("motion", "motion_v2"):
        return synth.uniform_frames(seed, n, w, h, bpc)
    return synth.uniform_yuv420(seed, n, w, h, bpc)
