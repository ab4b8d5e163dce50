"""The oracle against its stored fixtures (tests/golden, written by make_golden.py from the
oracle alone): a later edit of the oracle, or another compiler or platform, must reproduce
them to 1e-12 of each tensor's scale (libm's exp and log may differ in the last bit between
platforms; the oracle's own arithmetic is in a fixed order)."""
import glob
import json
import os
import sys

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))

import make_golden  # noqa: E402

FILES = sorted(glob.glob(os.path.join(HERE, "golden", "oracle_*.json")))


def test_fixtures_exist():
    assert {os.path.basename(f) for f in FILES} == {f"oracle_{w}.json" for w in make_golden.WORKLOADS}


@pytest.mark.parametrize("path", FILES, ids=[os.path.basename(f) for f in FILES])
def test_oracle_reproduces_its_fixtures(path):
    with open(path) as f:
        fix = json.load(f)
    now = make_golden.golden(fix["workload"])
    assert set(now) == set(fix["outputs"])
    for key, want in fix["outputs"].items():
        got = now[key]
        assert got["size"] == want["size"], key
        scale = np.sqrt(want["sumsq"] / max(want["size"], 1))
        tol = 1e-12 * max(scale, 1e-300)
        assert abs(got["sum"] - want["sum"]) <= tol * want["size"], key
        assert abs(got["sumsq"] - want["sumsq"]) <= 1e-12 * want["sumsq"] + 1e-300, key
        assert set(got["at"]) == set(want["at"]), key
        for i, v in want["at"].items():
            assert abs(got["at"][i] - v) <= tol, (key, i)
