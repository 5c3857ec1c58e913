"""The oracles reproduce their stored regression record (tests/golden/oracle_regression.json,
written by tests/golden/make_golden.py, which calls only oracle/).  A change to an oracle's
arithmetic fails here until the record is regenerated in a commit that says why (no GPU)."""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))

import make_golden  # noqa: E402


def test_oracles_match_their_golden_record():
    with open(os.path.join(HERE, "golden", "oracle_regression.json")) as f:
        stored = json.load(f)["cases"]
    fresh = make_golden.compute()
    assert sorted(stored) == sorted(fresh)
    for case, arrays in stored.items():
        for name, want in arrays.items():
            want, got = np.asarray(want, dtype=np.float64), np.asarray(fresh[case][name], dtype=np.float64)
            assert want.shape == got.shape, (case, name)
            same_nan = np.array_equal(np.isnan(want), np.isnan(got))
            w, g = want[~np.isnan(want)], got[~np.isnan(got)]
            # across C libraries exp() may differ in its last bit: allow a few ulps of slack
            assert same_nan and np.allclose(g, w, rtol=1e-10, atol=1e-12), (case, name)
