"""Regression pin: the oracle reproduces its committed fixtures exactly.

The fixtures under tests/golden/ are written by tests/golden/make_golden.py,
which calls only the oracle.  A change to the oracle's arithmetic that moves
any of these values must be justified in its commit message.
"""
import json
import os

import numpy as np
import pytest

from tests.golden.make_golden import CASES, run_case

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_oracle_matches_fixture(case):
    name, wname, over, n, step, seed = case[:6]
    pover = case[6] if len(case) > 6 else {}
    with open(os.path.join(HERE, name + ".json")) as f:
        ref = json.load(f)
    got = run_case(wname, over, n, step, seed, pover)
    assert len(got) == len(ref["heads"])
    for a, b in zip(got, ref["heads"]):
        for key in ("J", "level", "keys_read", "values_read", "n_candidates",
                    "c_lo", "c_hi", "cb", "jbar_sha", "ubar_sha"):
            assert a[key] == b[key], key
        for key in ("rows8", "jref_sha"):
            assert a.get(key) == b.get(key), key
        assert np.allclose(a["o"], b["o"], rtol=1e-12, atol=1e-12)
        assert a["beta"] == pytest.approx(b["beta"], rel=1e-12, abs=1e-12)
