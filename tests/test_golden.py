"""The oracle still reproduces its stored small-problem fixture (drift guard).
CPU only."""
import json
import os

import numpy as np

from tests.golden.make_golden import compute

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_oracle_matches_fixture():
    with open(os.path.join(HERE, "oracle_small.json")) as fh:
        stored = json.load(fh)["values"]
    now = compute()
    assert set(stored) == set(now)
    for k in stored:
        a, b = np.array(now[k]), np.array(stored[k])
        assert np.abs(a - b).max() <= 1e-13 * max(1.0, np.abs(b).max()), k
