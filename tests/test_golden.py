"""The oracle against its stored digest on the tiny workload (CPU).

``tests/golden/tiny_oracle_digest.json`` was written by
``tests/golden/make_golden.py``, which calls only the oracle and the seeded
input generator.  A change to either (a different recipe, a changed step of
the oracle) moves these numbers; an intended change regenerates the file
and names the reason in its commit.
"""

import json
import os

import numpy as np

from tests.golden import make_golden

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "tiny_oracle_digest.json")


def test_oracle_matches_stored_digest():
    with open(GOLDEN) as f:
        want = json.load(f)
    got = make_golden.digest()
    assert got["workload"] == want["workload"]
    for key in make_golden.KEYS:
        g, w = got[key], want[key]
        assert g["shape"] == w["shape"], key
        for field in ("sum", "l2"):
            assert np.isclose(g[field], w[field], rtol=1e-12, atol=1e-14), (key, field)
        for field in ("first", "last"):
            np.testing.assert_allclose(g[field], w[field], rtol=1e-12, atol=1e-14, err_msg=f"{key} {field}")
