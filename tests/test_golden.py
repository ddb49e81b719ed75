"""The oracle reproduces its committed tiny-call record (drift / cross-machine check)."""
import json
import os

import numpy as np

from golden.make_golden import compute

HERE = os.path.dirname(os.path.abspath(__file__))


def test_tiny_call_record():
    with open(os.path.join(HERE, "golden", "tiny_call.json")) as f:
        doc = json.load(f)
    res = compute()
    for k, hexes in doc["values"].items():
        ref = np.array([float.fromhex(h) for h in hexes])
        got = res[k].reshape(-1)
        assert got.shape == ref.shape, k
        np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-15, err_msg=k)
