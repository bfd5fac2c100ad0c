"""The fp32 oracle reproduces its stored tiny-workload summary bit for bit on
this machine (the summary was written by tests/golden/make_golden.py, which
calls only the oracle)."""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))

import make_golden  # noqa: E402


def test_tiny_summary_is_reproduced():
    with open(os.path.join(HERE, "golden", "oracle_tiny.json")) as f:
        stored = json.load(f)
    got = make_golden.summary()
    for k in ("visible", "rec_sha256", "image_sha256", "loss", "e_fwd", "e_bwd", "touched"):
        assert got[k] == stored[k], k
    assert np.isclose(float(got["grad2d_abs_sum"]), float(stored["grad2d_abs_sum"]), rtol=1e-12)
