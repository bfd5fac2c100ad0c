"""The bounds-checked build (libgs_gb300_checked.so: the library's sources with
-DGS_CHECKED) on the GPU.  Each case runs tests/checked_child.py in a child
process with GS_CHECKED=1, so that the child loads the checked library while
this process keeps the plain one:

- the tiny workload's oracle parity runs pass through the checked library with
  no failed bounds check;
- one training step of tiny, small, medium and a 4-view slice of the batched
  workload gives, through the checked library, the same deterministic outputs
  as the plain one (tile ranges, sorted keys and ids, image, compacted lists,
  last_step bit for bit; loss and gradients, which float atomics sum in a
  varying order, to rounding), with no failed check;
- a listed index equal to n planted in gs_adam_deferred's list and a sorted id
  beyond n planted in the fused raster's list are caught at their sites, with
  that index and bound, and the rest of each output is unchanged.

The plain library reports itself unchecked and compiles every check away.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
CHILD = os.path.join(HERE, "checked_child.py")


@pytest.fixture(scope="module")
def ready():
    from differentiable_rasterizer_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _child(*args):
    env = dict(os.environ, GS_CHECKED="1")
    r = subprocess.run([sys.executable, CHILD, *args], env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, (r.stdout[-4000:], r.stderr[-4000:])
    return r.stdout


def test_plain_build_reports_no_checks(ready):
    from differentiable_rasterizer_gb300 import abi
    rep = abi.gs_check_report()
    assert rep == {"checked": False, "failures": 0, "site": "none", "index": 0, "bound": 0}


def test_checked_build_passes_the_tiny_parity_runs_with_no_failed_check(ready):
    assert "parity ok" in _child("parity")


def test_checked_build_gives_the_plain_build_outputs_with_no_failed_check(ready, tmp_path):
    sys.path.insert(0, HERE)
    import checked_child
    path = str(tmp_path / "checked.json")
    _child("outputs", path)
    with open(path) as f:
        checked = json.load(f)
    for w in checked_child.WORKLOADS:
        plain = checked_child.workload_outputs(*w)
        got = checked[w[0]]
        for key in ("instances", "ranges", "keys", "ids", "image", "n_idx", "idx", "last_step"):
            assert got[key] == plain[key], (w[0], key)
        np.testing.assert_allclose(got["loss"], plain["loss"], rtol=1e-9, atol=0)
        np.testing.assert_allclose(got["grad_abs_sum"], plain["grad_abs_sum"], rtol=1e-4, atol=0)
        np.testing.assert_allclose(np.array(got["grad_sample"]), np.array(plain["grad_sample"]), rtol=1e-3,
                                   atol=1e-4 * plain["grad_max"])
        torch.cuda.empty_cache()


def test_planted_bad_indexes_are_caught_where_they_are_read(ready):
    assert "planted ok" in _child("planted")
