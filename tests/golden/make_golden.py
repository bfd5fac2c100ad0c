"""Writes tests/golden/oracle_tiny.json from the CPU oracle alone.

The pages print no worked example (no image, loss or gradient value), so the
stored values here are the oracle's own fp32 results on the seeded tiny
workload.  They pin the oracle against itself across machines and compilers
(x86-64 here, aarch64 on the GPU host): the fp32 forward must be bit-identical
everywhere, because the CUDA path is compared with it bit for bit.

Run:  python tests/golden/make_golden.py
"""
import hashlib
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from differentiable_rasterizer_gb300 import scenes  # noqa: E402


def summary():
    sc = scenes.make_scene("tiny")
    cam = sc.cameras[0]
    pr = oracle.project(sc.params, 0, cam, sc.opts)
    out = oracle.render(pr, cam, sc.opts, target=sc.target_uniform[0])
    g2 = out["grad2d"]
    return {
        "workload": "tiny (1000 Gaussians, 64x64, seed 0)",
        "visible": int(pr["visible"].sum()),
        "rec_sha256": hashlib.sha256(pr["rec"].tobytes() + pr["rect"].tobytes()).hexdigest(),
        "image_sha256": hashlib.sha256(out["image"].tobytes()).hexdigest(),
        "loss": repr(out["loss"]),
        "e_fwd": out["e_fwd"],
        "e_bwd": out["e_bwd"],
        "touched": int(out["touched"].sum()),
        "grad2d_abs_sum": repr(float(np.abs(g2).sum())),
    }


if __name__ == "__main__":
    with open(os.path.join(HERE, "oracle_tiny.json"), "w") as f:
        json.dump(summary(), f, indent=1, sort_keys=True)
        f.write("\n")
