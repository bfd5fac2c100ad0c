"""GPU parity on the full-size large and batched workloads (sampled tiles and
Gaussians, every record and every tile list), on the batched recipe at a
reduced size where every output is compared, and on the medium workload (the
one the bench times) for the next-ranked rows: the L1 + D-SSIM step, the step
on pruned lists, and the partial render + compose -- every output compared."""
import math

import numpy as np
import pytest
import torch

import oracle
from differentiable_rasterizer_gb300 import scenes

import parity

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from differentiable_rasterizer_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def test_large_full_size_sampled():
    st = parity.run_sampled_parity(scenes.make_scene("large"), n_tiles=64, n_gauss=400, seed=1)
    assert st["instances"] > 5_000_000


def test_batched_full_size_sampled_views():
    st = parity.run_sampled_parity(scenes.make_scene("batched"), check_views=(0, 9), n_tiles=32, n_gauss=200,
                                   seed=2)
    assert st["instances"] > 100_000_000


def test_batched_recipe_reduced_all_views_elementwise():
    sc = scenes.make_scene("batched", n=60000)
    cams = []
    for c in sc.cameras:
        cams.append(scenes.Camera(c.R, c.t, 350.0, 350.0, 240.0, 135.0, 480, 270))
    sc.cameras = cams
    parity.run_stage_parity(sc)


def test_medium_dssim_step_full():
    st = parity.run_dssim_parity(scenes.make_scene("medium"), 0.2)
    assert st["grads"]["bad"] == 0


def test_medium_pruned_step_full():
    sc = scenes.make_scene("medium")
    sc.opts = dict(sc.opts, tile_budget=768)
    st = parity.run_stage_parity(sc)
    assert st["pruned_tiles"][0] > 0


def test_medium_partial_render_full():
    parity.run_compose_parity(scenes.make_scene("medium"), 2)
