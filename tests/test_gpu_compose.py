"""GPU parity of partial render + compose against the oracle: the slab sub-ranges
of every tile list (bit-exact against the oracle's lists of each slab), each
slab's colour and transmittance, and the composed image -- against the oracle's
composition and against the one-pass oracle render within the bound the early
stop allows (the transmittance at which a pixel stops times the largest colour
value)."""
import math

import numpy as np
import pytest
import torch

import oracle
from differentiable_rasterizer_gb300 import pipeline, scenes

import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from differentiable_rasterizer_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _dense():
    sc = scenes.random_small_scene(21, n=4000, width=64, height=64, sh_degree=0, log_lo=-3.0, log_hi=-1.8,
                                   logit_mu=1.0, spread=1.2)
    sc.opts = dict(sc.opts, bg=(0.2, 0.5, 0.8))
    return sc


@pytest.mark.parametrize("S", [1, 2, 3])
def test_compose_tiny(S):
    parity.run_compose_parity(scenes.make_scene("tiny"), S)


@pytest.mark.parametrize("S", [2, 4, 8])
def test_compose_dense_lists_with_background(S):
    parity.run_compose_parity(_dense(), S)


def test_compose_ragged_resolution():
    sc = scenes.make_scene("tiny")
    cam = sc.cameras[0]
    sc.cameras = [scenes.Camera(cam.R, cam.t, 64.0, 64.0, 35.0, 22.5, 70, 45)]
    parity.run_compose_parity(sc, 3)


def test_compose_multi_view_degree3():
    sc = scenes.make_scene("medium", n=20000)
    cams = []
    for k, ang in enumerate((-0.1, 0.0, 0.12)):
        c, s = math.cos(ang), math.sin(ang)
        R = np.array([[c, 0, s], [0, 1, 0], [-s, 0, c]], np.float32)
        cams.append(scenes.Camera(R, np.array([0.5 * k, 0.2, 0.0], np.float32), 300.0, 300.0, 160.0, 90.0, 320, 180))
    sc.cameras = cams
    sc.opts = dict(sc.opts, exclude_crossing=1, bg=(0.1, 0.4, 0.7))
    parity.run_compose_parity(sc, 3)


def test_one_slab_matches_the_one_pass_gpu_render():
    sc = _dense()
    tr = pipeline.GaussianTrainer(sc.params, 0, sc.cameras, sc.opts, sc.lr)
    a = tr.render().clone()
    b = tr.render_partial([[]]).clone()
    torch.cuda.synchronize()
    # one pass adds T * bg rounded after the product, the composition with one fma
    assert (a - b).abs().max().item() <= 1e-6
