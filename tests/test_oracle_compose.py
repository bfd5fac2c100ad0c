"""Pins of the oracle's partial render + compose (Splaxel, English abstract:
each part renders its local Gaussian subset and only partial pixel values are
composed).  Subsets are depth slabs, so composing them front to back is the
one-pass compositing regrouped:

- one slab covering every depth composes to the one-pass render exactly;
- without the early stop (t_min = 0) any number of slabs composes to the one-pass
  render up to rounding, and the composed T is the one-pass final T;
- with the stop, the slabs behind a pixel's stop add at most t_min times the
  largest colour value, the bound the stop itself allows;
- slab order matters: composing back to front does not give the one-pass image.
"""
import numpy as np
import pytest

import oracle
from differentiable_rasterizer_gb300 import scenes


def _scene():
    sc = scenes.random_small_scene(21, n=1500, width=64, height=64, sh_degree=0, log_lo=-3.0, log_hi=-1.8,
                                   logit_mu=1.0, spread=1.2)
    sc.opts = dict(sc.opts, bg=(0.2, 0.5, 0.8))
    return sc


def _splits(pr, S):
    d = pr["rec"][pr["visible"] > 0, 9].astype(np.float64)
    return np.quantile(d, np.arange(1, S) / S)


def test_one_slab_is_the_one_pass_render():
    sc = _scene()
    cam = sc.cameras[0]
    pr = oracle.project(sc.params, 0, cam, sc.opts)
    ref = oracle.render(pr, cam, sc.opts, want_tfinal=True)
    C, T = oracle.compose(oracle.render_subsets(pr, cam, sc.opts, []), sc.opts["bg"])
    assert np.array_equal(T, ref["t_final"].astype(np.float64))
    # one-pass adds T * bg in fp32 at the end; the composition does it in fp64
    assert np.abs(C - ref["image"]).max() <= 1e-6


@pytest.mark.parametrize("S", [2, 3, 5])
def test_slabs_compose_to_the_one_pass_render_without_the_stop(S):
    sc = _scene()
    opts = dict(sc.opts, t_min=0.0)
    cam = sc.cameras[0]
    pr = oracle.project(sc.params, 0, cam, opts, "f64")
    ref = oracle.render(pr, cam, opts, prec="f64", want_tfinal=True)
    C, T = oracle.compose(oracle.render_subsets(pr, cam, opts, _splits(pr, S), prec="f64"), opts["bg"])
    assert np.abs(C - ref["image"]).max() <= 1e-12
    assert np.abs(T - ref["t_final"]).max() <= 1e-12


@pytest.mark.parametrize("S", [2, 4])
def test_slabs_behind_the_stop_add_at_most_t_min_times_the_colour(S):
    sc = _scene()
    cam = sc.cameras[0]
    pr = oracle.project(sc.params, 0, cam, sc.opts, "f64")
    ref = oracle.render(pr, cam, sc.opts, prec="f64")
    C, _ = oracle.compose(oracle.render_subsets(pr, cam, sc.opts, _splits(pr, S), prec="f64"), sc.opts["bg"])
    cmax = max(float(pr["rec"][pr["visible"] > 0, 6:9].max()), max(sc.opts["bg"]))
    d = np.abs(C - ref["image"])
    assert d.max() <= sc.opts["t_min"] * cmax * (1 + 1e-9)
    assert d.max() > 0          # some pixels do stop in this scene


def test_back_to_front_order_is_wrong():
    sc = _scene()
    opts = dict(sc.opts, t_min=0.0)
    cam = sc.cameras[0]
    pr = oracle.project(sc.params, 0, cam, opts, "f64")
    ref = oracle.render(pr, cam, opts, prec="f64")
    parts = oracle.render_subsets(pr, cam, opts, _splits(pr, 3), prec="f64")
    C, _ = oracle.compose(parts[::-1], opts["bg"])
    assert np.abs(C - ref["image"]).max() > 1e-2
