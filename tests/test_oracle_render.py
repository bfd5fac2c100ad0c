"""Pins of the oracle's compositing, ordering, loss and gradients.

- one Gaussian: image = alpha*c + (1-alpha)*bg with alpha from scipy's bivariate
  normal density (pins the power / conic sign conventions);
- the compositing weights plus the final transmittance sum to one;
- literal per-pixel candidate scan (every Gaussian against every pixel) equals
  the per-tile lists, bit for bit;
- per-tile order equals numpy's lexsort on (depth, index);
- a stack of clamped (alpha = 0.99) Gaussians stops where fp32 arithmetic of
  the transmittance product says it must;
- gradients of the L1 loss equal central finite differences in fp64 for every
  parameter (deg 0 and deg 3), excluding parameters whose +-h runs change a
  discrete decision.
"""
import math

import numpy as np
import pytest
from scipy.stats import multivariate_normal

import oracle
from differentiable_rasterizer_gb300 import scenes


def _one_gauss_scene(W=64, H=64, f=80.0, sh=0, bg=(0.1, 0.2, 0.3), **kw):
    cam = scenes.Camera(np.eye(3, dtype=np.float32), np.zeros(3, np.float32), f, f, W / 2, H / 2, W, H)
    opts = dict(scenes.DEFAULT_OPTS)
    opts["bg"] = bg
    opts.update(kw)
    return cam, opts


def test_single_gaussian_closed_form():
    cam, opts = _one_gauss_scene()
    rng = np.random.default_rng(3)
    for trial in range(5):
        p = np.zeros((14, 1))
        p[0:3, 0] = [rng.uniform(-0.3, 0.3), rng.uniform(-0.3, 0.3), rng.uniform(2.5, 4)]
        p[3:6, 0] = rng.uniform(-2.5, -1.5, 3)
        q = rng.standard_normal(4)
        p[6:10, 0] = q / np.linalg.norm(q)
        p[10, 0] = rng.normal(0, 1)
        p[11:14, 0] = rng.uniform(0, 1, 3)
        pr = oracle.project(p, 0, cam, opts, "f64")
        assert pr["visible"][0]
        out = oracle.render(pr, cam, opts, prec="f64")
        rec = pr["rec"][0]
        S2 = np.linalg.inv(np.array([[rec[2], rec[3]], [rec[3], rec[4]]]))
        mvn = multivariate_normal(mean=rec[:2], cov=S2)
        ys, xs = np.mgrid[0:cam.height, 0:cam.width]
        pts = np.stack([xs + 0.5, ys + 0.5], -1).reshape(-1, 2)
        G = mvn.pdf(pts) * 2 * np.pi * np.sqrt(np.linalg.det(S2))
        alpha = np.minimum(float(np.float32(opts["alpha_max"])), rec[5] * G)
        # support: the pixel's tile inside the rect
        r = pr["rect"][0]
        tx, ty = (pts[:, 0] // 16).astype(int), (pts[:, 1] // 16).astype(int)
        inside = (tx >= r[0]) & (tx < r[2]) & (ty >= r[1]) & (ty < r[3])
        used = inside & (alpha >= float(np.float32(opts["alpha_min"])))
        alpha = np.where(used, alpha, 0.0)
        bg = np.array([float(np.float32(b)) for b in opts["bg"]])
        expect = alpha[None, :] * rec[6:9, None] + (1 - alpha[None, :]) * bg[:, None]
        assert np.abs(out["image"].reshape(3, -1) - expect).max() < 1e-12


@pytest.mark.parametrize("name", ["tiny", "small-reduced"])
def test_weights_plus_final_transmittance_is_one(name):
    sc = scenes.make_scene("tiny") if name == "tiny" else scenes.make_scene("small", n=3000)
    cam = sc.cameras[0]
    p = sc.params.copy()
    opts_w = dict(sc.opts, bg=(0.0, 0.0, 0.0))
    opts_t = dict(sc.opts, bg=(1.0, 1.0, 1.0))
    p_one = p.copy(); p_one[11:14] = 1.0
    p_zero = p.copy(); p_zero[11:14] = 0.0
    sum_w = oracle.render(oracle.project(p_one, 0, cam, opts_w), cam, opts_w)["image"]
    t_fin = oracle.render(oracle.project(p_zero, 0, cam, opts_t), cam, opts_t)["image"]
    assert (t_fin > 0).all() and (t_fin <= 1).all()
    total = sum_w.astype(np.float64) + t_fin.astype(np.float64)
    # each composite adds one rounding; lists are short here
    assert np.abs(total - 1.0).max() < 64 * np.finfo(np.float32).eps
    # the stored final transmittance is the one the background was weighted with
    out = oracle.render(oracle.project(p_zero, 0, cam, opts_t), cam, opts_t, want_tfinal=True)
    assert np.array_equal(out["t_final"], t_fin[0]) and np.array_equal(out["t_final"], t_fin[2])


@pytest.mark.parametrize("excl", [0, 1])
def test_literal_equals_tile_lists(excl):
    sc = scenes.make_scene("tiny")
    cam = sc.cameras[0]
    opts = dict(sc.opts, exclude_crossing=excl)
    pr = oracle.project(sc.params, 0, cam, opts)
    a = oracle.render(pr, cam, opts, target=sc.target_uniform[0], mode=0, want_last=True, want_sig=True)
    b = oracle.render(pr, cam, opts, target=sc.target_uniform[0], mode=1, want_last=True, want_sig=True)
    assert np.array_equal(a["image"], b["image"])
    assert np.array_equal(a["grad2d"], b["grad2d"])
    assert np.array_equal(a["touched"], b["touched"]) and np.array_equal(a["last"], b["last"])
    assert (a["e_fwd"], a["e_bwd"], a["sig"], a["loss"]) == (b["e_fwd"], b["e_bwd"], b["sig"], b["loss"])
    assert a["touched"].sum() > 100


@pytest.mark.slow
def test_literal_equals_tile_lists_small_reduced():
    sc = scenes.make_scene("small", n=4000)
    cam = scenes.Camera(sc.cameras[0].R, sc.cameras[0].t, 250.0, 250.0, 160.0, 90.0, 320, 180)
    pr = oracle.project(sc.params, 0, cam, sc.opts)
    tgt = np.random.default_rng(0).uniform(0, 1, (3, 180, 320)).astype(np.float32)
    a = oracle.render(pr, cam, sc.opts, target=tgt, mode=0, want_sig=True)
    b = oracle.render(pr, cam, sc.opts, target=tgt, mode=1, want_sig=True)
    assert np.array_equal(a["image"], b["image"]) and np.array_equal(a["grad2d"], b["grad2d"])
    assert a["sig"] == b["sig"]


def test_tile_order_is_lexsort_depth_index():
    sc = scenes.make_scene("small", n=20000)
    cam = sc.cameras[0]
    pr = oracle.project(sc.params, 0, cam, sc.opts)
    off, ids = oracle.tile_lists(pr, cam)
    vis = pr["visible"].astype(bool)
    depth = pr["rec"][:, 9]
    rect = pr["rect"]
    tx = (cam.width + 15) // 16
    rng = np.random.default_rng(0)
    for t in rng.choice(len(off) - 1, 60, replace=False):
        x, y = t % tx, t // tx
        members = np.flatnonzero(vis & (rect[:, 0] <= x) & (x < rect[:, 2]) & (rect[:, 1] <= y) & (y < rect[:, 3]))
        order = members[np.lexsort((members, depth[members].view(np.uint32)))]
        assert np.array_equal(ids[off[t]:off[t + 1]], order)


@pytest.mark.parametrize("excl", [0, 1])
def test_alpha_stack_stops_by_fp32_transmittance(excl):
    """K coincident Gaussians, all clamped at alpha = 0.99: the number composited is the
    first k with the fp32 product of (1 - 0.99f) below 1e-4f (inclusive or exclusive of
    the crossing layer)."""
    cam, opts = _one_gauss_scene(W=16, H=16, f=16.0, bg=(0, 0, 0), exclude_crossing=excl)
    K = 5
    p = np.zeros((14, K), np.float32)
    p[2] = 2.0 + np.arange(K, dtype=np.float32) * 0.1
    p[3:6] = 0.0
    p[6] = 1.0
    p[10] = 20.0
    p[11:14] = 1.0
    pr = oracle.project(p, 0, cam, opts)
    out = oracle.render(pr, cam, opts, want_last=True)
    one_minus = np.float32(1.0) - np.float32(0.99)
    T, k = np.float32(1.0), 0
    while k < K:
        Tn = np.float32(T * one_minus)
        if excl and Tn < np.float32(1e-4):
            break
        T, k = Tn, k + 1
        if not excl and T < np.float32(1e-4):
            break
    centre = out["last"][8, 8]
    assert centre + 1 == k
    assert out["image"][0, 8, 8] == pytest.approx(1.0 - float(T), abs=1e-6)


# ----------------------------------------------------------------------------- finite differences
def _loss_and_sig(params, sc, prec="f64"):
    cam = sc.cameras[0]
    pr = oracle.project(params, sc.sh_degree, cam, sc.opts, prec)
    out = oracle.render(pr, cam, sc.opts, target=sc.target_uniform[0], prec=prec, grads=False, want_sig=True)
    return out["loss"], (out["sig"], pr["clamp"].tobytes())


def _analytic(params, sc):
    cam = sc.cameras[0]
    pr = oracle.project(params, sc.sh_degree, cam, sc.opts, "f64")
    out = oracle.render(pr, cam, sc.opts, target=sc.target_uniform[0], prec="f64")
    return oracle.vjp(params, sc.sh_degree, cam, sc.opts, out["grad2d"], out["touched"], pr["clamp"], prec="f64")


@pytest.mark.parametrize("sh,seed", [(0, 11), (3, 12), (3, 13)])
def test_gradients_match_central_differences(sh, seed):
    sc = scenes.random_small_scene(seed, n=6, width=32, height=32, sh_degree=sh)
    sc.opts = dict(sc.opts, bg=(0.2, 0.3, 0.4))
    p0 = sc.params.astype(np.float64)
    g = _analytic(p0, sc)
    _, sig0 = _loss_and_sig(p0, sc)
    checked = 0
    nz = 0
    for r in range(p0.shape[0]):
        for i in range(p0.shape[1]):
            h = 1e-6 * max(1.0, abs(p0[r, i]))
            pp = p0.copy(); pp[r, i] += h
            pm = p0.copy(); pm[r, i] -= h
            lp, sp = _loss_and_sig(pp, sc)
            lm, sm = _loss_and_sig(pm, sc)
            if sp != sig0 or sm != sig0:
                continue
            fd = (lp - lm) / (2 * h)
            checked += 1
            nz += abs(fd) > 1e-8
            assert abs(g[r, i] - fd) <= 1e-6 * abs(fd) + 1e-9, (r, i, g[r, i], fd)
    assert checked >= 0.8 * p0.size
    assert nz >= 0.5 * checked


def test_gradient_of_a_culled_or_untouched_gaussian_is_zero():
    sc = scenes.random_small_scene(5, n=4, width=32, height=32, sh_degree=0)
    p = sc.params.astype(np.float64)
    p[2, 0] = -1.0   # behind the camera
    g = _analytic(p, sc)
    assert np.all(g[:, 0] == 0)


def test_tile_masked_render_equals_full_render_on_those_tiles():
    sc = scenes.make_scene("small", n=5000)
    cam = scenes.Camera(sc.cameras[0].R, sc.cameras[0].t, 250.0, 250.0, 160.0, 90.0, 320, 180)
    pr = oracle.project(sc.params, 0, cam, sc.opts)
    tgt = np.random.default_rng(2).uniform(0, 1, (3, 180, 320)).astype(np.float32)
    full = oracle.render(pr, cam, sc.opts, target=tgt)
    tiles = 20 * 12
    mask = np.zeros(tiles, bool)
    mask[np.random.default_rng(3).choice(tiles, 40, replace=False)] = True
    part = oracle.render(pr, cam, sc.opts, target=tgt, tile_mask=mask)
    pix = np.repeat(np.repeat(mask.reshape(12, 20), 16, 0), 16, 1)[:180, :320]
    assert np.array_equal(part["image"][:, pix], full["image"][:, pix])
    assert not part["image"][:, ~pix].any()
    allm = oracle.render(pr, cam, sc.opts, target=tgt, tile_mask=np.ones(tiles, bool))
    assert np.array_equal(allm["grad2d"], full["grad2d"]) and allm["loss"] == full["loss"]
    assert (allm["e_fwd"], allm["e_bwd"], allm["e_comp"]) == (full["e_fwd"], full["e_bwd"], full["e_comp"])
