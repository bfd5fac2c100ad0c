"""Pins of the oracle's D-SSIM term and of the renderer's combined loss gradient.

- the window sum equals scipy's Gaussian filter (sigma 1.5, radius 5, zero
  outside the image), which pins the window weights and the border handling;
- SSIM(x, x) = 1 at every pixel and its gradient vanishes there (a maximum);
- SSIM is symmetric in its two images;
- on constant images, away from the border, the map equals the closed form
  (2 a b + C1) / (a^2 + b^2 + C1);
- the SSIM gradient equals central finite differences in fp64 at pixels in
  the interior, at the borders and in the corners;
- through the renderer and the projection VJP, the gradient of
  (1 - lambda) L1 + lambda (1 - SSIM) w.r.t. every 3D parameter equals central
  finite differences in fp64, which pins how the renderer takes another loss
  term's dL/dC and weights its own L1 term.
"""
import numpy as np
import pytest
from scipy.ndimage import gaussian_filter

import oracle
from oracle import dssim
from differentiable_rasterizer_gb300 import scenes


def _imgs(seed, H=19, W=23):
    rng = np.random.default_rng(seed)
    x = rng.uniform(0, 1, (3, H, W))
    y = np.clip(x + rng.normal(0, 0.2, x.shape), 0, 1)
    return x, y


def test_window_sum_is_scipy_gaussian_filter_with_zero_padding():
    x, _ = _imgs(1)
    ref = np.stack([gaussian_filter(c, sigma=1.5, mode="constant", cval=0.0, truncate=5.0 / 1.5) for c in x])
    np.testing.assert_allclose(dssim.wsum(x), ref, rtol=1e-13, atol=1e-15)
    w = dssim.window()
    assert w.shape == (11, 11)
    assert w.sum() == pytest.approx(1.0, abs=1e-15)
    np.testing.assert_array_equal(w, w.T)
    np.testing.assert_array_equal(w, w[::-1, ::-1])


def test_ssim_of_an_image_with_itself_is_one_and_stationary():
    x, _ = _imgs(2)
    np.testing.assert_allclose(dssim.ssim_map(x, x), 1.0, rtol=0, atol=1e-13)
    np.testing.assert_allclose(dssim.ssim_grad(x, x), 0.0, rtol=0, atol=1e-13)


def test_ssim_is_symmetric():
    x, y = _imgs(3)
    np.testing.assert_allclose(dssim.ssim_map(x, y), dssim.ssim_map(y, x), rtol=1e-14, atol=0)


@pytest.mark.parametrize("a,b", [(0.3, 0.7), (0.0, 0.5), (1.0, 1.0), (0.02, 0.9)])
def test_constant_images_closed_form_in_the_interior(a, b):
    H, W = 24, 30
    x = np.full((3, H, W), a)
    y = np.full((3, H, W), b)
    m = dssim.ssim_map(x, y)
    want = (2 * a * b + dssim.C1) / (a * a + b * b + dssim.C1)
    np.testing.assert_allclose(m[:, 5:H - 5, 5:W - 5], want, rtol=1e-10)
    # at the border the zero padding pulls the means (and the variance) away
    if a != b:
        assert not np.allclose(m[:, 0, 0], want, rtol=1e-6)


@pytest.mark.parametrize("seed", [4, 5])
def test_ssim_gradient_matches_central_differences(seed):
    x, y = _imgs(seed, H=17, W=21)
    g = dssim.ssim_grad(x, y)
    pix = [(0, 0, 0), (1, 16, 20), (2, 0, 20), (0, 16, 0), (1, 8, 10), (2, 3, 4), (0, 5, 0), (1, 0, 7)]
    h = 1e-6
    for c, i, j in pix:
        xp = x.copy(); xp[c, i, j] += h
        xm = x.copy(); xm[c, i, j] -= h
        fd = (dssim.ssim(xp, y) - dssim.ssim(xm, y)) / (2 * h)
        assert abs(g[c, i, j] - fd) <= 1e-6 * abs(fd) + 1e-11, (c, i, j, g[c, i, j], fd)
    assert np.count_nonzero(np.abs(g) > 1e-9) > 0.9 * g.size


# ----------------------------------------------------------------------------- through the renderer
def _combined_loss(params, sc, lam):
    cam = sc.cameras[0]
    pr = oracle.project(params, sc.sh_degree, cam, sc.opts, "f64")
    out = oracle.render(pr, cam, sc.opts, target=sc.target_uniform[0], prec="f64", grads=False, want_sig=True)
    l = dssim.loss(out["image"], sc.target_uniform[0], lam)
    return l, (out["sig"], pr["clamp"].tobytes()), out


@pytest.mark.parametrize("sh,seed,lam", [(0, 21, 0.2), (3, 22, 0.2), (0, 23, 1.0)])
def test_combined_loss_gradient_matches_central_differences(sh, seed, lam):
    sc = scenes.random_small_scene(seed, n=6, width=32, height=32, sh_degree=sh)
    sc.opts = dict(sc.opts, bg=(0.2, 0.3, 0.4))
    cam = sc.cameras[0]
    p0 = sc.params.astype(np.float64)
    l0, sig0, fwd = _combined_loss(p0, sc, lam)
    pr = oracle.project(p0, sc.sh_degree, cam, sc.opts, "f64")
    extra = dssim.dssim_dldc(fwd["image"], sc.target_uniform[0], lam)
    out = oracle.render(pr, cam, sc.opts, target=sc.target_uniform[0], prec="f64", dldc_extra=extra,
                        l1_weight=1.0 - lam)
    # the renderer's loss is its weighted L1 share alone
    assert out["loss"] == pytest.approx((1 - lam) * np.abs(fwd["image"] - sc.target_uniform[0]).mean(), rel=1e-12)
    g = oracle.vjp(p0, sc.sh_degree, cam, sc.opts, out["grad2d"], out["touched"], pr["clamp"], prec="f64")
    checked = nz = 0
    for r in range(p0.shape[0]):
        for i in range(p0.shape[1]):
            h = 1e-6 * max(1.0, abs(p0[r, i]))
            pp = p0.copy(); pp[r, i] += h
            pm = p0.copy(); pm[r, i] -= h
            lp, sp, _ = _combined_loss(pp, sc, lam)
            lm, sm, _ = _combined_loss(pm, sc, lam)
            if sp != sig0 or sm != sig0:
                continue
            fd = (lp - lm) / (2 * h)
            checked += 1
            nz += abs(fd) > 1e-8
            assert abs(g[r, i] - fd) <= 2e-6 * abs(fd) + 1e-9, (r, i, g[r, i], fd)
    assert checked >= 0.8 * p0.size
    assert nz >= 0.5 * checked
