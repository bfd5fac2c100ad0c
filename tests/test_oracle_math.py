"""Pins of the oracle's building blocks against mathematics and library routines.

Nothing here re-types the oracle's own formulas: every expected value comes from
an independent route (libm/numpy exp, scipy's complex spherical harmonics and
rotations, numerical Jacobians of the pinhole map, eigenvalue routines,
interval intersection for the tile rule, Gaussian densities from scipy.stats).
"""
import math

import numpy as np
import pytest
import scipy.special
from scipy.spatial.transform import Rotation

import oracle
from differentiable_rasterizer_gb300 import scenes


def ulp_diff(a, b):
    a = np.asarray(a, np.float32).view(np.int32).astype(np.int64)
    b = np.asarray(b, np.float32).view(np.int32).astype(np.int64)
    return np.abs(a - b)


# ----------------------------------------------------------------------------- portable exp
def test_pexp_within_one_ulp_of_correctly_rounded_exp():
    rng = np.random.default_rng(0)
    x = np.concatenate([np.linspace(-103.0, 88.5, 40001), rng.uniform(-20, 0, 20000),
                        rng.uniform(-0.35, 0.35, 5000)]).astype(np.float32)
    got = oracle.pexp_f32(x)
    ref = np.exp(x.astype(np.float64)).astype(np.float32)   # correctly rounded to within double rounding
    normal = ref > np.float32(1.17549435e-38)
    assert ulp_diff(got[normal], ref[normal]).max() <= 1
    # denormal range: absolute error below one denormal step
    assert np.abs(got[~normal].astype(np.float64) - np.exp(x[~normal].astype(np.float64))).max() <= 1.5e-45


def test_pexp_special_values():
    got = oracle.pexp_f32([0.0, -0.0, float("nan"), 100.0, -200.0, float("-inf"), float("inf")])
    assert got[0] == 1.0 and got[1] == 1.0
    assert np.isnan(got[2])
    assert np.isinf(got[3]) and got[4] == 0.0 and got[5] == 0.0 and np.isinf(got[6])


# ----------------------------------------------------------------------------- spherical harmonics
def _real_sh_scipy(l, m, theta, phi):
    """Real orthonormal SH without Condon-Shortley phase, from scipy's complex Y_l^m."""
    if m == 0:
        return scipy.special.sph_harm_y(l, 0, theta, phi).real
    Y = scipy.special.sph_harm_y(l, abs(m), theta, phi)
    if m > 0:
        return math.sqrt(2.0) * (-1) ** m * Y.real
    return math.sqrt(2.0) * (-1) ** m * Y.imag


@pytest.mark.parametrize("prec", ["f64", "f32"])
def test_sh_basis_matches_scipy(prec):
    rng = np.random.default_rng(1)
    d = rng.standard_normal((500, 3))
    d /= np.linalg.norm(d, axis=1, keepdims=True)
    theta = np.arccos(np.clip(d[:, 2], -1, 1))
    phi = np.arctan2(d[:, 1], d[:, 0])
    got = oracle.sh_basis(d, prec).astype(np.float64)
    tol = 1e-12 if prec == "f64" else 2e-6
    for l in range(4):
        for m in range(-l, l + 1):
            k = l * l + l + m
            ref = _real_sh_scipy(l, m, theta, phi)
            assert np.abs(got[:, k] - ref).max() < tol, (l, m)


def test_sh_basis_orthonormal_by_quadrature():
    xg, wg = np.polynomial.legendre.leggauss(16)       # cos(theta) nodes
    nphi = 32
    phi = (np.arange(nphi) + 0.5) * 2 * np.pi / nphi
    ct, ph = np.meshgrid(xg, phi, indexing="ij")
    st = np.sqrt(1 - ct ** 2)
    d = np.stack([st * np.cos(ph), st * np.sin(ph), ct], -1).reshape(-1, 3)
    w = (np.repeat(wg, nphi) * (2 * np.pi / nphi))
    Y = oracle.sh_basis(d, "f64")
    gram = (Y * w[:, None]).T @ Y
    assert np.abs(gram - np.eye(16)).max() < 1e-12


# ----------------------------------------------------------------------------- projection
def _cam(R=None, t=None, f=100.0, W=64, H=48, cx=None, cy=None):
    R = np.eye(3, dtype=np.float32) if R is None else np.asarray(R, np.float32)
    t = np.zeros(3, np.float32) if t is None else np.asarray(t, np.float32)
    return scenes.Camera(R, t, f, f, W / 2 if cx is None else cx, H / 2 if cy is None else cy, W, H)


def _params(mu, log_s, q, logit=0.0, rgb=(0.2, 0.5, 0.8), sh=0):
    P = scenes.PARAM_ROWS[sh]
    p = np.zeros((P, 1), np.float64)
    p[0:3, 0] = mu
    p[3:6, 0] = log_s
    p[6:10, 0] = q
    p[10, 0] = logit
    if sh == 0:
        p[11:14, 0] = rgb
    return p


def _sigma2d_from_conic(rec):
    A, B, C = rec[2], rec[3], rec[4]
    return np.linalg.inv(np.array([[A, B], [B, C]]))


def test_isotropic_on_axis_closed_form():
    opts = dict(scenes.DEFAULT_OPTS)
    for z, s, f in [(3.0, 0.05, 100.0), (10.0, 0.5, 300.0), (2.5, 0.01, 64.0)]:
        cam = _cam(f=f, W=640, H=480)
        p = _params([0, 0, z], [math.log(s)] * 3, [1, 0, 0, 0])
        out = oracle.project(p, 0, cam, opts, "f64")
        S2 = _sigma2d_from_conic(out["rec"][0])
        var = (f * s / z) ** 2 + float(np.float32(opts["lowpass"]))
        assert np.allclose(S2, var * np.eye(2), rtol=1e-10, atol=1e-12)
        assert out["rec"][0, 0] == pytest.approx(320.0) and out["rec"][0, 1] == pytest.approx(240.0)
        # f32 radius = ceil(3 sqrt(var)) (var from the closed form; skip exact integer boundaries)
        o32 = oracle.project(p.astype(np.float32), 0, cam, opts, "f32")
        r = 3 * math.sqrt(var)
        if abs(r - round(r)) > 1e-3:
            rect = o32["rect"][0]
            lo = math.floor((320.0 - math.ceil(r)) / 16)
            assert rect[0] == max(lo, 0)


def _pinhole(Xc, f, cx, cy):
    return np.array([f * Xc[0] / Xc[2] + cx, f * Xc[1] / Xc[2] + cy])


@pytest.mark.parametrize("seed", range(6))
def test_general_projection_matches_numerical_jacobian(seed):
    """Sigma2D = J Sigma J^T + lowpass*I with J the numerical Jacobian of the
    world->pixel map and Sigma from scipy's rotation; mean2d = pinhole(mean)."""
    rng = np.random.default_rng(seed)
    Rc = Rotation.from_euler("xyz", rng.uniform(-0.3, 0.3, 3)).as_matrix()
    tc = rng.uniform(-0.5, 0.5, 3)
    f, W, H = 200.0, 320, 240
    cam = _cam(Rc, tc, f, W, H)
    Rc, tc = cam.R.astype(np.float64), cam.t.astype(np.float64)
    mu = Rc.T @ (np.array([rng.uniform(-0.5, 0.5), rng.uniform(-0.5, 0.5), rng.uniform(3, 6)]) - tc)
    ls = rng.uniform(-3, -1.5, 3)
    q = rng.standard_normal(4)
    opts = dict(scenes.DEFAULT_OPTS)
    out = oracle.project(_params(mu, ls, q), 0, cam, opts, "f64")
    assert out["visible"][0] == 1
    rot = Rotation.from_quat([q[1], q[2], q[3], q[0]]).as_matrix()   # scipy is scalar-last
    Sig = rot @ np.diag(np.exp(2 * ls)) @ rot.T
    world_to_px = lambda X: _pinhole(Rc @ X + tc, f, W / 2, H / 2)
    h = 1e-6
    J = np.stack([(world_to_px(mu + h * e) - world_to_px(mu - h * e)) / (2 * h) for e in np.eye(3)], 1)
    S2_ref = J @ Sig @ J.T + float(np.float32(opts["lowpass"])) * np.eye(2)
    S2 = _sigma2d_from_conic(out["rec"][0])
    assert np.allclose(S2, S2_ref, rtol=1e-6, atol=1e-8)
    assert np.allclose(out["rec"][0, :2], world_to_px(mu), rtol=1e-12)
    assert out["rec"][0, 9] == pytest.approx((Rc @ mu + tc)[2], rel=1e-12)
    # the quaternion enters only through its direction, and q and -q agree
    out2 = oracle.project(_params(mu, ls, -2.5 * q), 0, cam, opts, "f64")
    assert np.allclose(out2["rec"], out["rec"], rtol=1e-12, atol=1e-14)


def test_radius_is_ceil_three_sigma_of_largest_eigenvalue():
    rng = np.random.default_rng(7)
    sc = scenes.make_scene("tiny")
    cam = sc.cameras[0]
    out = oracle.project(sc.params.astype(np.float64), 0, cam, sc.opts, "f64")
    vis = np.flatnonzero(out["visible"])
    for g in rng.choice(vis, 50, replace=False):
        rec = out["rec"][g]
        lam = np.linalg.eigvalsh(_sigma2d_from_conic(rec)).max()
        r = math.ceil(3 * math.sqrt(lam) - 1e-9)
        # rect must be exactly the tiles whose pixel span meets [m - r, m + r] (interval intersection)
        for ax, (lo_i, hi_i, ntiles) in enumerate([(0, 2, 4), (1, 3, 4)]):
            m = rec[ax]
            tiles = [t for t in range(ntiles) if 16 * t <= m + r and 16 * (t + 1) > m - r]
            got = list(range(out["rect"][g, lo_i], out["rect"][g, hi_i]))
            assert got == tiles, (g, ax)


def test_rect_is_interval_intersection_f32():
    sc = scenes.make_scene("small", n=20000)
    cam = sc.cameras[0]
    out = oracle.project(sc.params, 0, cam, sc.opts, "f32")
    vis = out["visible"].astype(bool)
    rec = out["rec"].astype(np.float64)
    # radius from the conic (f32 values) and the rect bounds: every visible rect is non-empty,
    # inside the grid, and contains the tile of a centre that lies in the image
    tx, ty = (cam.width + 15) // 16, (cam.height + 15) // 16
    rect = out["rect"][vis]
    assert (rect[:, 0] >= 0).all() and (rect[:, 2] <= tx).all() and (rect[:, 0] < rect[:, 2]).all()
    assert (rect[:, 1] >= 0).all() and (rect[:, 3] <= ty).all() and (rect[:, 1] < rect[:, 3]).all()
    inside = (rec[vis, 0] >= 0) & (rec[vis, 0] < cam.width) & (rec[vis, 1] >= 0) & (rec[vis, 1] < cam.height)
    ctx = np.floor(rec[vis, 0] / 16).astype(int)
    cty = np.floor(rec[vis, 1] / 16).astype(int)
    ok = (rect[:, 0] <= ctx) & (ctx < rect[:, 2]) & (rect[:, 1] <= cty) & (cty < rect[:, 3])
    assert ok[inside].all()


def test_culling_near_plane_and_non_finite():
    cam = _cam(W=64, H=64)
    opts = dict(scenes.DEFAULT_OPTS)
    base = _params([0, 0, 3.0], [-3] * 3, [1, 0, 0, 0]).astype(np.float32)
    assert oracle.project(base, 0, cam, opts)["visible"][0] == 1
    behind = base.copy(); behind[2, 0] = 0.1
    assert oracle.project(behind, 0, cam, opts)["visible"][0] == 0
    for row in (0, 3, 6, 10, 11):
        bad = base.copy(); bad[row, 0] = np.nan
        assert oracle.project(bad, 0, cam, opts)["visible"][0] == 0, row
    zero_q = base.copy(); zero_q[6:10, 0] = 0
    assert oracle.project(zero_q, 0, cam, opts)["visible"][0] == 0
    far_off = base.copy(); far_off[0, 0] = 50.0
    assert oracle.project(far_off, 0, cam, opts)["visible"][0] == 0


def test_opacity_is_sigmoid_and_colour_degree0_is_rgb():
    cam = _cam(W=64, H=64)
    opts = dict(scenes.DEFAULT_OPTS)
    for logit in (-6.0, -1.3, 0.0, 0.7, 4.0):
        p = _params([0, 0, 3.0], [-3] * 3, [1, 0, 0, 0], logit=logit).astype(np.float32)
        rec = oracle.project(p, 0, cam, opts)["rec"][0]
        assert abs(rec[5] - scipy.special.expit(np.float64(np.float32(logit)))) < 2e-7
        assert np.array_equal(rec[6:9], p[11:14, 0])


def test_degree3_dc_only_colour_equals_rgb():
    """k00 = (rgb - 0.5)/Y00 with the higher bands at zero gives colour = rgb."""
    cam = _cam(W=64, H=64)
    opts = dict(scenes.DEFAULT_OPTS)
    rgb = np.array([0.1, 0.55, 0.9])
    Y00 = 0.5 / math.sqrt(math.pi)
    p = np.zeros((59, 1))
    p[0:3, 0] = [0.1, -0.1, 3.0]; p[3:6, 0] = -3; p[6, 0] = 1
    p[11:14, 0] = (rgb - 0.5) / Y00
    rec = oracle.project(p, 3, cam, opts, "f64")["rec"][0]
    assert np.allclose(rec[6:9], rgb, atol=1e-14)
