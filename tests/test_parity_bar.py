"""The gradient bar of the GPU comparisons, on CPU.

The oracle's ``grad2d_mag`` (per entry, the sum of the magnitudes of the terms
the 2D gradient sums) is pinned by what fixes it: it bounds |grad2d|; where no
term can cancel (one Gaussian, bg 0, every dL/dC of one sign) it equals |grad2d|
on the entries whose terms share a sign; flipping every dL/dC sign flips grad2d
and leaves it unchanged.  The bar built on it must reject a gradient whose small
entries are dropped, even at the 1080p scale where the literal 1e-6 floor
accepts it, and must accept rounding-size differences."""
import numpy as np

import oracle
from differentiable_rasterizer_gb300 import scenes

import parity


def _one_gaussian_scene():
    sc = scenes.make_scene("tiny")
    keep = np.argsort(np.abs(sc.params[0]) + np.abs(sc.params[1]))[:1]   # a Gaussian near the optical axis
    p = np.ascontiguousarray(sc.params[:, keep])
    p[3:6] = -2.2                     # a few pixels wide
    p[10] = 2.0                       # opaque enough to composite
    return sc, p


def test_mag_equals_abs_grad_where_terms_share_a_sign_and_ignores_the_signs():
    sc, p = _one_gaussian_scene()
    cam = sc.cameras[0]
    pr = oracle.project(p, 0, cam, sc.opts)
    assert pr["visible"][0]
    H, W = cam.height, cam.width
    lo = oracle.render(pr, cam, sc.opts, target=np.zeros((3, H, W), np.float32), want_mag=True)
    hi = oracle.render(pr, cam, sc.opts, target=np.ones((3, H, W), np.float32), want_mag=True)
    g, m = lo["grad2d"][0], lo["grad2d_mag"][0]
    assert lo["touched"][0] and np.abs(g).max() > 0
    # d conic A, C, opacity and colour: every pixel's term has the sign of dL/dC
    for k in (2, 4, 5, 6, 7, 8):
        assert np.isclose(m[k], abs(g[k]), rtol=1e-12, atol=0.0), (k, m[k], g[k])
    # d mean2d and d conic B change sign across the Gaussian: they cancel, the magnitudes do not
    for k in (0, 1, 3):
        assert m[k] > abs(g[k])
    # every dL/dC sign flipped: grad2d flips, its scale does not move
    assert np.array_equal(hi["grad2d"][0], -g)
    assert np.array_equal(hi["grad2d_mag"][0], m)


def test_mag_bounds_grad_on_scenes_with_cancellation():
    for name, opts in (("tiny", None), ("medium", dict(bg=(0.3, 0.1, 0.7)))):
        sc = scenes.make_scene(name, n=1500) if name == "medium" else scenes.make_scene(name)
        cam = sc.cameras[0]
        if name == "medium":
            cam = scenes.Camera(cam.R, cam.t, 60.0, 60.0, 40.0, 24.0, 80, 48)
        o = dict(sc.opts, **(opts or {}))
        pr = oracle.project(sc.params, sc.sh_degree, cam, o)
        tgt = np.random.default_rng(5).uniform(0, 1, (3, cam.height, cam.width)).astype(np.float32)
        out = oracle.render(pr, cam, o, target=tgt, want_mag=True)
        t = out["touched"] > 0
        g, m = out["grad2d"][t], out["grad2d_mag"][t]
        assert t.sum() > 20
        assert (m >= np.abs(g)).all()
        assert (m > np.abs(g) * (1 + 1e-9)).any()          # terms do cancel somewhere
        ok, st = parity.grad_report(g, g, m)
        assert ok and st["bad_scaled"] == 0
        # the dense scale bounds the dense gradient as well
        ref = oracle.vjp(sc.params, sc.sh_degree, cam, o, out["grad2d"], out["touched"], pr["clamp"])
        mag = oracle.vjp_mag(sc.params, sc.sh_degree, cam, o, out["grad2d_mag"], out["touched"], pr["clamp"])
        assert (mag >= np.abs(ref) * (1 - 1e-9)).all()
        assert np.array_equal(mag[:, ~t], np.zeros_like(mag[:, ~t]))


def _tiny_reference():
    sc = scenes.make_scene("tiny")
    cam = sc.cameras[0]
    pr = oracle.project(sc.params, 0, cam, sc.opts)
    out = oracle.render(pr, cam, sc.opts, target=sc.target_uniform[0], want_mag=True)
    t = out["touched"] > 0
    ref = oracle.vjp(sc.params, 0, cam, sc.opts, out["grad2d"], out["touched"], pr["clamp"])
    mag = oracle.vjp_mag(sc.params, 0, cam, sc.opts, out["grad2d_mag"], out["touched"], pr["clamp"])
    return out["grad2d"][t], out["grad2d_mag"][t], ref[:, t], mag[:, t]


def test_bar_rejects_dropped_small_entries_at_full_size_scale():
    g, m, d, dm = _tiny_reference()
    # 1e-4: the tiny view's 4096 pixels against 1080p's 2 M, the scale the mean L1 gives there
    for ref, mag, axis in ((g * 1e-4, m * 1e-4, 0), (d * 1e-4, dm * 1e-4, 1)):
        assert np.abs(ref).max() < 1e-5
        small = np.abs(ref) < 1e-2 * np.abs(ref).max(axis=axis, keepdims=True)
        assert small.sum() > 50 and (ref[small] != 0).sum() > 50
        dropped = np.where(small, 0.0, ref)
        ok_lit, st_lit = parity.grad_report(dropped, ref)          # the literal bar alone
        assert ok_lit, st_lit                                     # ... does not see it
        ok, st = parity.grad_report(dropped, ref, mag, axis=axis)
        assert not ok and st["bad_scaled"] > 0, st
        # a sign error on one significant entry
        flip = ref.copy()
        k = np.unravel_index(np.argmax(np.abs(ref)), ref.shape)
        flip[k] = -flip[k]
        assert not parity.grad_report(flip, ref, mag, axis=axis)[0]


def test_bar_accepts_rounding_size_differences():
    g, m, d, dm = _tiny_reference()
    rng = np.random.default_rng(7)
    for ref, mag, axis in ((g, m, 0), (d, dm, 1), (g * 1e-4, m * 1e-4, 0), (d * 1e-4, dm * 1e-4, 1)):
        # what fp32 terms summed in another order leave: up to ~1e-5 of the magnitude sum
        noisy = ref + rng.uniform(-1e-5, 1e-5, ref.shape) * mag
        ok, st = parity.grad_report(noisy, ref, mag, axis=axis)
        assert ok, st
        ok, st = parity.grad_report(ref.astype(np.float32), ref, mag, axis=axis)
        assert ok, st
