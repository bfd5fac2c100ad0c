"""Pins of the oracle's per-tile pruning (ByteSplat, English abstract: pruning that
weighs rendering quality against the per-tile shared-memory budget).

The rule read from the pages: a tile list longer than the budget K keeps its K
most opaque entries, equal opacities going to the nearer (earlier) entry, in
depth order.  The checks characterise that selection without restating it:

- each pruned list has min(len, K) entries and is a subsequence of the
  unpruned one;
- no dropped entry is more opaque than a kept one, and a dropped entry as opaque
  as the least opaque kept one lies behind every kept entry of that opacity
  (with quantised opacities, so such ties occur);
- these three properties leave exactly one valid subset, which a brute-force
  search over all subsets confirms on small lists;
- K at least the longest list changes nothing; the literal per-pixel scan
  prunes to the same image as the per-tile lists;
- gradients through a pruned render equal central finite differences;
- the image error against the unpruned render vanishes once K covers every list.
"""
import itertools

import numpy as np
import pytest

import oracle
from differentiable_rasterizer_gb300 import scenes


def _dense(seed=21, n=4000, quantise=False):
    sc = scenes.random_small_scene(seed, n=n, width=64, height=64, sh_degree=0, log_lo=-3.0, log_hi=-1.8,
                                   logit_mu=1.0, spread=1.2)
    if quantise:
        rng = np.random.default_rng(seed + 1)
        sc.params[10] = rng.choice(np.array([-1.0, 0.0, 0.5, 2.0], np.float32), size=sc.params.shape[1])
    return sc


def _check_selection(full, kept, opac, K):
    assert kept.size == min(full.size, K)
    pos = {g: i for i, g in enumerate(full)}
    kp = np.array([pos[g] for g in kept], np.int64)
    assert np.all(np.diff(kp) > 0), "kept entries out of list order"
    dropped = np.setdiff1d(np.arange(full.size), kp)
    if dropped.size == 0:
        return 0
    ko, do = opac[full[kp]], opac[full[dropped]]
    assert do.max() <= ko.min(), "a dropped entry is more opaque than a kept one"
    tie = ko.min()
    ties_kept = kp[ko == tie]
    ties_dropped = dropped[do == tie]
    if ties_dropped.size:
        assert ties_dropped.min() > ties_kept.max(), "a tie was resolved in favour of the farther entry"
    return int(ties_dropped.size)


@pytest.mark.parametrize("quantise,K", [(False, 100), (False, 333), (True, 150), (True, 37)])
def test_pruned_lists_are_the_most_opaque_nearest_first(quantise, K):
    sc = _dense(quantise=quantise)
    cam = sc.cameras[0]
    pr = oracle.project(sc.params, 0, cam, sc.opts)
    off, ids = oracle.tile_lists(pr, cam)
    offk, idsk = oracle.tile_lists(pr, cam, budget=K)
    opac = pr["rec"][:, 5]
    pruned_tiles = ties = 0
    for t in range(off.size - 1):
        full = ids[off[t]:off[t + 1]]
        kept = idsk[offk[t]:offk[t + 1]]
        ties += _check_selection(full, kept, opac, K)
        pruned_tiles += full.size > K
    assert pruned_tiles >= 4
    if quantise:
        assert ties > 0


def test_the_properties_leave_one_subset_brute_force():
    """On short lists: of all subsets of size K, exactly one satisfies the three
    properties, and it is the oracle's."""
    rng = np.random.default_rng(5)
    checked = 0
    for trial in range(40):
        m = int(rng.integers(4, 10))
        K = int(rng.integers(1, m))
        opac = rng.choice(np.array([0.1, 0.3, 0.3, 0.7, 0.9]), size=m)
        full = np.arange(m)
        valid = []
        for sub in itertools.combinations(range(m), K):
            try:
                _check_selection(full, np.array(sub), opac, K)
                valid.append(sub)
            except AssertionError:
                pass
        assert len(valid) == 1, (opac, K, valid)
        checked += 1
    assert checked == 40


def test_budget_covering_every_list_changes_nothing():
    sc = _dense(n=1500)
    cam = sc.cameras[0]
    pr = oracle.project(sc.params, 0, cam, sc.opts)
    off, ids = oracle.tile_lists(pr, cam)
    K = int(np.diff(off).max())
    offk, idsk = oracle.tile_lists(pr, cam, budget=K)
    assert np.array_equal(off, offk) and np.array_equal(ids, idsk)
    tgt = sc.target_uniform[0]
    a = oracle.render(pr, cam, sc.opts, target=tgt)
    b = oracle.render(pr, cam, dict(sc.opts, tile_budget=K), target=tgt)
    assert np.array_equal(a["image"], b["image"]) and a["loss"] == b["loss"]
    assert np.array_equal(a["grad2d"], b["grad2d"])
    offm, _ = oracle.tile_lists(pr, cam, budget=K - 1)
    assert offm[-1] < off[-1]
    c = oracle.render(pr, cam, dict(sc.opts, tile_budget=K // 4), target=tgt)
    assert not np.array_equal(a["image"], c["image"])


@pytest.mark.parametrize("K", [5, 40])
def test_literal_scan_prunes_like_the_tile_lists(K):
    sc = _dense(n=300, quantise=True)
    cam = sc.cameras[0]
    opts = dict(sc.opts, tile_budget=K)
    pr = oracle.project(sc.params, 0, cam, opts)
    tgt = sc.target_uniform[0]
    a = oracle.render(pr, cam, opts, target=tgt, mode=0, want_sig=True)
    b = oracle.render(pr, cam, opts, target=tgt, mode=1, want_sig=True)
    assert np.array_equal(a["image"], b["image"]) and a["sig"] == b["sig"]
    assert np.array_equal(a["grad2d"], b["grad2d"])


def _loss_sig(params, sc, opts):
    cam = sc.cameras[0]
    pr = oracle.project(params, sc.sh_degree, cam, opts, "f64")
    out = oracle.render(pr, cam, opts, target=sc.target_uniform[0], prec="f64", grads=False, want_sig=True)
    return out["loss"], (out["sig"], pr["clamp"].tobytes())


def test_pruned_render_gradients_match_central_differences():
    sc = scenes.random_small_scene(11, n=8, width=32, height=32, sh_degree=0)
    opts = dict(sc.opts, bg=(0.2, 0.3, 0.4), tile_budget=3)
    cam = sc.cameras[0]
    p0 = sc.params.astype(np.float64)
    pr = oracle.project(p0, 0, cam, opts, "f64")
    off, _ = oracle.tile_lists(pr, cam, "f64")
    assert np.diff(off).max() > 3          # pruning is active
    out = oracle.render(pr, cam, opts, target=sc.target_uniform[0], prec="f64")
    g = oracle.vjp(p0, 0, cam, opts, out["grad2d"], out["touched"], pr["clamp"], prec="f64")
    _, sig0 = _loss_sig(p0, sc, opts)
    checked = nz = 0
    for r in range(p0.shape[0]):
        for i in range(p0.shape[1]):
            h = 1e-6 * max(1.0, abs(p0[r, i]))
            pp = p0.copy(); pp[r, i] += h
            pm = p0.copy(); pm[r, i] -= h
            lp, sp = _loss_sig(pp, sc, opts)
            lm, sm = _loss_sig(pm, sc, opts)
            if sp != sig0 or sm != sig0:
                continue
            fd = (lp - lm) / (2 * h)
            checked += 1
            nz += abs(fd) > 1e-8
            assert abs(g[r, i] - fd) <= 1e-6 * abs(fd) + 1e-9, (r, i, g[r, i], fd)
    assert checked >= 0.7 * p0.size and nz >= 0.3 * checked   # pruned-away Gaussians have none


def test_error_against_the_unpruned_render_vanishes_with_a_large_budget():
    sc = _dense(n=2000)
    cam = sc.cameras[0]
    pr = oracle.project(sc.params, 0, cam, sc.opts)
    off, _ = oracle.tile_lists(pr, cam)
    ref = oracle.render(pr, cam, sc.opts)["image"]
    errs = []
    for K in (50, 200, int(np.diff(off).max())):
        img = oracle.render(pr, cam, dict(sc.opts, tile_budget=K))["image"]
        errs.append(float(np.abs(img.astype(np.float64) - ref).max()))
    assert errs[0] > 0 and errs[-1] == 0.0
