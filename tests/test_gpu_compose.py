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


def _splits(sc, S):
    """Per view: S - 1 fp32 depth quantiles of the visible Gaussians."""
    out = []
    for cam in sc.cameras:
        pr = oracle.project(sc.params, sc.sh_degree, cam, sc.opts)
        d = pr["rec"][pr["visible"] > 0, 9].astype(np.float64)
        z = np.unique(np.quantile(d, np.arange(1, S) / S).astype(np.float32)) if S > 1 else np.zeros(0, np.float32)
        assert z.size == S - 1
        out.append([float(x) for x in z])
    return out


def run_compose_parity(sc, S):
    splits = _splits(sc, S)
    tr = pipeline.GaussianTrainer(sc.params, sc.sh_degree, sc.cameras, sc.opts, sc.lr)
    img = tr.render_partial(splits).clone()
    torch.cuda.synchronize()
    cparts = tr.c_parts.cpu().numpy()
    tparts = tr.t_parts.cpu().numpy()
    sub = tr.sub_ranges.cpu().numpy().view(np.uint32).reshape(S, sc.n_views, -1, 2)
    ids = tr.ids.cpu().numpy().view(np.uint32)
    tcomp = tr.t_composed.cpu().numpy()
    img = img.cpu().numpy()
    stats = {}
    for v, cam in enumerate(sc.cameras):
        pr = oracle.project(sc.params, sc.sh_degree, cam, sc.opts)
        parts = oracle.render_subsets(pr, cam, sc.opts, splits[v])
        z = np.concatenate([[-np.inf], np.asarray(splits[v], np.float64), [np.inf]])
        depth = pr["rec"][:, 9].astype(np.float64)
        for s in range(S):
            # the slab's tile lists
            slab = dict(pr, visible=(pr["visible"].astype(bool) & (depth >= z[s]) & (depth < z[s + 1])).astype(np.uint8))
            off, oids = oracle.tile_lists(slab, cam)
            r = sub[s, v].astype(np.int64)
            assert np.array_equal(r[:, 1] - r[:, 0], np.diff(off)), f"view {v} slab {s}: sub-range lengths"
            pos = np.repeat(r[:, 0] - off[:-1], np.diff(off)) + np.arange(off[-1])
            assert np.array_equal(ids[pos], oids.astype(np.uint32)), f"view {v} slab {s}: sub-range ids"
            if s + 1 < S:
                assert np.array_equal(r[:, 1], sub[s + 1, v][:, 0]), "slabs must tile the list"
            # the slab's partial render
            Cs, Ts = parts[s]
            assert np.abs(cparts[s, v].astype(np.float64) - Cs).max() <= parity.IMG_ATOL, f"view {v} slab {s}: C"
            assert np.abs(tparts[s, v].astype(np.float64) - Ts).max() <= 1e-6, f"view {v} slab {s}: T"
        C, T = oracle.compose(parts, sc.opts["bg"])
        d = np.abs(img[v].astype(np.float64) - C)
        assert d.max() <= parity.IMG_ATOL, f"view {v}: composed image {d.max()}"
        assert np.abs(tcomp[v] - T).max() <= 1e-6
        one = oracle.render(pr, cam, sc.opts)["image"].astype(np.float64)
        cmax = max(float(pr["rec"][pr["visible"] > 0, 6:9].max(initial=0.0)), max(sc.opts["bg"]))
        # T where a pixel stops: below t_min, or (crossing entry excluded) below t_min / (1 - alpha_max)
        t_stop = sc.opts["t_min"] / ((1.0 - sc.opts["alpha_max"]) if sc.opts.get("exclude_crossing") else 1.0)
        d1 = np.abs(img[v].astype(np.float64) - one)
        assert d1.max() <= t_stop * cmax + parity.IMG_ATOL, f"view {v}: vs one pass {d1.max()}"
        stats.setdefault("vs_one_pass_max", []).append(float(d1.max()))
        stats.setdefault("vs_compose_max", []).append(float(d.max()))
    print(f"[compose parity] {sc.name} S={S}: {stats}")
    return stats


def _dense():
    sc = scenes.random_small_scene(21, n=4000, width=64, height=64, sh_degree=0, log_lo=-3.0, log_hi=-1.8,
                                   logit_mu=1.0, spread=1.2)
    sc.opts = dict(sc.opts, bg=(0.2, 0.5, 0.8))
    return sc


@pytest.mark.parametrize("S", [1, 2, 3])
def test_compose_tiny(S):
    run_compose_parity(scenes.make_scene("tiny"), S)


@pytest.mark.parametrize("S", [2, 4, 8])
def test_compose_dense_lists_with_background(S):
    run_compose_parity(_dense(), S)


def test_compose_ragged_resolution():
    sc = scenes.make_scene("tiny")
    cam = sc.cameras[0]
    sc.cameras = [scenes.Camera(cam.R, cam.t, 64.0, 64.0, 35.0, 22.5, 70, 45)]
    run_compose_parity(sc, 3)


def test_compose_multi_view_degree3():
    sc = scenes.make_scene("medium", n=20000)
    cams = []
    for k, ang in enumerate((-0.1, 0.0, 0.12)):
        c, s = math.cos(ang), math.sin(ang)
        R = np.array([[c, 0, s], [0, 1, 0], [-s, 0, c]], np.float32)
        cams.append(scenes.Camera(R, np.array([0.5 * k, 0.2, 0.0], np.float32), 300.0, 300.0, 160.0, 90.0, 320, 180))
    sc.cameras = cams
    sc.opts = dict(sc.opts, exclude_crossing=1, bg=(0.1, 0.4, 0.7))
    run_compose_parity(sc, 3)


def test_one_slab_matches_the_one_pass_gpu_render():
    sc = _dense()
    tr = pipeline.GaussianTrainer(sc.params, 0, sc.cameras, sc.opts, sc.lr)
    a = tr.render().clone()
    b = tr.render_partial([[]]).clone()
    torch.cuda.synchronize()
    # one pass adds T * bg rounded after the product, the composition with one fma
    assert (a - b).abs().max().item() <= 1e-6
