"""GPU parity of per-tile pruning (gs_prune_tiles) against the oracle's pruned
lists, then the whole step on those lists: dense lists with distinct and with
quantised (tied) opacities, a single tile list long enough for the re-gathering
path, several views, and a budget that covers every list (nothing changes).
Rendering quality is measured against the unpruned oracle render."""
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


def _dense(seed=21, n=4000, quantise=False):
    sc = scenes.random_small_scene(seed, n=n, width=64, height=64, sh_degree=0, log_lo=-3.0, log_hi=-1.8,
                                   logit_mu=1.0, spread=1.2)
    if quantise:
        rng = np.random.default_rng(seed + 1)
        sc.params[10] = rng.choice(np.array([-1.0, 0.0, 0.5, 2.0], np.float32), size=sc.params.shape[1])
    return sc


@pytest.mark.parametrize("quantise,K", [(False, 100), (False, 333), (True, 150), (True, 37)])
def test_pruned_step_matches_the_oracle(quantise, K):
    sc = _dense(quantise=quantise)
    sc.opts = dict(sc.opts, tile_budget=K)
    st = parity.run_stage_parity(sc)
    assert sum(st["pruned_tiles"]) >= 4


def test_long_list_regathers_opacities():
    """One 16x16 tile with 20000 entries: longer than the shared-memory cache of
    opacities, so every radix pass gathers them again."""
    sc = scenes.random_small_scene(32, n=20000, width=16, height=16, sh_degree=0, log_lo=-2.0, log_hi=-1.0,
                                   logit_mu=-3.0, spread=0.3)
    sc.opts = dict(sc.opts, tile_budget=9000)
    st = parity.run_stage_parity(sc)
    assert st["instances"] > 16384 and st["pruned_entries"][0] > 0


def test_pruned_multi_view_degree3():
    sc = scenes.make_scene("medium", n=20000)
    cams = []
    for k, ang in enumerate((-0.1, 0.0, 0.12)):
        c, s = math.cos(ang), math.sin(ang)
        R = np.array([[c, 0, s], [0, 1, 0], [-s, 0, c]], np.float32)
        cams.append(scenes.Camera(R, np.array([0.5 * k, 0.2, 0.0], np.float32), 300.0, 300.0, 160.0, 90.0, 320, 180))
    sc.cameras = cams
    sc.opts = dict(sc.opts, tile_budget=64)
    st = parity.run_stage_parity(sc)
    assert min(st["pruned_tiles"]) > 0


def test_budget_covering_every_list_is_the_unpruned_step():
    sc = _dense(n=2000)
    tgt = torch.from_numpy(parity.oracle_targets(sc)).cuda()
    out = []
    for budget in (None, 10 ** 6):
        tr = pipeline.GaussianTrainer(sc.params, sc.sh_degree, sc.cameras, sc.opts, sc.lr, tile_budget=budget)
        tr.project()
        tr.bin_sort()
        tr.raster(tgt)
        torch.cuda.synchronize()
        out.append((tr.image.cpu().numpy(), tr.ranges.cpu().numpy(), tr.touched.cpu().numpy()))
    assert np.array_equal(out[0][1], out[1][1])
    assert np.array_equal(parity.bits(out[0][0]), parity.bits(out[1][0]))
    assert np.array_equal(out[0][2], out[1][2])


def test_quality_against_the_unpruned_oracle():
    """PSNR of the pruned GPU render against the unpruned oracle render rises with
    the budget and is exact once the budget covers every list."""
    sc = _dense(n=4000)
    cam = sc.cameras[0]
    ref = oracle.render(oracle.project(sc.params, 0, cam, sc.opts), cam, sc.opts)["image"].astype(np.float64)
    off, _ = oracle.tile_lists(oracle.project(sc.params, 0, cam, sc.opts), cam)
    psnr = []
    for K in (64, 256, 768, int(np.diff(off).max())):
        tr = pipeline.GaussianTrainer(sc.params, 0, sc.cameras, sc.opts, sc.lr, tile_budget=K)
        img = tr.render().cpu().numpy().astype(np.float64)
        mse = float(((img - ref) ** 2).mean())
        psnr.append(math.inf if mse <= 1e-20 else 10 * math.log10(1.0 / mse))
    print(f"[prune quality] PSNR vs unpruned oracle at budgets 64/256/768/max: {psnr}")
    assert psnr[0] < psnr[1] <= psnr[2] and psnr[-1] > 90
