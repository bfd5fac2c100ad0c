"""GPU parity: the CUDA path through the C ABI against the CPU oracle, stage by
stage, on seeded inputs (tiny, ragged, dense lists, every bucket-sort size class
including multi-level key-range splits, a view binned in two tile-row bands,
multi-view with RGB and with SH 3, degree-3, small, medium), plus edge cases (no
Gaussians, everything culled, instance capacity growth), the deferred Adam with
catch-up and flush, several training steps, and the pipelined host-input steps."""
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


def _variant(sc, **kw):
    sc.opts = dict(sc.opts, **kw)
    return sc


def test_tiny():
    parity.run_stage_parity(scenes.make_scene("tiny"))


def test_tiny_exclude_crossing_and_background():
    parity.run_stage_parity(_variant(scenes.make_scene("tiny"), exclude_crossing=1, bg=(0.25, 0.5, 0.75)))


def test_ragged_resolution_partial_tiles():
    sc = scenes.make_scene("tiny")
    cam = sc.cameras[0]
    sc.cameras = [scenes.Camera(cam.R, cam.t, 64.0, 64.0, 35.0, 22.5, 70, 45)]
    sc.target_uniform = np.random.default_rng(9).uniform(0, 1, (1, 3, 45, 70)).astype(np.float32)
    parity.run_stage_parity(sc)


def test_dense_lists_span_several_chunks_and_stop_early():
    """~4000 large, fairly opaque Gaussians on 64x64: tile lists longer than one
    shared-memory chunk, many pixels reach T < 1e-4 mid-list."""
    sc = scenes.random_small_scene(21, n=4000, width=64, height=64, sh_degree=0, log_lo=-3.0, log_hi=-1.8,
                                   logit_mu=1.0, spread=1.2)
    st = parity.run_stage_parity(sc)
    assert st["instances"] > 16 * 600
    assert st["e_fwd"] < st["instances"] * 256   # early stops happened


def _border_scene(seed, sh_degree):
    """Gaussians placed where the per-tile candidate masks have their edge cases:
    tiny ones centred on tile-border pixel centres and tile corners (boxes that
    start or end exactly at a tile edge, or cover a single pixel), ones whose
    support spans a whole tile or the whole view (boxes 0..16 in both axes), thin
    rotated ones crossing borders diagonally, and opacities from just above the
    1/255 cut to the 0.99 clamp."""
    rng = np.random.default_rng(seed)
    W = H = 64
    fx, z = 64.0, 2.0
    groups = []
    # tiny: centre u = 16 k + {-0.5, 0, 0.5} on one axis or both (tile corners)
    for _ in range(300):
        k = rng.integers(1, 4, size=2)
        off = rng.choice([-0.5, 0.0, 0.5], size=2)
        u = np.where(rng.random(2) < 0.7, 16.0 * k + off, rng.uniform(0.5, 63.5, 2))
        groups.append((u, rng.uniform(-7.5, -5.5, 3), rng.normal(size=4)))
    # spanning a tile or the view
    for _ in range(40):
        groups.append((rng.uniform(0, 64, 2), rng.uniform(-1.8, -0.8, 3), rng.normal(size=4)))
    # thin and rotated
    for _ in range(160):
        ls = np.array([rng.uniform(-2.6, -2.0), rng.uniform(-6.5, -5.5), rng.uniform(-6.5, -5.5)])
        groups.append((16.0 * rng.integers(1, 4, size=2) + rng.uniform(-3, 3, 2), ls, rng.normal(size=4)))
    n = len(groups)
    P = 14 if sh_degree == 0 else 59
    params = np.zeros((P, n), np.float32)
    for i, (u, ls, q) in enumerate(groups):
        zi = z + rng.uniform(0.0, 1.5)
        params[0, i] = (u[0] - 32.0) * zi / fx
        params[1, i] = (u[1] - 32.0) * zi / fx
        params[2, i] = zi
        params[3:6, i] = ls
        params[6:10, i] = q / np.linalg.norm(q)
    params[10] = rng.choice([-5.4, -2.0, 0.0, 2.0, 6.0], size=n) + rng.normal(0, 0.05, n)
    if sh_degree == 0:
        params[11:14] = rng.uniform(0, 1, (3, n))
    else:
        params[11:14] = rng.uniform(-1.7, 1.7, (3, n))
        params[14:59] = rng.normal(0, 0.2, (45, n))
    cam = scenes.Camera(np.eye(3, dtype=np.float32), np.zeros(3, np.float32), fx, fx, 32.0, 32.0, W, H)
    target = rng.uniform(0, 1, (1, 3, H, W)).astype(np.float32)
    return scenes.Scene("tile-borders", params, sh_degree, [cam], "uniform", target, None, scenes.DEFAULT_LR,
                        dict(scenes.DEFAULT_OPTS))


@pytest.mark.parametrize("sh", [0, 3])
def test_gaussians_on_tile_borders_corners_and_spanning_tiles(sh):
    st = parity.run_stage_parity(_border_scene(40 + sh, sh))
    assert st["instances"] > 500


def test_saved_pass_bits_scratch_gives_the_recomputed_results():
    """The fused raster with its saved-pass-bits scratch -- covering every list,
    covering half of the list positions, absent -- renders the same image and
    gives the same E counts and touched sets, and grad2d up to the atomics'
    summation order; with the whole scratch no chunk's bits are recomputed."""
    from differentiable_rasterizer_gb300 import abi
    sc = scenes.random_small_scene(23, n=6000, width=64, height=64, sh_degree=0, log_lo=-3.0, log_hi=-1.8,
                                   logit_mu=-2.0, spread=1.2)
    tr = pipeline.GaussianTrainer(sc.params, sc.sh_degree, sc.cameras, sc.opts, sc.lr)
    target = torch.from_numpy(sc.target_uniform).cuda()
    tr.project()
    tr.bin_sort()
    lens = np.diff(tr.ranges.cpu().numpy().view(np.uint32).reshape(-1, 2), axis=1)
    assert lens.max() > 4 * 256   # chunks evicted from the three-chunk ring
    n_inst = tr.n_instances

    def run(ws, words):
        tr.grad2d.zero_()
        tr.touched.zero_()
        tr.eval_counts.zero_()
        abi.gs_raster_fused_fwd_bwd(tr.proj, tr.n, tr.ranges.data_ptr(), tr.ids.data_ptr(), tr.cams, tr.V, tr.opts,
                                    target.data_ptr(), tr.image.data_ptr(), tr.loss.data_ptr(),
                                    tr.grad2d.data_ptr(), tr.touched.data_ptr(), tr.eval_counts.data_ptr(),
                                    tr.stream_handle(), ws, words)
        torch.cuda.synchronize()
        out = {k: getattr(tr, k).clone() for k in ("image", "loss", "grad2d", "touched", "eval_counts")}
        work = torch.zeros(abi.GS_RASTER_WORK_COUNTERS, dtype=torch.int64, device="cuda")
        tr.grad2d.zero_()
        tr.touched.zero_()
        abi.gs_raster_work_counts(tr.proj, tr.n, tr.ranges.data_ptr(), tr.ids.data_ptr(), tr.cams, tr.V, tr.opts,
                                  target.data_ptr(), tr.image.data_ptr(), tr.loss.data_ptr(), tr.grad2d.data_ptr(),
                                  tr.touched.data_ptr(), work.data_ptr(), tr.stream_handle(), ws, words)
        out["work"] = dict(zip(abi.RASTER_WORK_NAMES, work.cpu().tolist()))
        return out

    lists = tr.V * tr.tiles
    full = run(tr.bits_ws.data_ptr(), abi.raster_bits_ws_words(n_inst, lists))
    half = run(tr.bits_ws.data_ptr(), abi.raster_bits_ws_words(n_inst // 2, lists // 2))
    none = run(None, 0)
    assert none["work"]["recomputed_chunks"] > half["work"]["recomputed_chunks"] > full["work"]["recomputed_chunks"] == 0
    for got in (half, none):
        for k in ("image", "touched", "eval_counts"):
            assert torch.equal(got[k], full[k]), k
        g, f = got["grad2d"].double(), full["grad2d"].double()
        assert float((g - f).abs().max()) <= 1e-5 * float(f.abs().max())
        assert abs(float(got["loss"][0]) - float(full["loss"][0])) <= 1e-12 * abs(float(full["loss"][0]))


def test_sort_bucket_sizes_over_2048_use_the_large_block_sort():
    """~6000 wide Gaussians on a 32x32 view: 4 tile buckets of ~6000 instances."""
    sc = scenes.random_small_scene(31, n=6000, width=32, height=32, sh_degree=0, log_lo=-1.5, log_hi=-1.0,
                                   logit_mu=-2.0, spread=0.6)
    st = parity.run_stage_parity(sc)
    assert st["instances"] > 4 * 2048


def test_sort_bucket_over_16384_is_split_by_key_range():
    """20000 Gaussians on one 16x16 tile: a single bucket larger than a block sort
    holds, split into sub-buckets by key range."""
    sc = scenes.random_small_scene(32, n=20000, width=16, height=16, sh_degree=0, log_lo=-2.0, log_hi=-1.0,
                                   logit_mu=-3.0, spread=0.3)
    st = parity.run_stage_parity(sc)
    assert st["instances"] > 16384


def test_sort_split_recursion_on_equal_depths():
    """40001 Gaussians on one tile: 20000 at depth exactly 2, 10000 at each of the
    next two float32 values, one at depth 100.  The first split puts the 40000 near
    ones in one sub-bucket, the second separates the three depths (two sub-buckets
    of 10000 go to the block sort), the third splits the 20000 of equal depth by
    index."""
    n = 40001
    sc = scenes.random_small_scene(34, n=n, width=16, height=16, sh_degree=0, log_lo=-2.0, log_hi=-1.0,
                                   logit_mu=-3.0, spread=0.3)
    z = np.full(n, 2.0, np.float32)
    z1 = np.nextafter(np.float32(2.0), np.float32(3.0))
    z[20000:30000] = z1
    z[30000:40000] = np.nextafter(z1, np.float32(3.0))
    z[40000] = 100.0
    sc.params[2] = z[np.random.default_rng(5).permutation(n)]
    st = parity.run_stage_parity(sc)
    assert st["instances"] == n


@pytest.mark.parametrize("n", [1500, 6000])
def test_sort_slices_with_clustered_depths_fall_back_to_the_block_sort(n):
    """One 16x16 tile holding n instances (a 257-2048 and a 2049-8192 bucket) whose
    depths sit in two tight clusters plus a far outlier: the key-range slices put
    most keys in a slice too large for a warp, so the bucket goes to the block's
    bitonic network; equal depths are ordered by index."""
    sc = scenes.random_small_scene(35, n=n, width=16, height=16, sh_degree=0, log_lo=-2.0, log_hi=-1.0,
                                   logit_mu=-3.0, spread=0.3)
    rng = np.random.default_rng(6)
    z = np.where(rng.uniform(size=n) < 0.5, np.float32(3.0), np.float32(3.0001)).astype(np.float32)
    z[: n // 10] = np.float32(3.0)            # ties broken by index
    z[-1] = np.float32(50.0)                  # stretches the key interval
    sc.params[2] = z
    st = parity.run_stage_parity(sc)
    assert st["instances"] == n


def test_sort_slices_spread_over_warps_and_threads():
    """One tile of 1900 instances with depths spread over a wide interval but a
    dense band holding ~200 of them: slices of one key (threads), of tens (warps)
    and empty ones in one bucket."""
    n = 1900
    sc = scenes.random_small_scene(36, n=n, width=16, height=16, sh_degree=0, log_lo=-2.0, log_hi=-1.0,
                                   logit_mu=-3.0, spread=0.3)
    rng = np.random.default_rng(7)
    z = rng.uniform(2.0, 40.0, n).astype(np.float32)
    z[:200] = rng.uniform(10.0, 10.05, 200).astype(np.float32)
    sc.params[2] = z
    st = parity.run_stage_parity(sc)
    assert st["instances"] == n


def test_wide_view_bins_in_two_tile_row_bands():
    """An 8192x1296 view has 512 x 81 tiles, more than one block's shared-memory
    counters hold: the binning runs in two bands of tile rows (80 + 1).  The
    Gaussians sit across the band boundary."""
    sc = scenes.random_small_scene(35, n=3000, width=8192, height=1296, sh_degree=0, log_lo=-2.5, log_hi=-1.5,
                                   spread=1.2)
    cam = sc.cameras[0]
    sc.cameras = [scenes.Camera(cam.R, cam.t, 1000.0, 1000.0, 4096.0, 1280.0, 8192, 1296)]
    st = parity.run_stage_parity(sc)
    assert st["instances"] > 3000


def test_multi_view_small_reduced():
    sc = scenes.make_scene("small", n=20000)
    base = sc.cameras[0]
    cams = []
    for k, ang in enumerate((-0.15, 0.0, 0.2)):
        c, s = math.cos(ang), math.sin(ang)
        R = np.array([[c, 0, s], [0, 1, 0], [-s, 0, c]], np.float32)
        cams.append(scenes.Camera(R, np.array([0.3 * k, 0, 0.5], np.float32), 250.0, 250.0, 160.0, 90.0, 320, 180))
    sc.cameras = cams
    parity.run_stage_parity(sc)


def test_multi_view_degree3_exclude_crossing_background():
    """Three views of the SH-3 medium recipe at reduced size, with the crossing
    Gaussian excluded at the stop and a non-zero background."""
    sc = scenes.make_scene("medium", n=20000)
    cams = []
    for k, ang in enumerate((-0.1, 0.0, 0.12)):
        c, s = math.cos(ang), math.sin(ang)
        R = np.array([[c, 0, s], [0, 1, 0], [-s, 0, c]], np.float32)
        cams.append(scenes.Camera(R, np.array([0.5 * k, 0.2, 0.0], np.float32), 300.0, 300.0, 160.0, 90.0, 320, 180))
    sc.cameras = cams
    sc.opts = dict(sc.opts, exclude_crossing=1, bg=(0.1, 0.4, 0.7))
    st = parity.run_stage_parity(sc)
    assert st["instances"] > 0


def test_degree3_medium_recipe_reduced():
    sc = scenes.make_scene("medium", n=60000)
    c = sc.cameras[0]
    sc.cameras = [scenes.Camera(c.R, c.t, 350.0, 350.0, 240.0, 135.0, 480, 270)]
    parity.run_stage_parity(sc)


def test_small_full():
    parity.run_stage_parity(scenes.make_scene("small"))


@pytest.mark.slow
def test_medium_full():
    parity.run_stage_parity(scenes.make_scene("medium"))


def test_no_gaussians_and_all_culled():
    sc = scenes.make_scene("tiny", n=1)
    sc.params = sc.params[:, :0].copy()
    tr = pipeline.GaussianTrainer(sc.params, 0, sc.cameras, _variant(sc, bg=(0.1, 0.2, 0.3)).opts, sc.lr)
    tgt = torch.zeros((1, 3, 64, 64), device="cuda")
    tr.train_step(tgt)
    torch.cuda.synchronize()
    img = tr.image.cpu().numpy()
    assert np.allclose(img[0, 0], 0.1) and np.allclose(img[0, 2], 0.3)
    assert tr.n_instances == 0
    # everything behind the camera
    sc = scenes.make_scene("tiny")
    sc.params[2] = -3.0
    tr = pipeline.GaussianTrainer(sc.params, 0, sc.cameras, sc.opts, sc.lr)
    tr.train_step(torch.from_numpy(sc.target_uniform).cuda())
    torch.cuda.synchronize()
    assert tr.n_instances == 0 and tr.n_idx.cpu().numpy().sum() == 0
    assert np.array_equal(tr.rows(tr.params).cpu().numpy(), sc.params)


def test_capacity_growth_retries():
    sc = scenes.make_scene("tiny")
    tr = pipeline.GaussianTrainer(sc.params, 0, sc.cameras, sc.opts, sc.lr, capacity=16)
    tr.project()
    cnt = tr.bin_sort()
    assert tr.capacity >= cnt > 16
    off, ids = oracle.tile_lists(oracle.project(sc.params, 0, sc.cameras[0], sc.opts), sc.cameras[0])
    assert cnt == ids.size
    assert np.array_equal(tr.ids[:cnt].cpu().numpy().view(np.uint32), ids.astype(np.uint32))


def test_adam_deferred_catch_up_and_flush_bitexact():
    rng = np.random.default_rng(5)
    n, sh = 5000, 3
    P = scenes.PARAM_ROWS[sh]
    p0 = rng.standard_normal((P, n)).astype(np.float32)
    lr = (1e-3, 2e-3, 3e-3, 4e-2, 5e-3)
    lr_rows = scenes.lr_rows(lr, sh)
    cams = scenes.make_scene("tiny").cameras
    tr = pipeline.GaussianTrainer(p0, sh, cams, dict(scenes.DEFAULT_OPTS), lr)
    po, mo, vo = p0.copy(), np.zeros_like(p0), np.zeros_like(p0)
    lo = np.zeros(n, np.int32)
    for t in range(1, 9):
        mask = rng.uniform(size=n) < (0.02 if t < 6 else 0.5)
        idx = np.flatnonzero(mask).astype(np.uint32)
        g = (rng.standard_normal((P, n)) * mask).astype(np.float32)
        tr.grads.copy_(tr.to_device_layout(g))
        tr.idx[tr.V, :idx.size].copy_(torch.from_numpy(idx.view(np.int32)))
        tr.n_idx[tr.V] = idx.size
        tr.adam(t)
        go = g.copy()
        oracle.adam_deferred(po, mo, vo, go, lo, lr_rows, idx, t, 0.9, 0.999, 1e-8)
    torch.cuda.synchronize()
    assert np.array_equal(parity.bits(tr.rows(tr.params).cpu().numpy()), parity.bits(po))
    assert np.array_equal(parity.bits(tr.rows(tr.adam_m).cpu().numpy()), parity.bits(mo))
    assert np.array_equal(tr.last_step.cpu().numpy(), lo)
    tr.adam(8, flush=True)
    oracle.adam_deferred(po, mo, vo, go, lo, lr_rows, None, 8, 0.9, 0.999, 1e-8, flush=True)
    torch.cuda.synchronize()
    assert np.array_equal(parity.bits(tr.rows(tr.params).cpu().numpy()), parity.bits(po))
    assert np.array_equal(parity.bits(tr.rows(tr.adam_v).cpu().numpy()), parity.bits(vo))
    assert (tr.last_step.cpu().numpy() == 8).all()


def test_three_training_steps_track_the_oracle():
    """Step t+1 checked against the oracle started from the GPU's state after step t."""
    sc = scenes.make_scene("small", n=20000)
    c = sc.cameras[0]
    sc.cameras = [scenes.Camera(c.R, c.t, 250.0, 250.0, 160.0, 90.0, 320, 180)]
    targets = parity.oracle_targets(sc)
    tr = pipeline.GaussianTrainer(sc.params, 0, sc.cameras, sc.opts, sc.lr)
    tgt = torch.from_numpy(targets).cuda()
    for step in range(3):
        p_before = tr.rows(tr.params).cpu().numpy()
        tr.train_step(tgt)
        torch.cuda.synchronize()
        pr = oracle.project(p_before, 0, sc.cameras[0], sc.opts)
        out = oracle.render(pr, sc.cameras[0], sc.opts, target=targets[0])
        assert np.abs(tr.image.cpu().numpy()[0] - out["image"]).max() <= parity.IMG_ATOL
        assert abs(tr.loss.item() - out["loss"]) <= 1e-9
        assert tr.last_step.cpu().numpy().max() == step + 1
    # deferred state equals dense after a flush: every Gaussian reaches step 3
    tr.flush()
    torch.cuda.synchronize()
    assert (tr.last_step.cpu().numpy() == 3).all()


@pytest.mark.parametrize("sh_degree", [0, 3])
def test_maximum_view_count(sh_degree):
    """GS_MAX_VIEWS (32) views of a small scene in one step: every per-view
    stage and the union over all of them (SH 3: the decode whose geometry and
    colour halves run in different warps, with every view bit in use)."""
    sc = scenes.random_small_scene(51, n=400, width=40, height=24, sh_degree=sh_degree, log_lo=-3.0, log_hi=-2.0)
    cams = []
    for k in range(32):
        ang = -0.3 + 0.6 * k / 31
        c, s = math.cos(ang), math.sin(ang)
        R = np.array([[c, 0, s], [0, 1, 0], [-s, 0, c]], np.float32)
        cams.append(scenes.Camera(R, np.array([0.05 * (k % 4), 0.0, 0.1 * (k // 16)], np.float32), 40.0, 40.0,
                                  20.0, 12.0, 40, 24))
    sc.cameras = cams
    sc.target_uniform = np.random.default_rng(52).uniform(0, 1, (32, 3, 24, 40)).astype(np.float32)
    st = parity.run_stage_parity(sc)
    assert len(st["visible"]) == 32 and min(st["visible"]) > 0


def test_pipelined_host_steps_match_device_steps():
    """train_steps_host (targets copied in on a second stream, one step ahead) gives
    the same losses as device-resident steps, and leaves each step's loss in its row."""
    sc = scenes.make_scene("tiny")
    tgt = torch.from_numpy(np.ascontiguousarray(sc.target_uniform, np.float32))
    a = pipeline.GaussianTrainer(sc.params, sc.sh_degree, sc.cameras, sc.opts, sc.lr)
    b = pipeline.GaussianTrainer(sc.params, sc.sh_degree, sc.cameras, sc.opts, sc.lr)
    dev = tgt.cuda()
    ref = [a.train_step(dev).cpu().numpy().copy() for _ in range(4)]
    host = tgt.pin_memory()
    loss = torch.empty((4, 1), dtype=torch.float64).pin_memory()
    b.train_steps_host([host] * 4, loss)
    torch.cuda.synchronize()
    got = loss.numpy()
    assert abs(got[0, 0] - ref[0][0]) <= 1e-9 * abs(ref[0][0])
    for k in range(1, 4):
        assert abs(got[k, 0] - ref[k][0]) <= 1e-5 * abs(ref[k][0]), (k, got[k, 0], ref[k][0])
    assert b.t == 4


@pytest.mark.parametrize("seed", [101, 102, 103, 104, 105, 106])
def test_randomised_configurations(seed):
    """Seeded random configurations: Gaussian count, a resolution that is not a
    multiple of 16, SH degree 0 or 3, 1-3 views, either stop variant and a random
    background; every stage compared as in the fixed cases."""
    rng = np.random.default_rng(seed)
    sh = int(rng.choice([0, 3]))
    n = int(rng.integers(500, 6000))
    W, H = int(rng.integers(40, 200)), int(rng.integers(30, 150))
    sc = scenes.random_small_scene(seed, n=n, width=W, height=H, sh_degree=sh, log_lo=float(rng.uniform(-4.0, -2.5)),
                                   log_hi=float(rng.uniform(-2.3, -1.2)), logit_mu=float(rng.uniform(-1.0, 1.5)),
                                   spread=float(rng.uniform(0.4, 1.4)))
    views = int(rng.integers(1, 4))
    base = sc.cameras[0]
    cams = []
    for k in range(views):
        ang = 0.08 * (k - (views - 1) / 2)
        c, s = math.cos(ang), math.sin(ang)
        R = np.array([[c, 0, s], [0, 1, 0], [-s, 0, c]], np.float32)
        cams.append(scenes.Camera(R, np.array([0.05 * k, 0.0, 0.0], np.float32), base.fx, base.fy, base.cx, base.cy,
                                  W, H))
    sc.cameras = cams
    sc.target_uniform = rng.uniform(0, 1, (views, 3, H, W)).astype(np.float32)
    sc.opts = dict(sc.opts, exclude_crossing=int(rng.integers(0, 2)), bg=tuple(float(x) for x in rng.uniform(0, 1, 3)))
    parity.run_stage_parity(sc)


def _corrupt_rows(sc, seed):
    """Rows of the scene's parameters made non-finite or degenerate, one kind per row:
    NaN / +inf means, NaN / +inf log-scales, zero, NaN and +inf quaternions, NaN
    logits, NaN / +inf colours (degree 3: DC coefficients); degree 3 also gets -inf
    higher-band coefficients (a colour clamped at 0: visible on both sides)."""
    rng = np.random.default_rng(seed)
    p = sc.params.copy()
    kinds = [(0, np.nan), (1, np.inf), (2, np.nan), (3, np.nan), (4, np.inf), ("q", 0.0), ("q", np.nan),
             ("q", np.inf), (10, np.nan), (11, np.nan), (12, np.inf)]
    rows = rng.choice(p.shape[1], 4 * len(kinds), replace=False)
    culled = []
    for i, g in enumerate(rows):
        what, val = kinds[i % len(kinds)]
        if what == "q":
            p[6:10, g] = val
        else:
            p[what, g] = val
        culled.append(g)
    clamped = []
    if sc.sh_degree == 3:
        extra = rng.choice(np.setdiff1d(np.arange(p.shape[1]), rows), 40, replace=False)
        p[11 + 3 * 5, extra] = -np.inf
        clamped = list(extra)
    sc.params = p
    return np.asarray(culled), np.asarray(clamped, np.int64)


@pytest.mark.parametrize("sh", [0, 3])
def test_non_finite_and_degenerate_rows_are_culled_as_the_oracle_culls_them(sh):
    """NaN / inf parameters and zero quaternions go through projection, binning,
    raster, compaction and Adam on the GPU exactly as through the oracle: the rows
    culled there (and only those) are culled here, every other output compared as
    usual, and the culled rows' parameters come out of Adam untouched."""
    if sh == 0:
        sc = scenes.make_scene("tiny")
    else:
        sc = scenes.make_scene("medium", n=20000)
        c = sc.cameras[0]
        sc.cameras = [scenes.Camera(c.R, c.t, 350.0, 350.0, 240.0, 135.0, 480, 270)]
        sc.target_kind = "uniform"
        sc.target_uniform = np.random.default_rng(9).uniform(0, 1, (1, 3, 270, 480)).astype(np.float32)
    culled, clamped = _corrupt_rows(sc, 30 + sh)
    pr = oracle.project(sc.params, sc.sh_degree, sc.cameras[0], sc.opts)
    assert not pr["visible"][culled].any()
    if clamped.size:
        assert pr["visible"][clamped].sum() > 10 and (pr["clamp"][clamped][pr["visible"][clamped] > 0] > 0).all()
    st = parity.run_stage_parity(sc)
    assert st["visible"][0] > 0


def test_checkpoint_resume_reproduces_the_next_step(tmp_path):
    """Three steps, a checkpoint (state_dict flushes the deferred Adam states, then
    copies; saved to disk), then step 4 two ways: in the same trainer, and in a
    fresh trainer loaded from the file.  The loaded state is the saved one bit for
    bit, and so is everything step 4 decides (records, lists, image, counts,
    touched and union lists).  The loss and the gradients are sums of atomic
    additions whose order varies from run to run -- even two runs of one trainer
    from one state differ in their last bits -- so they are held to the parity
    bars (loss 1e-9 relative; gradients the scaled gradient bar, its scale taken
    from the oracle at the checkpointed parameters), and Adam, fed one trainer's
    gradients, to bit equality."""
    sc = scenes.make_scene("medium", n=20000)
    c = sc.cameras[0]
    sc.cameras = [scenes.Camera(c.R, c.t, 350.0, 350.0, 240.0, 135.0, 480, 270)]
    targets = parity.oracle_targets(sc)
    tgt = torch.from_numpy(targets).cuda()

    def trainer():
        return pipeline.GaussianTrainer(sc.params, sc.sh_degree, sc.cameras, sc.opts, sc.lr)

    a = trainer()
    for _ in range(3):
        a.train_step(tgt)
    path = tmp_path / "ckpt.pt"
    saved = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in a.state_dict().items()}
    torch.save(saved, path)
    assert (a.last_step.cpu().numpy() == 3).all()
    b = trainer()
    b.load_state_dict(torch.load(path))
    assert b.t == 3
    for name, key in (("params", "params"), ("adam_m", "m"), ("adam_v", "v"), ("last_step", "last_step")):
        assert torch.equal(getattr(b, name).cpu(), saved[key]) and torch.equal(getattr(a, name), getattr(b, name))
    p3 = a.rows(a.params).cpu().numpy()
    out = []
    for tr in (a, b):
        tr.t += 1
        tr.project()
        tr.bin_sort()
        tr.raster(tgt)
        tr.compact()
        torch.cuda.synchronize()
        n_idx = tr.n_idx.cpu().numpy().copy()
        vis = tr.tiles_touched[0].cpu().numpy() > 0          # culled Gaussians' records are not written
        out.append(dict(vis=vis, rec=tr.rec[0].cpu().numpy()[vis], ids=tr.ids[:tr.n_instances].cpu().numpy().copy(),
                        keys=tr.keys[:tr.n_instances].cpu().numpy().copy(), img=tr.image.cpu().numpy().copy(),
                        loss=float(tr.loss[0]), n_idx=n_idx, idx=tr.idx[1, :n_idx[1]].cpu().numpy().copy(),
                        grads=tr.rows(tr.grads).cpu().numpy().copy()))
    x, y = out
    for k in ("vis", "rec", "ids", "keys", "img", "n_idx", "idx"):
        assert np.array_equal(x[k], y[k]), k
    assert abs(x["loss"] - y["loss"]) <= 1e-9 * abs(x["loss"])
    pr = oracle.project(p3, sc.sh_degree, sc.cameras[0], sc.opts)
    ro = oracle.render(pr, sc.cameras[0], sc.opts, target=targets[0], want_mag=True)
    mag = oracle.vjp_mag(p3, sc.sh_degree, sc.cameras[0], sc.opts, ro["grad2d_mag"], ro["touched"], pr["clamp"])
    u = x["idx"].astype(np.int64)
    ok, st = parity.grad_report(y["grads"][:, u], x["grads"][:, u], mag[:, u], axis=1)
    assert ok, st
    b.grads.copy_(a.grads)
    for tr in (a, b):
        tr.adam(tr.t)
    torch.cuda.synchronize()
    for name in ("params", "adam_m", "adam_v", "last_step"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    assert int(a.last_step.max()) == 4 and int(a.last_step.min()) == 3   # still deferred where untouched


@pytest.mark.parametrize("exclude", [0, 1])
def test_work_counting_variant_matches_the_fused_kernel(exclude):
    """gs_raster_work_counts renders and differentiates exactly like the fused call
    (image, loss, touched set bit for bit; 2D gradients at the bar), and its counts
    obey what the method fixes: every composited (pixel, entry) is processed once
    in the backward (queued + per-Gaussian = E_comp); every entry the composite
    walks is composited, except, with the crossing entry excluded, the one each
    stopping pixel stops at; every chunk of every list is staged unless its tile
    stopped early."""
    from differentiable_rasterizer_gb300 import abi
    sc = scenes.random_small_scene(71, n=5000, width=96, height=80, sh_degree=0, log_lo=-3.2, log_hi=-1.6,
                                   logit_mu=1.0, spread=1.2)
    sc.opts = dict(sc.opts, exclude_crossing=exclude)
    tgt = torch.from_numpy(parity.oracle_targets(sc)).cuda()
    tr = pipeline.GaussianTrainer(sc.params, 0, sc.cameras, sc.opts, sc.lr)
    tr.project()
    tr.bin_sort()
    tr.eval_counts.zero_()
    tr.raster(tgt)
    torch.cuda.synchronize()
    ref = dict(img=tr.image.clone(), loss=tr.loss.clone(), g=tr.grad2d.clone(), t=tr.touched.clone(),
               c=tr.eval_counts.cpu().numpy().copy())
    tr.grad2d.zero_()
    tr.touched.zero_()
    w = tr.work_counts(tgt)
    torch.cuda.synchronize()
    assert torch.equal(tr.image, ref["img"]) and torch.equal(tr.touched, ref["t"])
    assert abs(float(tr.loss[0]) - float(ref["loss"][0])) <= 1e-12 * abs(float(ref["loss"][0]))
    m = ref["t"][0].cpu().numpy() > 0
    ok, st = parity.grad_report(tr.grad2d[0].cpu().numpy()[m][:, :9], ref["g"][0].cpu().numpy()[m][:, :9])
    assert ok, st
    e_comp = int(ref["c"][2])
    assert w["sparse_entries"] + w["dense_entries"] == e_comp, (w, e_comp)
    pixels = sc.cameras[0].width * sc.cameras[0].height
    if exclude:
        assert e_comp <= w["composite_walks"] <= e_comp + pixels
    else:
        assert w["composite_walks"] == e_comp, (w, e_comp)
    assert w["pairs"] >= w["pair_exps"] >= w["composite_walks"] - (pixels if exclude else 0)
    ranges = tr.ranges.cpu().numpy().view(np.uint32).reshape(-1, 2)
    lens = (ranges[:, 1] - ranges[:, 0]).astype(np.int64)
    assert (lens > 256).any()
    assert 0 < w["chunks"] <= int(((lens + 255) // 256).sum())
    assert 0 < w["restaged_chunks"] and w["recomputed_chunks"] <= w["restaged_chunks"]
    # a warp's walk takes as many steps as its busiest lane has entries
    assert w["sparse_steps"] <= w["sparse_entries"] <= 32 * w["sparse_steps"]
