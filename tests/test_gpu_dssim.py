"""GPU parity of the L1 + D-SSIM loss path against the oracle: the D-SSIM kernel
on its own (random, smooth and flat images, several views, images smaller than
the window and sizes that leave ragged output tiles), and whole steps through
forward-with-state -> D-SSIM -> backward-from-state (tiny, ragged, an image
smaller than the window, several SH-3 views with a background, lambda 0 and 1,
the small workload at full size).  With lambda = 0 the three-launch path must
reproduce the fused L1 kernel."""
import math

import numpy as np
import pytest
import torch

import oracle
from differentiable_rasterizer_gb300 import abi, pipeline, scenes

import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from differentiable_rasterizer_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _dssim_gpu(x, y, lam):
    V, _, H, W = x.shape
    xd = torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda()
    yd = torch.from_numpy(np.ascontiguousarray(y, np.float32)).cuda()
    loss = torch.full((V,), 123.0, dtype=torch.float64, device="cuda")
    dldc = torch.full((V, 3, H, W), float("nan"), dtype=torch.float32, device="cuda")
    abi.gs_dssim_loss_grad(xd.data_ptr(), yd.data_ptr(), V, W, H, lam, loss.data_ptr(), dldc.data_ptr(),
                           torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return loss.cpu().numpy(), dldc.cpu().numpy()


def _images(kind, V, H, W, seed):
    rng = np.random.default_rng(seed)
    if kind == "random":
        x = rng.uniform(0, 1, (V, 3, H, W))
        y = np.clip(x + rng.normal(0, 0.15, x.shape), 0, 1)
    elif kind == "smooth":
        # slow ramps plus a few soft blobs; large flat parts make D close to C2
        yy, xx = np.mgrid[0:H, 0:W] / max(H, W)
        base = 0.3 + 0.4 * xx + 0.2 * yy
        x = np.stack([np.stack([base + 0.05 * c for c in range(3)])] * V)
        for _ in range(6):
            cy, cx, r = rng.uniform(0, 1), rng.uniform(0, 1), rng.uniform(0.02, 0.1)
            x += rng.uniform(-0.2, 0.2) * np.exp(-((yy - cy) ** 2 + (xx - cx) ** 2) / (2 * r * r))
        y = np.clip(x + rng.normal(0, 0.01, x.shape), 0, 1)
        x = np.clip(x, 0, 1)
    else:   # flat: constant images, S from the closed form away from the border
        x = np.full((V, 3, H, W), 0.7)
        y = np.full((V, 3, H, W), 0.69)
    return x.astype(np.float32), y.astype(np.float32)


@pytest.mark.parametrize("kind,V,H,W,lam", [
    ("random", 1, 64, 64, 0.2),      # exactly 2 x 2 output tiles
    ("random", 2, 77, 100, 0.2),     # ragged output tiles, two views
    ("smooth", 1, 96, 130, 0.2),
    ("flat", 1, 40, 45, 0.2),
    ("random", 1, 5, 7, 0.2),        # smaller than the window
    ("random", 1, 33, 1, 1.0),       # one column
    ("smooth", 1, 50, 70, 1.0),
    ("random", 1, 40, 40, 0.0),      # pure L1
])
def test_dssim_kernel_matches_the_oracle(kind, V, H, W, lam):
    x, y = _images(kind, V, H, W, seed=H * 1000 + W)
    loss, dldc = _dssim_gpu(x, y, lam)
    st = {}
    for v in range(V):
        parity.check_dssim_stage(x[v], y[v], lam, loss[v], dldc[v], st, tag=f"{kind} view {v}")
    print(f"[dssim kernel] {kind} V={V} {H}x{W} lambda={lam}: {st}")
    if lam == 0.0:
        N = 3 * H * W
        want = np.sign(x.astype(np.float64) - y) * np.float32(1.0 / N)
        assert np.array_equal(dldc, want.astype(np.float32))


def test_dssim_tiny():
    parity.run_dssim_parity(scenes.make_scene("tiny"), 0.2)


def test_dssim_ragged_resolution_lambda_one():
    sc = scenes.make_scene("tiny")
    cam = sc.cameras[0]
    sc.cameras = [scenes.Camera(cam.R, cam.t, 64.0, 64.0, 35.0, 22.5, 70, 45)]
    sc.target_uniform = np.random.default_rng(9).uniform(0, 1, (1, 3, 45, 70)).astype(np.float32)
    parity.run_dssim_parity(sc, 1.0)


def test_dssim_image_smaller_than_the_window():
    sc = scenes.random_small_scene(41, n=30, width=9, height=6, sh_degree=0, fx=12.0)
    parity.run_dssim_parity(sc, 0.2)


def test_dssim_multi_view_degree3_background():
    sc = scenes.make_scene("medium", n=20000)
    cams = []
    for k, ang in enumerate((-0.1, 0.0, 0.12)):
        c, s = math.cos(ang), math.sin(ang)
        R = np.array([[c, 0, s], [0, 1, 0], [-s, 0, c]], np.float32)
        cams.append(scenes.Camera(R, np.array([0.5 * k, 0.2, 0.0], np.float32), 300.0, 300.0, 160.0, 90.0, 320, 180))
    sc.cameras = cams
    sc.opts = dict(sc.opts, exclude_crossing=1, bg=(0.1, 0.4, 0.7))
    parity.run_dssim_parity(sc, 0.2)


def test_dssim_small_full():
    parity.run_dssim_parity(scenes.make_scene("small"), 0.2)


def test_lambda_zero_reproduces_the_fused_l1_kernel():
    sc = scenes.make_scene("medium", n=20000)
    c = sc.cameras[0]
    sc.cameras = [scenes.Camera(c.R, c.t, 350.0, 350.0, 240.0, 135.0, 480, 270)]
    targets = parity.oracle_targets(sc)
    tgt = torch.from_numpy(targets).cuda()
    out = []
    for lam in (None, 0.0):
        tr = pipeline.GaussianTrainer(sc.params, sc.sh_degree, sc.cameras, sc.opts, sc.lr, dssim_lambda=lam)
        tr.project()
        tr.bin_sort()
        tr.eval_counts.zero_()
        tr.raster(tgt)
        torch.cuda.synchronize()
        out.append(dict(img=tr.image.cpu().numpy(), loss=tr.loss.cpu().numpy(), g=tr.grad2d.cpu().numpy()[..., :9],
                        t=tr.touched.cpu().numpy(), c=tr.eval_counts.cpu().numpy()))
        del tr
    a, b = out
    assert np.array_equal(parity.bits(a["img"]), parity.bits(b["img"]))
    assert np.array_equal(a["t"], b["t"]) and np.array_equal(a["c"], b["c"])
    assert abs(a["loss"][0] - b["loss"][0]) <= 1e-12 * a["loss"][0]
    m = a["t"][0] > 0
    pr = oracle.project(sc.params, sc.sh_degree, sc.cameras[0], sc.opts)
    mag = oracle.render(pr, sc.cameras[0], sc.opts, target=targets[0], want_mag=True)["grad2d_mag"]
    ok, st = parity.grad_report(b["g"][0][m], a["g"][0][m], mag[m])
    assert ok, st


def test_backward_with_stored_pass_bits_equals_recomputing_them():
    """The stored-state backward reading every chunk's pass bits from the scratch
    the forward filled gives what recomputing them gives (lists spanning several
    chunks)."""
    from differentiable_rasterizer_gb300 import abi
    sc = scenes.random_small_scene(21, n=4000, width=64, height=64, sh_degree=0, log_lo=-3.0, log_hi=-1.8,
                                   logit_mu=1.0, spread=1.2)
    tgt = torch.from_numpy(parity.oracle_targets(sc)).cuda()
    tr = pipeline.GaussianTrainer(sc.params, 0, sc.cameras, sc.opts, sc.lr, dssim_lambda=0.2)
    tr.project()
    tr.bin_sort()
    tr.raster(tgt)                      # with stored bits
    torch.cuda.synchronize()
    g_bits, t_bits = tr.grad2d.clone(), tr.touched.clone()
    lens = np.diff(tr.ranges.cpu().numpy().view(np.uint32).reshape(-1, 2), axis=1)
    assert lens.max() > 2 * 256                       # tiles whose backward reads several chunks' bits
    tr.grad2d.zero_()
    tr.touched.zero_()
    abi.gs_raster_backward_state(tr.proj, tr.n, tr.ranges.data_ptr(), tr.ids.data_ptr(), tr.cams, tr.V, tr.opts,
                                 tr.t_final.data_ptr(), tr.last_idx.data_ptr(), None, 0, tr.dldc.data_ptr(),
                                 tr.grad2d.data_ptr(), tr.touched.data_ptr(), tr.stream_handle())
    torch.cuda.synchronize()
    assert torch.equal(t_bits, tr.touched)
    m = t_bits[0].cpu().numpy() > 0
    pr = oracle.project(sc.params, 0, sc.cameras[0], sc.opts)
    mag = oracle.render(pr, sc.cameras[0], sc.opts, target=parity.oracle_targets(sc)[0],
                        dldc_extra=tr.dldc[0].cpu().numpy(), l1_weight=0.0, want_mag=True)["grad2d_mag"]
    ok, st = parity.grad_report(g_bits.cpu().numpy()[0][m][:, :9], tr.grad2d.cpu().numpy()[0][m][:, :9], mag[m])
    assert ok, st


def test_dssim_maximum_view_count():
    """The D-SSIM step over GS_MAX_VIEWS (32) views."""
    sc = scenes.random_small_scene(53, n=300, width=36, height=20, sh_degree=0, log_lo=-3.0, log_hi=-2.0)
    cams = []
    for k in range(32):
        ang = -0.3 + 0.6 * k / 31
        c, s = math.cos(ang), math.sin(ang)
        R = np.array([[c, 0, s], [0, 1, 0], [-s, 0, c]], np.float32)
        cams.append(scenes.Camera(R, np.zeros(3, np.float32), 36.0, 36.0, 18.0, 10.0, 36, 20))
    sc.cameras = cams
    sc.target_uniform = np.random.default_rng(54).uniform(0, 1, (32, 3, 20, 36)).astype(np.float32)
    parity.run_dssim_parity(sc, 0.2)
