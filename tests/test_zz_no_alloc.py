"""gs_grad_compact_static -- the compaction entry point for callers that cannot
allocate device memory while they run (its scratch is a fixed array inside the
library) -- gives the same outputs as gs_grad_compact with a caller-provided
workspace, on two calls in a row (the second sees the scratch the first left).

This file is named so that pytest collects it last."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ready():
    from differentiable_rasterizer_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _rastered_trainer():
    from differentiable_rasterizer_gb300 import pipeline, scenes
    sc = scenes.make_scene("medium", n=60000)
    c = sc.cameras[0]
    sc.cameras = [scenes.Camera(c.R, c.t, 350.0, 350.0, 240.0, 135.0, 480, 270)]
    tr = pipeline.GaussianTrainer(sc.params, sc.sh_degree, sc.cameras, sc.opts, sc.lr)
    target = torch.rand((1, 3, 270, 480), generator=torch.Generator().manual_seed(3)).cuda()
    tr.project()
    tr.bin_sort()
    tr.raster(target)
    torch.cuda.synchronize()
    return tr


def _run(tr, grad2d0, touched0, static):
    from differentiable_rasterizer_gb300 import abi
    tr.grad2d.copy_(grad2d0)
    tr.touched.copy_(touched0)
    tr.grads.zero_()
    tr.idx.zero_()
    tr.n_idx.fill_(-1)
    args = (tr.grad2d.data_ptr(), tr.touched.data_ptr(), tr.params.data_ptr(), tr.n, tr.sh_degree, tr.cams, tr.V,
            tr.opts, tr.idx.data_ptr(), tr.n_idx.data_ptr(), tr.grads.data_ptr())
    if static:
        abi.gs_grad_compact_static(*args, tr.stream_handle())
    else:
        abi.gs_grad_compact(*args, tr.compact_ws.data_ptr(), tr.compact_ws.numel(), tr.stream_handle())
    torch.cuda.synchronize()
    n_idx = tr.n_idx.cpu().numpy().copy()
    idx = [tr.idx[v, :n_idx[v]].cpu().numpy().copy() for v in range(tr.V + 1)]
    return n_idx, idx, tr.grads.cpu().numpy().copy(), bool(tr.grad2d.any()), bool(tr.touched.any())


def test_static_scratch_matches_workspace_entry_point_twice(ready):
    import parity
    tr = _rastered_trainer()
    g0, t0 = tr.grad2d.clone(), tr.touched.clone()
    assert t0.any()
    ref_n, ref_idx, ref_grads, _, _ = _run(tr, g0, t0, static=False)
    for call in range(2):
        n_idx, idx, grads, g2d_left, touched_left = _run(tr, g0, t0, static=True)
        assert np.array_equal(n_idx, ref_n), call
        for a, b in zip(idx, ref_idx):
            assert np.array_equal(a, b), call
        ok, st = parity.grad_report(grads, ref_grads)
        assert ok, (call, st)
        assert not g2d_left and not touched_left, call


def test_static_entry_rejects_more_than_its_maximum(ready):
    from differentiable_rasterizer_gb300 import abi, scenes
    cams = abi.cameras(scenes.make_scene("tiny").cameras)
    opts = abi.render_opts(scenes.DEFAULT_OPTS)
    with pytest.raises(abi.GsError) as e:
        abi.gs_grad_compact_static(16, 16, 16, (1 << 22) + 1, 0, cams, 1, opts, 16, 16, 16, None)
    assert e.value.status == abi.GS_ERR_INVALID_ARG
