"""gs_grad_compact_static -- the compaction entry point for callers that cannot
allocate device memory while they run (its scratch is a fixed array inside the
library) -- gives exactly the outputs of gs_grad_compact with a caller-provided
workspace, on two calls in a row (the second sees the scratch the first left),
with one view (the union is that view's list) and with three (the union pass
runs over the array's flag region), and the device's free memory does not move
across its calls.

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


def _rastered_trainer(views):
    from differentiable_rasterizer_gb300 import pipeline, scenes
    if views == 1:
        sc = scenes.make_scene("medium", n=60000)
    else:
        sc = scenes.make_scene("batched", n=60000)
        sc.cameras = sc.cameras[::16 // views][:views]
    sc.cameras = [scenes.Camera(c.R, c.t, 350.0, 350.0, 240.0, 135.0, 480, 270) for c in sc.cameras]
    tr = pipeline.GaussianTrainer(sc.params, sc.sh_degree, sc.cameras, sc.opts, sc.lr)
    target = torch.rand((views, 3, 270, 480), generator=torch.Generator().manual_seed(3)).cuda()
    tr.project()
    tr.bin_sort()
    tr.raster(target)
    torch.cuda.synchronize()
    return tr


def _run(tr, grad2d0, touched0, static):
    """One compaction call on copies of the rastered state; returns its outputs and
    the device's free bytes just before and just after the call."""
    from differentiable_rasterizer_gb300 import abi
    tr.grad2d.copy_(grad2d0)
    tr.touched.copy_(touched0)
    tr.grads.zero_()
    tr.idx.zero_()
    tr.n_idx.fill_(-1)
    args = (tr.grad2d.data_ptr(), tr.touched.data_ptr(), tr.params.data_ptr(), tr.n, tr.sh_degree, tr.cams, tr.V,
            tr.opts, tr.idx.data_ptr(), tr.n_idx.data_ptr(), tr.grads.data_ptr())
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    if static:
        abi.gs_grad_compact_static(*args, tr.stream_handle())
    else:
        abi.gs_grad_compact(*args, tr.compact_ws.data_ptr(), tr.compact_ws.numel(), tr.stream_handle())
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    n_idx = tr.n_idx.cpu().numpy().copy()
    idx = [tr.idx[v, :n_idx[v]].cpu().numpy().copy() for v in range(tr.V + 1)]
    return dict(n_idx=n_idx, idx=idx, grads=tr.grads.cpu().numpy().copy(), g2d_left=bool(tr.grad2d.any()),
                touched_left=bool(tr.touched.any()), free=(free0, free1))


@pytest.mark.parametrize("views", [1, 3])
def test_static_scratch_matches_workspace_entry_point_twice(ready, views):
    tr = _rastered_trainer(views)
    g0, t0 = tr.grad2d.clone(), tr.touched.clone()
    assert t0.any()
    if views > 1:   # the union differs from every single view's list
        per_view = t0.cpu().numpy().astype(bool)
        assert (per_view.any(0).sum() > per_view.sum(1)).all()
    ref = _run(tr, g0, t0, static=False)
    for call in range(3):   # the first call may look up the array's address; the next two must not allocate
        got = _run(tr, g0, t0, static=True)
        assert np.array_equal(got["n_idx"], ref["n_idx"]), call
        for a, b in zip(got["idx"], ref["idx"]):
            assert np.array_equal(a, b), call
        # both calls run the same deterministic kernels (scans; views summed in order in registers)
        assert np.array_equal(got["grads"].view(np.uint32), ref["grads"].view(np.uint32)), call
        assert not got["g2d_left"] and not got["touched_left"], call
        if call > 0:
            assert got["free"][0] == got["free"][1], (call, got["free"])


def test_static_entry_rejects_more_than_its_maximum(ready):
    from differentiable_rasterizer_gb300 import abi, scenes
    cams = abi.cameras(scenes.make_scene("tiny").cameras)
    opts = abi.render_opts(scenes.DEFAULT_OPTS)
    with pytest.raises(abi.GsError) as e:
        abi.gs_grad_compact_static(16, 16, 16, (1 << 22) + 1, 0, cams, 1, opts, 16, 16, 16, None)
    assert e.value.status == abi.GS_ERR_INVALID_ARG
