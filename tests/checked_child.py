"""Runs in a child process of test_gpu_checked.py with GS_CHECKED=1 in its
environment, so that the bounds-checked library (libgs_gb300_checked.so) is the
one the binding loads.  Modes:

  parity        the oracle parity runs of the tiny workload (fused step, L1 +
                D-SSIM, pruned tile lists, partial render + compose) through the
                checked library; no bounds check may fail.
  outputs OUT   one training step of each workload in WORKLOADS; writes the
                outputs that are deterministic (tile ranges, sorted keys and ids,
                image, compacted lists, last_step) as digests, and summaries of
                the ones that are not (loss, gradients: float atomics), so that the
                parent compares them with the plain library's; no check may fail.
  planted       a listed index equal to n given to gs_adam_deferred, and a sorted
                id beyond n given to the fused raster: each check must fire at its
                site with that index and bound, and everything the bad index does
                not reach must equal the run without it.

workload_outputs() is also what the parent runs with the plain library.
"""
import hashlib
import json
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
for p in (ROOT, HERE):
    if p not in sys.path:
        sys.path.insert(0, p)

from differentiable_rasterizer_gb300 import abi, pipeline, scenes  # noqa: E402

# (name, scene, Gaussian count override, every k-th camera)
WORKLOADS = (("tiny", "tiny", None, 1), ("small", "small", None, 1), ("medium", "medium", None, 1),
             ("batched_4_views_2m", "batched", 2_000_000, 4))


def _sha(t: torch.Tensor) -> str:
    return hashlib.sha256(t.contiguous().cpu().numpy().tobytes()).hexdigest()


def workload_outputs(name, scene, n, every):
    sc = scenes.make_scene(scene, n=n)
    sc.cameras = sc.cameras[::every]
    tr = pipeline.GaussianTrainer(sc.params, sc.sh_degree, sc.cameras, sc.opts, sc.lr)
    if sc.target_kind == "uniform":
        target = torch.from_numpy(sc.target_uniform).cuda()
    else:
        target = tr.render(tr.to_device_layout(sc.perturbed_params)).clone()
    tr.t = 1
    tr.project()
    tr.bin_sort()
    tr.raster(target)
    torch.cuda.synchronize()
    out = {"instances": int(tr.n_instances), "ranges": _sha(tr.ranges), "keys": _sha(tr.keys[:tr.n_instances]),
           "ids": _sha(tr.ids[:tr.n_instances]), "image": _sha(tr.image),
           "loss": [float(x) for x in tr.loss.cpu().tolist()]}
    tr.compact()
    tr.adam(tr.t)
    torch.cuda.synchronize()
    n_idx = tr.n_idx.cpu().tolist()
    out["n_idx"] = [int(x) for x in n_idx]
    out["idx"] = [_sha(tr.idx[v, :n_idx[v]]) for v in range(tr.V + 1)]
    out["last_step"] = _sha(tr.last_step)
    g = tr.grads[:, :tr.P].double()
    out["grad_abs_sum"] = [float(x) for x in g.abs().sum(0).cpu().tolist()]
    gen = torch.Generator().manual_seed(5)
    pick = torch.randint(0, tr.n, (4096,), generator=gen).cuda()
    out["grad_sample"] = tr.grads[pick, :tr.P].cpu().numpy().tolist()
    out["grad_max"] = float(g.abs().max())
    return out


def _expect_clean(tag):
    r = abi.gs_check_report()
    assert r["checked"], "the loaded library is not the bounds-checked build"
    assert r["failures"] == 0, (tag, r)


def mode_parity():
    import parity
    parity.run_stage_parity(scenes.make_scene("tiny"), device="cuda:0")
    _expect_clean("tiny step")
    parity.run_dssim_parity(scenes.make_scene("tiny"), 0.2, device="cuda:0")
    _expect_clean("tiny L1 + D-SSIM")
    pruned = scenes.make_scene("tiny")
    pruned.opts = dict(pruned.opts, tile_budget=64)
    parity.run_stage_parity(pruned, device="cuda:0")
    _expect_clean("tiny pruned")
    parity.run_compose_parity(scenes.make_scene("tiny"), 2)
    _expect_clean("tiny compose")


def mode_outputs(path):
    res = {}
    for w in WORKLOADS:
        res[w[0]] = workload_outputs(*w)
        _expect_clean(w[0])
    with open(path, "w") as f:
        json.dump(res, f)


def _planted_adam():
    n, sh = 1000, 0
    stride = abi.gs_param_stride(sh)
    gen = torch.Generator().manual_seed(11)
    params = torch.randn((n, stride), generator=gen).cuda()
    grads = torch.randn((n, stride), generator=gen).cuda()
    lr = (1e-3, 2e-3, 3e-3, 4e-3, 5e-3)

    def run(listed):
        p, m, v = params.clone(), torch.zeros_like(params), torch.zeros_like(params)
        last = torch.zeros(n, dtype=torch.int32, device="cuda")
        idx = torch.tensor(listed, dtype=torch.int32, device="cuda")
        n_idx = torch.tensor([len(listed)], dtype=torch.int64, device="cuda")
        abi.gs_adam_deferred(p.data_ptr(), grads.data_ptr(), m.data_ptr(), v.data_ptr(), last.data_ptr(), n, sh,
                             idx.data_ptr(), n_idx.data_ptr(), 1, lr, 0.9, 0.999, 1e-8, 0,
                             torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        return p, m, v, last

    good = run(list(range(20)))
    _expect_clean("adam, good list")
    bad = run(list(range(10)) + [n] + list(range(10, 20)))
    r = abi.gs_check_report()
    # 4 float4 chunks of the bad entry in the update kernel, 1 in the stamp kernel
    assert (r["site"], r["index"], r["bound"], r["failures"]) == ("adam_id", n, n, 5), r
    for a, b in zip(good, bad):
        assert torch.equal(a, b)


def _planted_raster():
    sc = scenes.make_scene("tiny")
    tr = pipeline.GaussianTrainer(sc.params, sc.sh_degree, sc.cameras, sc.opts, sc.lr)
    target = torch.from_numpy(sc.target_uniform).cuda()
    tr.project()
    tr.bin_sort()
    r = tr.ranges.view(-1, 2).cpu().numpy().astype(np.int64)
    lens = r[:, 1] - r[:, 0]
    tile = int(np.argmax(lens))
    assert lens[tile] >= 3
    tr.raster(target)
    torch.cuda.synchronize()
    image_good = tr.image.clone()
    _expect_clean("raster, good lists")
    tr.grad2d.zero_()
    tr.touched.zero_()
    bad_id = tr.n + 5
    tr.ids[r[tile, 0] + 1] = bad_id
    tr.raster(target)
    torch.cuda.synchronize()
    rep = abi.gs_check_report()
    assert (rep["site"], rep["index"], rep["bound"]) == ("raster_id", bad_id, tr.n) and rep["failures"] >= 1, rep
    assert torch.isfinite(tr.image).all()
    # every tile but the planted one renders as before
    ty, tx = divmod(tile, (tr.W + 15) // 16)
    keep = torch.ones_like(tr.image, dtype=torch.bool)
    keep[..., ty * 16:(ty + 1) * 16, tx * 16:(tx + 1) * 16] = False
    assert torch.equal(tr.image[keep], image_good[keep])


def mode_planted():
    _expect_clean("start")   # also asserts that the checked build is the one loaded
    _planted_adam()
    _planted_raster()


if __name__ == "__main__":
    assert os.environ.get("GS_CHECKED") == "1", "run with GS_CHECKED=1"
    torch.cuda.set_device(0)
    mode = sys.argv[1]
    if mode == "parity":
        mode_parity()
    elif mode == "outputs":
        mode_outputs(sys.argv[2])
    elif mode == "planted":
        mode_planted()
    else:
        raise SystemExit(f"unknown mode {mode}")
    print(f"checked build: {mode} ok")
