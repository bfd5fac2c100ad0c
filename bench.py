#!/usr/bin/env python
"""Benchmark of one 3DGS training step (projection, binning + sort, fused
forward/backward rasterization, compaction + VJP, deferred Adam) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config medium] [--impl gpu|reference]
                    [--dssim LAMBDA] [--tile-budget K] [--partial S]

The options time the variants: the L1 + D-SSIM loss, per-tile pruned lists,
and (a separate line) the forward render as S composed depth slabs.

Prints ONE JSON line (rank 0).  The metric is Gaussian-pixel evaluations per
second (forward evaluations up to each pixel's stop, plus backward evaluations
up to each pixel's last composited entry) over the whole step, with the fused
raster kernel's own time, its roofline fraction, the end-to-end number through
the public API from pinned host memory, and the CPU oracle timed on a bounded
sample.  Under torchrun (N > 1) every rank trains its own replica of the
workload (the step has no cross-GPU exchange on one node here); the value is
the sum over ranks divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "fused raster fwd+bwd Gaussian-pixel evals/s and ms/iter at 1 GB300; % of roofline"
# D-SSIM loss kernel: FP32 operations per pixel and channel of the separable form
# (5 windowed moments at 2 x 11 fma each plus 3 products, 32 for S and its three
# derivatives, 3 derivative maps at 2 x 11 fma, 11 for dL/dC and the loss terms).
OPS_DSSIM = 222
UNIT = "Gaussian-pixel evals/s"

WORKLOADS = {
    "tiny": "tiny: 1,000 Gaussians, RGB, one 64x64 view",
    "small": "small: 100,000 Gaussians, RGB, one 1280x720 view",
    "medium": "medium: 1,000,000 Gaussians in 64 clusters, SH degree 3, one 1920x1080 view, fx=fy=1400",
    "large": "large: 11,200,000 Gaussians, SH degree 3, one 4096x2160 view, fx=fy=3000",
    "batched": "batched: 20,000,000 Gaussians, SH degree 3, 16 views 1920x1080, gradients summed",
}

# Work of the fused raster kernel.  The metric's units are the method's
# evaluations (E_fwd: list entries up to each pixel's stop; E_bwd: entries up to
# its last composited one), but the kernel executes far fewer: the per-Gaussian
# support box and alpha cut skip, with results unchanged, every pair that cannot
# pass.  The roofline therefore charges what the kernel executes, counted by its
# counting variant (gs_raster_work_counts) in one untimed launch, at the FP32
# operations each item performs in the source (an fma counts once; compares,
# integer and shared-memory work not counted):
#   candidate tested:    10  (dx, dy, power)
#   exponential:         14  (portable exp 12: scale, round, 2-fma reduction,
#                             7-fma Horner; alpha = min(0.99, o G) 2)
#   composite:            9  (T update, weight, C += c w T)
#   backward, per pixel: 56  + 1 SFU reciprocal (power, exp, alpha, 1 / (1 - alpha),
#                             T before the entry, dL/dC . c, 9 gradient terms,
#                             dL/dC . colour behind)
#   backward, per Gaussian: the same 56 + 1 SFU per (entry, pixel), and 12 adds
#                             per lane per warp step (recursive-halving warp sum)
#   per pixel:           15  (background, L1 difference, signs, S init)
W_OPS = {"pairs": 10, "pair_exps": 14, "composite_walks": 9, "sparse_entries": 56, "dense_entries": 56,
         "dense_steps": 12 * 32}
W_OPS_PIXEL = 15
# The per-evaluation model the metric's units suggest (kept beside it for
# comparison): every forward evaluation 14 FP32 ops + exp, every backward
# evaluation 47 + exp + reciprocal, exp as the polynomial's 14 FP32 ops.
OPS_FWD, OPS_BWD, OPS_EXP = 14, 47, 14
SMS, FP32_LANES, SFU_LANES = 152, 128, 16


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    src = "measured"
    try:
        with open(path) as f:
            mp = json.load(f)
    except OSError:
        mp, src = {}, "fallback"
    mhz = float(mp.get("sm_max_mhz", 2070.0))
    return dict(src=src, sm_max_mhz=mhz, hbm_gbs=float(mp.get("hbm_gbs", 6800.0)),
                fp32_tops=SMS * FP32_LANES * mhz * 1e6 / 1e12,
                sfu_tops=SMS * SFU_LANES * mhz * 1e6 / 1e12)


def _code_only(text: str) -> str:
    """Source text without its comments and blank lines: an edit of a comment does
    not change the kernel the counters were taken of."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def source_sha():
    """sha256 of the fused kernel's code (raster.cu + gs_common.cuh, comments removed)."""
    h = hashlib.sha256()
    for p in ("differentiable_rasterizer_gb300/csrc/raster.cu", "differentiable_rasterizer_gb300/csrc/gs_common.cuh"):
        with open(os.path.join(ROOT, p), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()


def profile_figures():
    """Figures of the fused kernel from the committed ncu capture (DRAM bytes per launch,
    issue slots busy), or None where the capture does not match the current source."""
    path = os.path.join(ROOT, "profiles", "raster_fused_medium_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except OSError:
        return {}
    return d if d.get("source_sha256") == source_sha() else {}


# ----------------------------------------------------------------------------- clocks
CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def start_clock_sampler(path, gpu_index):
    try:
        f = open(path, "w")
        p = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + CLOCK_QUERY, "--format=csv",
                              "-lms", "200"], stdout=f, stderr=subprocess.DEVNULL)
        return p, f
    except (OSError, FileNotFoundError):
        return None, None


def stop_clock_sampler(handle, path):
    p, f = handle
    if p is None:
        return None
    p.terminate()
    try:
        p.wait(timeout=5)
    except subprocess.TimeoutExpired:
        p.kill()
    f.close()
    sm, mx, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    with open(path) as fh:
        for line in fh:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9 or parts[0] == "index":
                continue
            try:
                sm.append(float(parts[1].split()[0]))
                mx.append(float(parts[2].split()[0]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
    if not sm:
        return None
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- oracle (CPU) sample
def band_camera(cam, rows):
    """The same camera restricted to `rows` image rows around the centre (identical pixels)."""
    from differentiable_rasterizer_gb300 import scenes
    rows = min(rows, cam.height)
    y0 = (cam.height - rows) // 2
    return scenes.Camera(cam.R, cam.t, cam.fx, cam.fy, cam.cx, cam.cy - y0, cam.width, rows), y0


def oracle_sample_step(sc, targets, rows, state, t):
    """One oracle training step (O1..O12) on a band of `rows` rows of every view."""
    import oracle
    from differentiable_rasterizer_gb300 import scenes
    cams, tg = [], []
    for v, cam in enumerate(sc.cameras):
        bc, y0 = band_camera(cam, rows)
        cams.append(bc)
        tg.append(targets[v][:, y0:y0 + bc.height, :])
    sub = scenes.Scene(sc.name, sc.params, sc.sh_degree, cams, "given", None, None, sc.lr, sc.opts)
    lr_rows = scenes.lr_rows(sc.lr, sc.sh_degree)
    t0 = time.perf_counter()
    out = oracle.train_step(sub, np.stack(tg), state, t, lr_rows, scenes.ADAM_BETAS, scenes.ADAM_EPS)
    dt = time.perf_counter() - t0
    ev = sum(v["render"]["e_fwd"] + v["render"]["e_bwd"] for v in out["views"])
    return ev, dt


def cpu_targets_band(sc, rows):
    """Targets on the band only, rendered by the oracle from the perturbed scene."""
    import oracle
    if sc.target_kind == "uniform":
        return sc.target_uniform
    out = []
    for cam in sc.cameras:
        bc, y0 = band_camera(cam, rows)
        pr = oracle.project(sc.perturbed_params, sc.sh_degree, bc, sc.opts)
        img = oracle.render(pr, bc, sc.opts)["image"]
        full = np.zeros((3, cam.height, cam.width), np.float32)
        full[:, y0:y0 + bc.height] = img
        out.append(full)
    return np.stack(out)


def run_reference(args):
    """The CPU oracle as it stands, on bounded samples of the same workload."""
    from differentiable_rasterizer_gb300 import scenes
    import oracle
    oracle.build()
    sc = scenes.make_scene(args.config, seed=args.seed)
    rows = args.ref_rows
    targets = cpu_targets_band(sc, rows)
    state = dict(params=sc.params.copy(), m=np.zeros_like(sc.params), v=np.zeros_like(sc.params),
                 last_step=np.zeros(sc.n, np.int32))
    for w in range(args.warmup):
        oracle_sample_step(sc, targets, rows, state, w + 1)
    ev_tot, t_tot = 0, 0.0
    for k in range(args.steps):
        ev, dt = oracle_sample_step(sc, targets, rows, state, args.warmup + k + 1)
        ev_tot += ev
        t_tot += dt
    val = ev_tot / t_tot
    sample = f"{rows} central image rows of every view (full projection of all Gaussians, band render, VJP, " \
             f"compaction, deferred Adam) per step"
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_tot / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded)", "config": {"workload": WORKLOADS[args.config], "sample": sample},
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- ranks
def job_throughput(units, ms, world, device="cpu"):
    """Whole-job throughput of `world` replica ranks (one per GPU): the units every
    rank processed, summed, over the slowest rank's time.  Returns (units/s, slowest
    ms).  Every rank must call it (it is a collective when world > 1)."""
    import torch
    import torch.distributed as dist
    u = torch.tensor([float(units)], dtype=torch.float64, device=device)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(u, op=dist.ReduceOp.SUM)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(u.item()) / (float(t.item()) / 1e3), float(t.item())


# ----------------------------------------------------------------------------- GPU arm
def run_gpu(args):
    import torch
    import torch.distributed as dist
    from differentiable_rasterizer_gb300 import build as gs_build, pipeline, scenes

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    gs_build.build()

    sc = scenes.make_scene(args.config, seed=args.seed)
    tr = pipeline.GaussianTrainer(sc.params, sc.sh_degree, sc.cameras, sc.opts, sc.lr, device="cuda",
                                  dssim_lambda=args.dssim, tile_budget=args.tile_budget)
    if sc.target_kind == "uniform":
        target = torch.from_numpy(sc.target_uniform).cuda()
    else:
        pert = tr.to_device_layout(sc.perturbed_params)
        target = tr.render(pert).clone()     # training target: render of the perturbed scene
        del pert
    torch.cuda.synchronize()
    prune_quality = None
    if args.tile_budget:
        # quality of the pruned render against the unpruned one (which matches the oracle)
        pruned = tr.render().clone()
        tr.tile_budget = None
        full = tr.render().clone()
        tr.tile_budget = args.tile_budget
        mse = float(((pruned.double() - full.double()) ** 2).mean())
        prune_quality = {"psnr_vs_unpruned_db": (10 * math.log10(1.0 / mse)) if mse > 0 else None,
                         "max_abs_diff": float((pruned - full).abs().max()),
                         "pixels_changed": float((pruned != full).any(1).double().mean())}
        del pruned, full
    torch.cuda.synchronize()

    stream = torch.cuda.current_stream()

    def step(ev=None):
        tr.t += 1
        if ev is not None:
            ev[0].record(stream)
        tr.project()
        if ev is not None:
            ev[1].record(stream)
        tr.bin_sort()
        if ev is not None:
            ev[2].record(stream)
        if args.dssim is None:
            tr.raster(target)
        else:
            tr.raster_dssim(target, events=None if ev is None else (ev[6], ev[7]))
        if ev is not None:
            ev[3].record(stream)
        tr.compact()
        if ev is not None:
            ev[4].record(stream)
        tr.adam(tr.t)
        if ev is not None:
            ev[5].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # ---- device-resident timed region
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clock_path = os.path.join(os.environ.get("GS_BENCH_CLOCKS_DIR", tempfile.gettempdir()),
                              f"bench_clocks_r{rank}.csv")
    sampler = start_clock_sampler(clock_path, local)
    time.sleep(0.5)
    tr.eval_counts.zero_()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_start.record(stream)
    for k in range(args.steps):
        step(evs[k])
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = stop_clock_sampler(sampler, clock_path)
    total_ms = t_start.elapsed_time(t_end)
    stage_ms = np.array([[e[i].elapsed_time(e[i + 1]) for i in range(5)] for e in evs])
    if args.log_steps and rank == 0:
        with open(args.log_steps, "w") as f:
            for k in range(args.steps):
                f.write(json.dumps({"step": k, "ms": float(evs[k][0].elapsed_time(evs[k][5])),
                                    "stage_ms": dict(zip(["project", "bin_sort", "raster", "grad_compact",
                                                          "adam_deferred"], [float(x) for x in stage_ms[k]]))}) + "\n")
            # the state after the last timed step
            f.write(json.dumps({"after_steps": args.steps, "loss": [float(x) for x in tr.loss.cpu().tolist()],
                                "instances": int(tr.n_instances), "union": int(tr.n_idx[tr.V].item()),
                                "per_view_nonzero": [int(x) for x in tr.n_idx[:tr.V].cpu().tolist()]}) + "\n")
    counts = tr.eval_counts.cpu().numpy().astype(np.float64)
    e_fwd, e_bwd, e_comp = counts / args.steps
    evals_per_step = e_fwd + e_bwd
    raster_ms = float(stage_ms[:, 2].mean())
    if args.dssim is not None:
        split = np.array([[e[2].elapsed_time(e[6]), e[6].elapsed_time(e[7]), e[7].elapsed_time(e[3])] for e in evs])
        fwd_ms, dssim_ms, bwd_ms = (float(x) for x in split.mean(0))

    # ---- end to end through the public API: every step's target copied in from pinned
    # host memory (step k + 1's copy overlapping step k) and its loss copied out
    target_host = target.cpu().pin_memory()
    loss_host = torch.empty((args.steps, tr.V), dtype=torch.float64).pin_memory()
    tr.train_steps_host([target_host] * 2, torch.empty((2, tr.V), dtype=torch.float64).pin_memory())   # buffers, stream
    tr.eval_counts.zero_()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    tr.train_steps_host([target_host] * args.steps, loss_host)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    e2e_evals = float(tr.eval_counts.cpu().numpy()[:2].sum())

    value, total_ms = job_throughput(evals_per_step * args.steps, total_ms, world, "cuda")
    e2e_value, e2e_ms = job_throughput(e2e_evals, e2e_ms, world, "cuda")

    pk = peaks()
    prof = profile_figures() if args.dssim is None else {}
    t_raster = (raster_ms if args.dssim is None else fwd_ms + bwd_ms) / 1e3
    roofline = raster_roofline(tr, target, args, pk, prof, t_raster, e_fwd, e_bwd)

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded; target = render of "
            "the scene with means perturbed by N(0, 0.01))",
            "config": {"workload": WORKLOADS[args.config], "n_gaussians": sc.n, "views": sc.n_views,
                       "resolution": [sc.cameras[0].width, sc.cameras[0].height], "sh_degree": sc.sh_degree,
                       "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                       "l2": "inputs larger than L2: each step streams params, Adam state and grads "
                             f"({4 * sc.params.size * 4 / 1e9:.2f} GB) through HBM"},
            "evals_per_step": {"e_fwd": e_fwd, "e_bwd": e_bwd, "e_comp": e_comp},
            "instances": tr.n_instances,
            "fused_raster": {"ms": raster_ms, "evals_per_s": evals_per_step / (raster_ms / 1e3)},
            "stage_ms": dict(zip(["project", "bin_sort", "raster_fused", "grad_compact", "adam_deferred"],
                                 [float(x) for x in stage_ms.mean(0)])),
            "roofline": roofline,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": int(target.numel() * 4),
                    "d2h_bytes_per_step": int(tr.V * 8)},
            "gpu_launches": int(tr.kernel_launches_per_step() * args.steps),
            "clocks": clocks}
    if args.tile_budget:
        line["config"]["tile_budget"] = args.tile_budget
        line["prune_quality"] = prune_quality
    if args.dssim is not None:
        pixels = sc.n_views * sc.cameras[0].width * sc.cameras[0].height
        ops_d = pixels * 3 * OPS_DSSIM
        t_d = ops_d / (pk["fp32_tops"] * 1e12)
        line["config"]["loss"] = f"(1 - {args.dssim}) L1 + {args.dssim} (1 - SSIM), 11x11 Gaussian window"
        line["raster_split_ms"] = {"forward_state": fwd_ms, "dssim_loss_grad": dssim_ms, "backward_state": bwd_ms}
        line["dssim"] = {"ms": dssim_ms, "bound": "alu", "achieved": ops_d / (dssim_ms / 1e3) / 1e12,
                         "peak": pk["fp32_tops"], "unit": "TFLOP/s", "frac": t_d / (dssim_ms / 1e3),
                         "hbm_bytes": pixels * 3 * 12, "hbm_frac": pixels * 3 * 12 / (dssim_ms / 1e3) /
                         (pk["hbm_gbs"] * 1e9),
                         "work": f"{OPS_DSSIM} FP32 ops per pixel and channel (separable window: 5 moments x 22 "
                                 "fma + 3 products, 32 for S and its derivatives, 3 derivative maps x 22 fma, 11 "
                                 "for dL/dC and the loss); 12 bytes (image, target in, dL/dC out)"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(sc, args)
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def raster_roofline(tr, target, args, pk, prof, t_raster, e_fwd, e_bwd):
    """Roofline of the fused raster kernel against its executed work (see W_OPS),
    counted in one untimed launch of the counting variant on a fresh step's lists.
    With the L1 + D-SSIM loss the raster runs as two launches (forward storing its
    state, backward from it) that test the same candidates, composite the same
    entries and walk the same backward entries (chunk by chunk, dense or sparse
    by the same pass bits) as the fused kernel on those lists: the counting
    variant's counts are theirs."""
    tr.project()
    tr.bin_sort()
    work = tr.work_counts(target)
    tr.compact()                      # consumes grad2d / touched as a step would
    import torch
    torch.cuda.synchronize()
    pixels = tr.V * tr.W * tr.H
    ops = sum(W_OPS[k] * work[k] for k in W_OPS) + W_OPS_PIXEL * pixels
    sfu = work["sparse_entries"] + work["dense_entries"]
    t_model = e_fwd * (OPS_FWD + OPS_EXP) + e_bwd * (OPS_BWD + OPS_EXP)
    fp32 = pk["fp32_tops"] * 1e12
    r = {"bound": "alu", "peak": pk["fp32_tops"], "unit": "TFLOP/s",
         "traffic": prof.get("dram_bytes_per_launch") if args.config == "medium" else None,
         "kernel": "raster_fused_kernel<kFused>" if args.dssim is None else
                   "raster_fused_kernel<kFwd> + raster_fused_kernel<kBwdState> (D-SSIM kernel excluded)",
         "peak_basis": f"FP32 pipe: 152 SMs x 128 lanes x {pk['sm_max_mhz']:.0f} MHz (sm_max_mhz, {pk['src']}; "
                       f"an fma counts once); SFU: 152 x 16 lanes",
         "frac_per_evaluation_model": (t_model / fp32) / t_raster}
    t_work = max(ops / fp32, sfu / (pk["sfu_tops"] * 1e12))
    r.update(achieved=ops / t_raster / 1e12, frac=t_work / t_raster, executed=work,
             ops_per_launch=ops, sfu_per_launch=sfu,
             work="executed FP32 ops: " + ", ".join(f"{v} per {k}" for k, v in W_OPS.items()) +
                  f", {W_OPS_PIXEL} per pixel (counting variant, one untimed launch); SFU: one reciprocal "
                  "per backward entry" + ("" if args.dssim is None else
                                          "; counted on the fused kernel, whose candidates, composites and "
                                          "backward entries are those of the two D-SSIM launches"))
    for key, src in (("issue_active_ncu", "issue_active_pct"), ("pipe_fma_ncu", "pipe_fma_pct"),
                     ("pipe_alu_ncu", "pipe_alu_pct"), ("pipe_xu_ncu", "pipe_xu_pct"),
                     ("pipe_lsu_ncu", "pipe_lsu_pct")):
        if prof.get(src) is not None and args.config == "medium" and args.dssim is None:
            r[key] = prof[src] / 100.0
    r["note"] = ("frac = the time the executed FP32 work needs at the FP32-pipe peak over the kernel's mean "
                 "CUDA-event time; frac_per_evaluation_model charges every E_fwd / E_bwd evaluation instead "
                 "(above 1: the kernel skips provably failing pairs).  The *_ncu fields are the hardware's own "
                 "shares for the same kernel from the committed ncu capture of the medium workload.")
    return r


def run_partial(args):
    """Forward render as S depth slabs rendered on their own and composed, against the
    one-pass forward render of the same scene (both: projection, binning, raster)."""
    import torch
    from differentiable_rasterizer_gb300 import build as gs_build, pipeline, scenes
    torch.cuda.set_device(0)
    gs_build.build()
    sc = scenes.make_scene(args.config, seed=args.seed)
    tr = pipeline.GaussianTrainer(sc.params, sc.sh_degree, sc.cameras, sc.opts, sc.lr, device="cuda")
    S = args.partial
    tr.project()
    splits = []
    for v in range(tr.V):
        d = tr.depth[v][tr.tiles_touched[v] > 0].double().sort().values
        splits.append([float(np.float32(d[int(len(d) * s / S)].item())) for s in range(1, S)])
    stream = torch.cuda.current_stream()

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / args.steps

    one_ms = timed(lambda: tr.render())
    one = tr.image.clone()
    part_ms = timed(lambda: tr.render_partial(splits))
    diff = float((tr.image - one).abs().max())
    line = {"metric": "partial render + compose: ms per forward render (projection, binning, raster)",
            "value": part_ms, "unit": "ms", "higher_is_better": False, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "dtype": "f32", "data": "synthetic (seeded)",
            "config": {"workload": WORKLOADS[args.config], "subsets": S, "split": "per-view depth quantiles"},
            "one_pass_ms": one_ms, "max_abs_diff_vs_one_pass": diff,
            "gpu_launches_note": "slab sub-ranges 1 + S forward rasters + compose 1 on top of the one-pass launches"}
    print(json.dumps(line), flush=True)


def cpu_baseline(sc, args):
    """The oracle timed on a bounded sample (a band of rows) of the same workload, one core."""
    rows = args.cpu_rows
    targets = cpu_targets_band(sc, rows)
    state = dict(params=sc.params.copy(), m=np.zeros_like(sc.params), v=np.zeros_like(sc.params),
                 last_step=np.zeros(sc.n, np.int32))
    ev, dt = oracle_sample_step(sc, targets, rows, state, 1)
    full = all(rows >= cam.height for cam in sc.cameras)
    where = "every image row" if full else f"{rows} central image rows of each view"
    return {"value": ev / dt, "unit": UNIT, "cores": 1, "kind": "oracle", "seconds": dt,
            "sample": f"one oracle training step on {where} "
                      f"(all {sc.n} Gaussians projected; render, L1, gradients, VJP, compaction, "
                      f"deferred Adam), {int(ev)} evaluations; host has {os.cpu_count()} cores"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="medium", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--partial", type=int, default=None, metavar="S",
                    help="time the forward render as S depth slabs rendered separately and composed")
    ap.add_argument("--tile-budget", type=int, default=None, metavar="K",
                    help="prune every tile list to its K most opaque entries before rasterizing")
    ap.add_argument("--dssim", type=float, default=None, metavar="LAMBDA",
                    help="train with (1 - LAMBDA) L1 + LAMBDA D-SSIM (three raster launches instead of the fused one)")
    ap.add_argument("--seed", type=int, default=None,
                    help="seed of the synthetic scene (default: the workload's own: tiny 0 ... batched 4)")
    ap.add_argument("--log-steps", default=None, metavar="PATH",
                    help="also write one JSON line per timed step (stage ms, loss, instances, union size) to PATH")
    ap.add_argument("--cpu-rows", type=int, default=1080)
    ap.add_argument("--ref-rows", type=int, default=68)
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)   # at least 3 untimed warm-up steps
    if args.impl == "reference":
        if int(os.environ.get("RANK", "0")) != 0:
            return
        run_reference(args)
        return
    if args.partial:
        run_partial(args)
        return
    run_gpu(args)


if __name__ == "__main__":
    main()
