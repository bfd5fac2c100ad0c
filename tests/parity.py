"""Stage-by-stage parity of the CUDA path (through the C ABI) with the CPU oracle.

Test infrastructure: imported by the GPU tests and by the smoke check only.
Every comparison feeds both sides the same seeded inputs; expected values come
from the oracle alone.

Bars (the method's statement): tile lists, sort order and compacted index sets
bit-exact; images within 1e-5 absolute; gradients within relative 2e-3 with an
absolute floor of 1e-6.  Projection records, evaluation counts and the touched
set are compared bit for bit as well, since the forward decisions are
specified to be reproducible (IEEE operations in a fixed order and one
portable exp on both sides).

Gradients pass two bars, both asserted.  The literal one, |gpu - ref| <=
1e-6 + 2e-3 |ref|, says little at full size: the L1 loss is a mean over 3HW
values, so at 1080p a pixel's dL/dC is 1.6e-7 and most gradient entries are
below the 1e-6 floor.  The scaled one reads "relative 2e-3, a margin for the
order of atomic accumulation" against what a sum in another order can change:
|gpu - ref| <= 2e-3 M + 1e-6 max(M), with M the oracle's sum of the magnitudes
of the terms each entry is made of (grad2d: ``grad2d_mag``; dense gradients:
sum_k |d param / d grad2d_k| M_k over views, ``oracle.vjp_mag``) and max(M)
taken per gradient component (grad2d column, parameter row).  M >= |ref|, and
M = |ref| where the terms do not cancel, so there the bar is 2e-3 |ref|.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from differentiable_rasterizer_gb300 import pipeline, scenes

IMG_ATOL = 1e-5
GRAD_RTOL = 2e-3
GRAD_ATOL = 1e-6


def oracle_targets(sc, prec="f32"):
    """Targets [V,3,H,W]: the scene's uniform noise, or the oracle's render of the perturbed scene."""
    if sc.target_kind == "uniform":
        return np.ascontiguousarray(sc.target_uniform, np.float32)
    out = []
    for cam in sc.cameras:
        pr = oracle.project(sc.perturbed_params, sc.sh_degree, cam, sc.opts, prec)
        out.append(oracle.render(pr, cam, sc.opts, prec=prec)["image"])
    return np.ascontiguousarray(np.stack(out), np.float32)


def bits(a):
    a = np.ascontiguousarray(a)
    return a.view(np.uint32) if a.dtype == np.float32 else a.view(np.uint64)


def grad_report(gpu, ref, mag=None, axis=0, rtol=GRAD_RTOL, atol=GRAD_ATOL):
    """(ok, stats) for the literal bar |gpu - ref| <= atol + rtol |ref| and, with
    ``mag`` (same shape as ref: the oracle's sum of term magnitudes), the scaled
    bar |gpu - ref| <= rtol mag + atol max(mag), max taken along ``axis`` (the axis
    over Gaussians: 0 for [m, 9] grad2d rows, 1 for [P, n] dense gradients)."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(gpu - ref)
    ok = err <= atol + rtol * np.abs(ref)
    scale = np.abs(ref).max() if ref.size else 0.0
    big = np.abs(ref) > 1e-3 * scale
    rel_big = (err[big] / np.abs(ref[big])).max() if big.any() else 0.0
    st = dict(n=int(ref.size), bad=int((~ok).sum()), max_abs_err=float(err.max(initial=0.0)),
              max_abs_ref=float(scale), max_rel_err_significant=float(rel_big), n_significant=int(big.sum()))
    if mag is not None:
        mag = np.asarray(mag, np.float64)
        assert mag.shape == ref.shape
        floor = mag.max(axis=axis, keepdims=True, initial=0.0) if mag.size else mag
        tol = rtol * mag + atol * floor
        ok_s = err <= tol
        st.update(bad_scaled=int((~ok_s).sum()),
                  max_err_over_scaled_tol=float((err / np.maximum(tol, 1e-300)).max(initial=0.0)),
                  max_err_over_mag=float((err / np.maximum(mag, 1e-300)).max(initial=0.0)))
        ok = ok & ok_s
    return bool(ok.all()), st


def run_stage_parity(sc, targets=None, device="cuda", check_adam=True, log=print):
    """Runs one full step stage by stage on the GPU and checks every stage against the oracle.

    Returns a dict of statistics; raises AssertionError on any mismatch."""
    stats = {}
    if targets is None:
        targets = oracle_targets(sc)
    V, n = sc.n_views, sc.n
    tr = pipeline.GaussianTrainer(sc.params, sc.sh_degree, sc.cameras, sc.opts, sc.lr, device=device)
    tgt_dev = torch.from_numpy(targets).to(device)
    P = sc.params.shape[0]

    # --- A1 projection: records bit-exact
    tr.project()
    torch.cuda.synchronize()
    rec = tr.rec.cpu().numpy()
    tt = tr.tiles_touched.cpu().numpy().view(np.uint32)
    rect = tr.rect.cpu().numpy().view(np.uint16)
    depth = tr.depth.cpu().numpy()
    oprojs = []
    for v, cam in enumerate(sc.cameras):
        pr = oracle.project(sc.params, sc.sh_degree, cam, sc.opts)
        oprojs.append(pr)
        vis = pr["visible"].astype(bool)
        assert np.array_equal(tt[v] > 0, vis), f"view {v}: visibility differs at {np.flatnonzero((tt[v] > 0) != vis)[:10]}"
        o = pr["rec"][vis]
        exp = np.stack([o[:, 0], o[:, 1], np.float32(-0.5) * o[:, 2], o[:, 3], np.float32(-0.5) * o[:, 4], o[:, 5],
                        o[:, 6], o[:, 7], o[:, 8]], 1).astype(np.float32)
        got = rec[v][vis][:, :9]
        diff = np.flatnonzero((bits(got) != bits(exp)).any(1))
        assert diff.size == 0, f"view {v}: projection records differ for {diff.size} Gaussians, e.g. " \
                               f"{np.flatnonzero(vis)[diff[:3]]}: gpu {got[diff[:1]]} oracle {exp[diff[:1]]}"
        assert np.array_equal(rect[v][vis].astype(np.int32), pr["rect"][vis])
        area = (pr["rect"][vis, 2] - pr["rect"][vis, 0]) * (pr["rect"][vis, 3] - pr["rect"][vis, 1])
        assert np.array_equal(tt[v][vis], area.astype(np.uint32))
        assert np.array_equal(bits(depth[v][vis]), bits(o[:, 9]))
    stats["visible"] = [int((tt[v] > 0).sum()) for v in range(V)]

    # --- A2 binning + sort: keys, ids and ranges bit-exact
    N = tr.bin_sort()
    torch.cuda.synchronize()
    keys = tr.keys[:N].cpu().numpy().view(np.uint64)
    ids = tr.ids[:N].cpu().numpy().view(np.uint32)
    ranges = tr.ranges.cpu().numpy().view(np.uint32).reshape(V, -1, 2)
    tiles = tr.tiles
    budget = int(sc.opts.get("tile_budget", 0))
    base = 0
    for v, cam in enumerate(sc.cameras):
        off, oids = oracle.tile_lists(oprojs[v], cam)
        m = oids.size
        tile_of = np.repeat(np.arange(tiles, dtype=np.uint64), np.diff(off).astype(np.int64))
        dbits = bits(oprojs[v]["rec"][oids, 9]).astype(np.uint64)
        exp_keys = ((np.uint64(v * tiles) + tile_of) << np.uint64(32)) | dbits
        assert np.array_equal(keys[base:base + m], exp_keys), f"view {v}: sorted keys differ"
        full = np.diff(off) > 0      # an empty tile only has to have start == end
        assert np.array_equal(ranges[v][full, 0], (off[:-1][full] + base).astype(np.uint32)), f"view {v}: range starts"
        assert np.array_equal(ranges[v][~full, 0], ranges[v][~full, 1]), f"view {v}: empty tiles"
        if not budget:
            assert np.array_equal(ids[base:base + m], oids.astype(np.uint32)), f"view {v}: sorted ids differ"
            assert np.array_equal(ranges[v][full, 1], (off[1:][full] + base).astype(np.uint32)), f"view {v}: ends"
        else:
            # pruned: each tile's kept ids at the start of its range, in list order
            offp, oidsp = oracle.tile_lists(oprojs[v], cam, budget=budget)
            lenp = np.diff(offp)
            assert np.array_equal(ranges[v][full, 1] - ranges[v][full, 0], lenp[full].astype(np.uint32)), \
                f"view {v}: pruned lengths"
            pos = np.repeat(off[:-1] + base - offp[:-1], lenp) + np.arange(offp[-1])
            assert np.array_equal(ids[pos], oidsp.astype(np.uint32)), f"view {v}: pruned ids differ"
            stats.setdefault("pruned_tiles", []).append(int((np.diff(off) > budget).sum()))
            stats.setdefault("pruned_entries", []).append(int(m - offp[-1]))
        base += m
    assert base == N
    stats["instances"] = int(N)

    # --- A3 fused raster: image, loss, counts, touched, per-Gaussian 2D gradients
    tr.eval_counts.zero_()
    tr.raster(tgt_dev)
    torch.cuda.synchronize()
    img = tr.image.cpu().numpy()
    loss = tr.loss.cpu().numpy()
    g2d = tr.grad2d.cpu().numpy()[..., :9].copy()
    touched = tr.touched.cpu().numpy().copy()
    counts = tr.eval_counts.cpu().numpy()
    efwd = ebwd = ecomp = 0
    orend = []
    for v, cam in enumerate(sc.cameras):
        out = oracle.render(oprojs[v], cam, sc.opts, target=targets[v], want_mag=True)
        orend.append(out)
        d = np.abs(img[v].astype(np.float64) - out["image"])
        stats.setdefault("img_max_abs_err", []).append(float(d.max()))
        stats.setdefault("img_exact_frac", []).append(float((bits(img[v]) == bits(out["image"])).mean()))
        assert d.max() <= IMG_ATOL, f"view {v}: image max abs err {d.max()}"
        assert abs(loss[v] - out["loss"]) <= 1e-9 * max(1.0, abs(out["loss"])), (loss[v], out["loss"])
        assert np.array_equal(touched[v], out["touched"]), f"view {v}: touched sets differ"
        tv = out["touched"] > 0
        ok, st = grad_report(g2d[v][tv], out["grad2d"][tv], out["grad2d_mag"][tv])
        stats.setdefault("grad2d", []).append(st)
        assert ok, f"view {v}: grad2d out of tolerance {st}"
        efwd += out["e_fwd"]
        ebwd += out["e_bwd"]
        ecomp += out["e_comp"]
    assert int(counts[0]) == efwd and int(counts[1]) == ebwd and int(counts[2]) == ecomp, (counts, efwd, ebwd, ecomp)
    stats["e_fwd"], stats["e_bwd"], stats["e_comp"] = efwd, ebwd, ecomp

    # --- A4 compaction + VJP + scatter-add
    tr.compact()
    torch.cuda.synchronize()
    idx = tr.idx.cpu().numpy().view(np.uint32)
    n_idx = tr.n_idx.cpu().numpy()
    ref_grads = np.zeros((P, n), np.float64)
    ref_mag = np.zeros((P, n), np.float64)
    for v, cam in enumerate(sc.cameras):
        exp_idx = oracle.compact(orend[v]["touched"])
        assert n_idx[v] == exp_idx.size and np.array_equal(idx[v][:n_idx[v]], exp_idx), f"view {v}: compacted list"
        oracle.vjp(sc.params, sc.sh_degree, cam, sc.opts, orend[v]["grad2d"], orend[v]["touched"],
                   oprojs[v]["clamp"], ref_grads)
        oracle.vjp_mag(sc.params, sc.sh_degree, cam, sc.opts, orend[v]["grad2d_mag"], orend[v]["touched"],
                       oprojs[v]["clamp"], ref_mag)
    union = oracle.compact(np.any(np.stack([o["touched"] for o in orend]), 0).astype(np.uint8))
    assert n_idx[V] == union.size and np.array_equal(idx[V][:n_idx[V]], union), "union list"
    grads = tr.rows(tr.grads).cpu().numpy()
    ok, st = grad_report(grads, ref_grads, ref_mag, axis=1)
    stats["grads"] = st
    assert ok, f"dense gradients out of tolerance {st}"
    assert not tr.grad2d.any().item() and not tr.touched.any().item(), "grad2d / touched not cleared"

    # --- A5 deferred Adam, fed the GPU's gradients: bit-exact with the oracle
    if check_adam:
        p_o = sc.params.copy()
        m_o = np.zeros_like(p_o)
        v_o = np.zeros_like(p_o)
        last_o = np.zeros(n, np.int32)
        g_o = grads.astype(np.float32).copy()
        lr_rows = scenes.lr_rows(sc.lr, sc.sh_degree)
        oracle.adam_deferred(p_o, m_o, v_o, g_o, last_o, lr_rows, union, 1, tr.betas[0], tr.betas[1], tr.eps)
        tr.adam(1)
        torch.cuda.synchronize()
        assert np.array_equal(bits(tr.rows(tr.params).cpu().numpy()), bits(p_o)), "Adam params"
        assert np.array_equal(bits(tr.rows(tr.adam_m).cpu().numpy()), bits(m_o)), "Adam m"
        assert np.array_equal(bits(tr.rows(tr.adam_v).cpu().numpy()), bits(v_o)), "Adam v"
        assert np.array_equal(tr.last_step.cpu().numpy(), last_o), "last_step"
    log(f"[parity] {sc.name}: {stats}")
    return stats


def _parallel(fn, items, threads=None):
    """fn over items on threads: each oracle call is one single-threaded C call made
    through ctypes, which releases the GIL, so independent views run side by side.
    The oracle's lazily built constants are built first, on this thread."""
    import concurrent.futures
    import os
    oracle.pexp_f32([0.0])
    oracle.sh_basis(np.array([[0.0, 0.0, 1.0]]))
    threads = threads or max(1, min(len(items), os.cpu_count() or 1))
    with concurrent.futures.ThreadPoolExecutor(threads) as ex:
        return list(ex.map(fn, items))


def run_sampled_parity(sc, check_views=None, n_tiles=48, n_gauss=300, seed=0, device="cuda", log=print):
    """Parity at full size where the oracle cannot render whole images quickly.

    Per checked view the oracle projects every Gaussian (visibility and records
    compared for all), builds every tile list (sorted keys/ids/ranges compared for
    all), and renders a sample of tiles: random ones plus every tile of a sample
    of Gaussians, so those Gaussians' 2D gradients are complete.  The sampled
    Gaussians are drawn among those whose tile rect is at most 4 tiles in every
    checked view, and their tiles are rendered in every checked view, so that with
    all views checked their gradients summed over the views are complete too.
    Images are compared on the sampled tiles; the training target of the GPU (its
    render of the perturbed scene) must equal the oracle's render of the perturbed
    scene there bit for bit, and the oracle's loss terms use the oracle's own
    target.  With every view checked, the sampled Gaussians' membership of each
    view's compacted list and of the union, their dense gradients (summed over
    the views) and their Adam update are compared as well."""
    rng = np.random.default_rng(seed)
    V, n = sc.n_views, sc.n
    views = list(range(V)) if check_views is None else list(check_views)
    tr = pipeline.GaussianTrainer(sc.params, sc.sh_degree, sc.cameras, sc.opts, sc.lr, device=device)
    pert = tr.to_device_layout(sc.perturbed_params)
    target = tr.render(pert).clone()
    del pert
    tr.project()
    torch.cuda.synchronize()
    tt = tr.tiles_touched.cpu().numpy().view(np.uint32)
    N = tr.bin_sort()
    torch.cuda.synchronize()
    keys = tr.keys[:N].cpu().numpy().view(np.uint64)
    ids = tr.ids[:N].cpu().numpy().view(np.uint32)
    ranges = tr.ranges.cpu().numpy().view(np.uint32).reshape(V, -1, 2)
    tr.eval_counts.zero_()
    tr.raster(target)
    torch.cuda.synchronize()
    img = tr.image.cpu().numpy()
    tgt_gpu = target.cpu().numpy()
    stats = dict(instances=int(N), views=views)
    tiles = tr.tiles
    tiles_x = (sc.cameras[0].width + 15) // 16

    # phase 1, per view: every record, every tile list; which Gaussians have small rects
    def lists(v):
        cam = sc.cameras[v]
        pr = oracle.project(sc.params, sc.sh_degree, cam, sc.opts)
        vis = pr["visible"].astype(bool)
        assert np.array_equal(tt[v] > 0, vis), f"view {v}: visibility"
        o = pr["rec"][vis]
        exp = np.stack([o[:, 0], o[:, 1], np.float32(-0.5) * o[:, 2], o[:, 3], np.float32(-0.5) * o[:, 4], o[:, 5],
                        o[:, 6], o[:, 7], o[:, 8]], 1).astype(np.float32)
        rec = tr.rec[v][torch.from_numpy(np.flatnonzero(vis)).to(device)].cpu().numpy()
        assert np.array_equal(bits(rec[:, :9]), bits(exp)), f"view {v}: projection records"
        del rec
        off, oids = oracle.tile_lists(pr, cam)
        base = int(ranges[v][:, 0][np.diff(off) > 0].min()) if off[-1] else 0
        m = oids.size
        assert np.array_equal(ids[base:base + m], oids.astype(np.uint32)), f"view {v}: sorted ids"
        tile_of = np.repeat(np.arange(tiles, dtype=np.uint64), np.diff(off).astype(np.int64))
        dbits = bits(pr["rec"][oids, 9]).astype(np.uint64)
        assert np.array_equal(keys[base:base + m], ((np.uint64(v * tiles) + tile_of) << np.uint64(32)) | dbits), \
            f"view {v}: sorted keys"
        full = np.diff(off) > 0
        assert np.array_equal(ranges[v][full, 0], (off[:-1][full] + base).astype(np.uint32)), f"view {v}: ranges"
        assert np.array_equal(ranges[v][full, 1], (off[1:][full] + base).astype(np.uint32)), f"view {v}: range ends"
        rect = pr["rect"]
        area = (rect[:, 2] - rect[:, 0]) * (rect[:, 3] - rect[:, 1])
        return vis, vis & (area <= 4), int(m)

    p1 = _parallel(lists, views)
    stats["checked_instances"] = int(sum(x[2] for x in p1))
    any_vis = np.zeros(n, bool)
    small_everywhere = np.ones(n, bool)
    for vis, small, _ in p1:
        any_vis |= vis
        small_everywhere &= (~vis) | small
    del p1
    cand = np.flatnonzero(any_vis & small_everywhere)
    gs = np.sort(rng.choice(cand, min(n_gauss, cand.size), replace=False))
    sub = np.ascontiguousarray(sc.params[:, gs])
    sub_pert = np.ascontiguousarray(sc.perturbed_params[:, gs])
    g2d_gpu = tr.grad2d[:, torch.from_numpy(gs).to(device)].cpu().numpy()[..., :9]
    tch_gpu = tr.touched[:, torch.from_numpy(gs).to(device)].cpu().numpy()

    # phase 2, per view: the sampled tiles rendered (target and training render)
    def tiles_of(v):
        cam = sc.cameras[v]
        prs = oracle.project(sub, sc.sh_degree, cam, sc.opts)
        rect = prs["rect"]
        mask = np.zeros(tiles, bool)
        mask[np.random.default_rng([seed, v]).choice(tiles, n_tiles, replace=False)] = True
        for k in np.flatnonzero(prs["visible"]):
            for ty in range(rect[k, 1], rect[k, 3]):
                mask[ty * tiles_x + rect[k, 0]:ty * tiles_x + rect[k, 2]] = True
        prp = oracle.project(sc.perturbed_params, sc.sh_degree, cam, sc.opts)
        otgt = oracle.render(prp, cam, sc.opts, tile_mask=mask)["image"]
        del prp
        H, W = cam.height, cam.width
        pix = np.repeat(np.repeat(mask.reshape(-1, tiles_x), 16, 0), 16, 1)[:H, :W]
        assert np.array_equal(bits(tgt_gpu[v][:, pix]), bits(otgt[:, pix])), f"view {v}: target render"
        pr = oracle.project(sc.params, sc.sh_degree, cam, sc.opts)
        out = oracle.render(pr, cam, sc.opts, target=otgt, tile_mask=mask, want_mag=True)
        d = np.abs(img[v][:, pix].astype(np.float64) - out["image"][:, pix])
        assert d.max() <= IMG_ATOL, f"view {v}: image max abs err {d.max()}"
        assert np.array_equal(tch_gpu[v], out["touched"][gs]), f"view {v}: touched (sampled)"
        ok, st = grad_report(g2d_gpu[v], out["grad2d"][gs], out["grad2d_mag"][gs])
        assert ok, f"view {v}: grad2d (sampled) {st}"
        return dict(st=st, pix=int(pix.sum()), g2=out["grad2d"][gs], mag=out["grad2d_mag"][gs],
                    tch=out["touched"][gs], clamp=pr["clamp"][gs])

    p2 = _parallel(tiles_of, views)
    stats["grad2d"] = [x["st"] for x in p2]
    stats["sampled_pixels"] = [x["pix"] for x in p2]
    stats["sampled_gaussians"] = int(gs.size)
    if len(views) == V:
        tr.compact()
        torch.cuda.synchronize()
        n_idx = tr.n_idx.cpu().numpy()
        idx = tr.idx.cpu().numpy().view(np.uint32)
        tch_any = np.zeros(gs.size, bool)
        for v in range(V):
            lst = idx[v][:n_idx[v]]
            assert np.all(np.diff(lst.astype(np.int64)) > 0), f"view {v}: compacted list not ascending"
            assert np.array_equal(np.isin(gs, lst), p2[v]["tch"] > 0), f"view {v}: compacted list (sampled)"
            tch_any |= p2[v]["tch"] > 0
        union = idx[V][:n_idx[V]]
        assert np.all(np.diff(union.astype(np.int64)) > 0), "union list not ascending"
        assert np.array_equal(np.isin(gs, union), tch_any), "union list (sampled)"
        if V > 1:
            allv = np.unique(np.concatenate([idx[v][:n_idx[v]] for v in range(V)]))
            assert np.array_equal(union, allv), "union = the per-view lists merged"
        stats["union"] = int(n_idx[V])
        ref = np.zeros(sub.shape, np.float64)
        mag = np.zeros(sub.shape, np.float64)
        for v in range(V):
            cam = sc.cameras[v]
            oracle.vjp(sub, sc.sh_degree, cam, sc.opts, p2[v]["g2"], p2[v]["tch"], p2[v]["clamp"], ref)
            oracle.vjp_mag(sub, sc.sh_degree, cam, sc.opts, p2[v]["mag"], p2[v]["tch"], p2[v]["clamp"], mag)
        gidx = torch.from_numpy(gs).to(device)
        got = tr.rows(tr.grads)[:, gidx].cpu().numpy()
        m = tch_any
        ok, st = grad_report(got[:, m], ref[:, m], mag[:, m], axis=1)
        assert ok, f"dense gradients (sampled) {st}"
        stats["grads"] = st
        # Adam for the sampled Gaussians, fed the GPU's gradients, at the scene's learning rates
        p_o = sub.copy()
        m_o = np.zeros_like(p_o)
        v_o = np.zeros_like(p_o)
        last_o = np.zeros(gs.size, np.int32)
        sel = np.flatnonzero(tch_any).astype(np.uint32)
        g_o = got.astype(np.float32).copy()
        oracle.adam_deferred(p_o, m_o, v_o, g_o, last_o, scenes.lr_rows(sc.lr, sc.sh_degree), sel, 1,
                             tr.betas[0], tr.betas[1], tr.eps)
        tr.adam(1)
        torch.cuda.synchronize()
        assert np.array_equal(bits(tr.rows(tr.params)[:, gidx].cpu().numpy()), bits(p_o)), "Adam params (sampled)"
        assert np.array_equal(bits(tr.rows(tr.adam_m)[:, gidx].cpu().numpy()), bits(m_o)), "Adam m (sampled)"
        assert np.array_equal(bits(tr.rows(tr.adam_v)[:, gidx].cpu().numpy()), bits(v_o)), "Adam v (sampled)"
        assert np.array_equal(tr.last_step[gidx].cpu().numpy(), last_o), "last_step (sampled)"
    log(f"[sampled parity] {sc.name}: {stats}")
    del tr
    torch.cuda.empty_cache()
    return stats


# ----------------------------------------------------------------------------- L1 + D-SSIM
# Bars of the D-SSIM stage, carried over from the step's own:
# - the SSIM map is an image-like per-pixel quantity: the loss, lambda times the
#   mean of 1 - S plus the L1 term, must agree within lambda * IMG_ATOL (which bounds
#   the mean of per-pixel errors of IMG_ATOL), plus half an ulp of each fp32
#   difference x - y in the L1 term;
# - dL/dC is a gradient, but the SSIM part is a sum of three terms
#   (w * dS/dmu_x + 2 x (w * dS/dE[x^2]) + y (w * dS/dE[xy])) / N that cancel
#   where x is close to y, so its relative error is taken against the sum of the
#   terms' magnitudes M (w * |dS/dmu_x| + 2|x| (w * |dS/dE[x^2]|) + |y| (w * |dS/dE[xy]|)):
#   |gpu - oracle| <= GRAD_RTOL * lambda / N * M + 4 u |oracle| + 1e-6 max|oracle|;
#   the L1 part is a signed constant that must be exact.  The last term is the
#   gradient bar's absolute floor relative to the map's scale: where the image and
#   the target are equal over a whole window M is 0, but the kernel's mean-centred
#   form leaves a residual of rounding size.
_U = 2.0 ** -24


def dssim_reference(x, y, lam):
    """Oracle loss and dL/dC of (1 - lam) L1 + lam (1 - SSIM) for images [3, H, W],
    with the elementwise and total tolerances above."""
    from oracle import dssim
    lam = float(np.float32(lam))   # the kernel is given lambda in fp32
    x = np.asarray(x, np.float64)
    y = np.asarray(y, np.float64)
    N = float(x.size)
    t = dssim.ssim_terms(x, y)
    l1 = float(np.abs(x - y).mean())
    loss = (1.0 - lam) * l1 + lam * (1.0 - float(t["S"].mean()))
    l1_part = np.sign(x - y) * float(np.float32((1.0 - lam) / N))
    g_ssim = (dssim.wsum(t["d_mu"]) + 2.0 * x * dssim.wsum(t["d_exx"]) + y * dssim.wsum(t["d_exy"])) / N
    dldc = l1_part - lam * g_ssim
    M = dssim.wsum(np.abs(t["d_mu"])) + 2 * np.abs(x) * dssim.wsum(np.abs(t["d_exx"])) \
        + np.abs(y) * dssim.wsum(np.abs(t["d_exy"]))
    tol = GRAD_RTOL * lam / N * M + 4 * _U * np.abs(dldc) + 1e-6 * float(np.abs(dldc).max())
    tol_loss = lam * IMG_ATOL + (1.0 - lam) * _U * l1 + 1e-12 * abs(loss)
    return dict(loss=loss, dldc=dldc, tol=tol, tol_loss=tol_loss, M=lam / N * M)


def check_dssim_stage(img, tgt, lam, loss_gpu, dldc_gpu, stats=None, tag=""):
    """GPU loss and dL/dC of the D-SSIM stage against the oracle on the same images."""
    ref = dssim_reference(img, tgt, lam)
    err = np.abs(np.asarray(dldc_gpu, np.float64) - ref["dldc"])
    bad = err > ref["tol"]
    assert not bad.any(), f"{tag} dL/dC out of tolerance at {np.argwhere(bad)[:5].tolist()}: " \
                          f"gpu {np.asarray(dldc_gpu)[bad][:3]} oracle {ref['dldc'][bad][:3]} tol {ref['tol'][bad][:3]}"
    assert abs(loss_gpu - ref["loss"]) <= ref["tol_loss"], (tag, loss_gpu, ref["loss"], ref["tol_loss"])
    if stats is not None:
        scale = np.maximum(ref["M"], 1e-300)
        stats.setdefault("dldc_err_over_M", []).append(float((err / scale).max()) if lam > 0 else 0.0)
        stats.setdefault("dldc_err_over_tol", []).append(float((err / ref["tol"]).max()))
        stats.setdefault("loss_err", []).append(float(abs(loss_gpu - ref["loss"])))
        stats.setdefault("loss_tol", []).append(float(ref["tol_loss"]))


def run_dssim_parity(sc, lam=0.2, targets=None, device="cuda", log=print):
    """One L1 + D-SSIM step stage by stage: forward with stored state (image, final
    T, last index, counts), the loss and dL/dC, the backward from the stored state
    (fed the GPU's dL/dC on both sides), compaction + VJP."""
    stats = {}
    if targets is None:
        targets = oracle_targets(sc)
    V, n = sc.n_views, sc.n
    P = sc.params.shape[0]
    tr = pipeline.GaussianTrainer(sc.params, sc.sh_degree, sc.cameras, sc.opts, sc.lr, device=device,
                                  dssim_lambda=lam)
    tgt_dev = torch.from_numpy(targets).to(device)
    tr.project()
    tr.bin_sort()
    tr.eval_counts.zero_()
    tr.raster(tgt_dev)
    torch.cuda.synchronize()
    img = tr.image.cpu().numpy()
    tfin = tr.t_final.cpu().numpy()
    last = tr.last_idx.cpu().numpy()
    loss = tr.loss.cpu().numpy()
    dldc = tr.dldc.cpu().numpy()
    g2d = tr.grad2d.cpu().numpy()[..., :9].copy()
    touched = tr.touched.cpu().numpy().copy()
    counts = tr.eval_counts.cpu().numpy()
    ref_grads = np.zeros((P, n), np.float64)
    ref_mag = np.zeros((P, n), np.float64)
    ef = eb = ec = 0
    touched_o = []
    for v, cam in enumerate(sc.cameras):
        pr = oracle.project(sc.params, sc.sh_degree, cam, sc.opts)
        fw = oracle.render(pr, cam, sc.opts, want_last=True, want_tfinal=True)
        d = np.abs(img[v].astype(np.float64) - fw["image"])
        assert d.max() <= IMG_ATOL, f"view {v}: image max abs err {d.max()}"
        assert np.array_equal(last[v], fw["last"]), f"view {v}: last index differs"
        assert np.abs(tfin[v].astype(np.float64) - fw["t_final"]).max() <= 1e-6, f"view {v}: final T"
        stats.setdefault("t_final_exact_frac", []).append(float((bits(tfin[v]) == bits(fw["t_final"])).mean()))
        ef += fw["e_fwd"]
        eb += fw["e_bwd"]
        ec += fw["e_comp"]
        check_dssim_stage(img[v], targets[v], lam, loss[v], dldc[v], stats, tag=f"view {v}")
        bw = oracle.render(pr, cam, sc.opts, target=targets[v], dldc_extra=dldc[v], l1_weight=0.0, want_mag=True)
        assert np.array_equal(touched[v], bw["touched"]), f"view {v}: touched sets differ"
        tv = bw["touched"] > 0
        ok, st = grad_report(g2d[v][tv], bw["grad2d"][tv], bw["grad2d_mag"][tv])
        stats.setdefault("grad2d", []).append(st)
        assert ok, f"view {v}: grad2d out of tolerance {st}"
        oracle.vjp(sc.params, sc.sh_degree, cam, sc.opts, bw["grad2d"], bw["touched"], pr["clamp"], ref_grads)
        oracle.vjp_mag(sc.params, sc.sh_degree, cam, sc.opts, bw["grad2d_mag"], bw["touched"], pr["clamp"], ref_mag)
        touched_o.append(bw["touched"])
    assert (int(counts[0]), int(counts[1]), int(counts[2])) == (ef, eb, ec), (counts, ef, eb, ec)
    tr.compact()
    torch.cuda.synchronize()
    union = oracle.compact(np.any(np.stack(touched_o), 0).astype(np.uint8))
    n_idx = tr.n_idx.cpu().numpy()
    assert n_idx[V] == union.size and np.array_equal(tr.idx.cpu().numpy().view(np.uint32)[V][:n_idx[V]], union)
    ok, st = grad_report(tr.rows(tr.grads).cpu().numpy(), ref_grads, ref_mag, axis=1)
    stats["grads"] = st
    assert ok, f"dense gradients out of tolerance {st}"
    log(f"[dssim parity] {sc.name} lambda={lam}: {stats}")
    return stats


# ----------------------------------------------------------------------------- partial render + compose
def depth_splits(sc, S):
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
    """Partial render + compose of S depth slabs against the oracle: slab sub-ranges,
    each slab's (C, T), the composition, and the one-pass render within the stop bound."""
    splits = depth_splits(sc, S)
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
            assert np.abs(cparts[s, v].astype(np.float64) - Cs).max() <= IMG_ATOL, f"view {v} slab {s}: C"
            assert np.abs(tparts[s, v].astype(np.float64) - Ts).max() <= 1e-6, f"view {v} slab {s}: T"
        C, T = oracle.compose(parts, sc.opts["bg"])
        d = np.abs(img[v].astype(np.float64) - C)
        assert d.max() <= IMG_ATOL, f"view {v}: composed image {d.max()}"
        assert np.abs(tcomp[v] - T).max() <= 1e-6
        one = oracle.render(pr, cam, sc.opts)["image"].astype(np.float64)
        cmax = max(float(pr["rec"][pr["visible"] > 0, 6:9].max(initial=0.0)), max(sc.opts["bg"]))
        # T where a pixel stops: below t_min, or (crossing entry excluded) below t_min / (1 - alpha_max)
        t_stop = sc.opts["t_min"] / ((1.0 - sc.opts["alpha_max"]) if sc.opts.get("exclude_crossing") else 1.0)
        d1 = np.abs(img[v].astype(np.float64) - one)
        assert d1.max() <= t_stop * cmax + IMG_ATOL, f"view {v}: vs one pass {d1.max()}"
        stats.setdefault("vs_one_pass_max", []).append(float(d1.max()))
        stats.setdefault("vs_compose_max", []).append(float(d.max()))
    print(f"[compose parity] {sc.name} S={S}: {stats}")
    return stats
