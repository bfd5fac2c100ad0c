"""CPU oracle for the 3DGS training step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It wraps ``gs_oracle.c`` (plain C,
single-threaded, untiled) through ctypes and shares no code with the CUDA path.

Every function takes the seeded inputs as numpy arrays.  ``prec`` selects the
fp32 build (the precision the workloads fix; its forward decisions are the
reference for bit-exact indexing) or the fp64 build (finite-difference checks).
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gs_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libgs_oracle.so")

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-ffp-contract=off", "-fno-fast-math", "-Wall", "-Wno-unused-function"]
# fmaf() is correctly rounded by definition; on x86-64 let it be the FMA instruction
# instead of libm's software emulation (same results, much faster).  aarch64 has it natively.
if platform.machine() in ("x86_64", "AMD64"):
    CFLAGS += ["-mfma"]


def build(force: bool = False) -> str:
    """Compile gs_oracle.c in both precisions into one shared library."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    o32 = os.path.join(os.path.dirname(_LIB), "gs_oracle_f32.o")
    o64 = os.path.join(os.path.dirname(_LIB), "gs_oracle_f64.o")
    subprocess.check_call(["gcc", *CFLAGS, "-DREAL=float", "-c", _SRC, "-o", o32])
    subprocess.check_call(["gcc", *CFLAGS, "-DREAL=double", "-DREAL_IS_DOUBLE", "-c", _SRC, "-o", o64])
    tmp = _LIB + ".tmp%d" % os.getpid()
    subprocess.check_call(["gcc", "-shared", "-o", tmp, o32, o64, "-lm"])
    os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        _declare(_lib)
    return _lib


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int


def _declare(L):
    for s in ("_f32", "_f64"):
        getattr(L, "oracle_project" + s).argtypes = [_P, _I64, _I32, _P, _I32, _I32, _P, _P, _P, _P, _P]
        getattr(L, "oracle_project" + s).restype = _I32
        getattr(L, "oracle_render" + s).argtypes = [_P, _P, _P, _I64, _I32, _I32, _P, _I32, _P, _P, _P, _P, _P, _P, _P, _P,
                                                    _P, _P, ctypes.c_double, _P, _P]
        getattr(L, "oracle_render" + s).restype = _I32
        getattr(L, "oracle_vjp" + s).argtypes = [_P, _I64, _I32, _P, _I32, _I32, _P, _P, _P, _P, _P]
        getattr(L, "oracle_vjp" + s).restype = _I32
        getattr(L, "oracle_tile_lists" + s).argtypes = [_P, _P, _P, _I64, _I32, _I32, _I64, _P, _P]
        getattr(L, "oracle_tile_lists" + s).restype = _I64
        getattr(L, "oracle_compact" + s).argtypes = [_P, _I64, _P]
        getattr(L, "oracle_compact" + s).restype = _I64
        getattr(L, "oracle_sh_basis" + s).argtypes = [_P, _I64, _P]
        getattr(L, "oracle_sh_basis" + s).restype = None
        getattr(L, "oracle_adam_dense_step" + s).argtypes = [_P, _P, _P, _P, _I64, _I64, _P, _I32] + [ctypes.c_float if s == "_f32" else ctypes.c_double] * 3
        getattr(L, "oracle_adam_dense_step" + s).restype = None
        getattr(L, "oracle_adam_deferred" + s).argtypes = [_P, _P, _P, _P, _P, _I64, _I64, _P, _P, _I64, _I32] + [ctypes.c_float if s == "_f32" else ctypes.c_double] * 3 + [_I32]
        getattr(L, "oracle_adam_deferred" + s).restype = None
    L.oracle_pexp_f32.argtypes = [ctypes.c_float]
    L.oracle_pexp_f32.restype = ctypes.c_float


def _dt(prec):
    return np.float32 if prec == "f32" else np.float64


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def cam16(cam) -> np.ndarray:
    """Camera as 16 doubles: R (row-major), t, fx, fy, cx, cy (values taken from float32)."""
    R = np.asarray(cam.R, np.float32).reshape(9)
    t = np.asarray(cam.t, np.float32).reshape(3)
    v = np.concatenate([R, t, np.asarray([cam.fx, cam.fy, cam.cx, cam.cy], np.float32)]).astype(np.float64)
    return np.ascontiguousarray(v)


def optsv(opts: dict) -> np.ndarray:
    """Options as 10 doubles: near_z, lowpass, alpha_min, alpha_max, t_min, bg (3),
    exclude_crossing, tile_budget (0: no pruning; values taken from float32 where fp)."""
    f = lambda x: float(np.float32(x))
    return np.array([f(opts["near_z"]), f(opts["lowpass"]), f(opts["alpha_min"]), f(opts["alpha_max"]),
                     f(opts["t_min"]), f(opts["bg"][0]), f(opts["bg"][1]), f(opts["bg"][2]),
                     float(opts.get("exclude_crossing", 0)), float(int(opts.get("tile_budget", 0)))], np.float64)


def pexp_f32(x) -> np.ndarray:
    """The portable fp32 exponential, element by element."""
    L = lib()
    x = np.asarray(x, np.float32).ravel()
    return np.array([L.oracle_pexp_f32(float(v)) for v in x], np.float32)


def sh_basis(dirs, prec="f32"):
    dt = _dt(prec)
    d = np.ascontiguousarray(np.asarray(dirs, dt).reshape(-1, 3))
    out = np.zeros((d.shape[0], 16), dt)
    getattr(lib(), "oracle_sh_basis_" + prec)(_ptr(d), d.shape[0], _ptr(out))
    return out


def project(params, sh_degree, cam, opts, prec="f32"):
    """O1..O6 for one view. Returns dict(rec[n,10], rect[n,4], visible[n], clamp[n])."""
    dt = _dt(prec)
    p = np.ascontiguousarray(np.asarray(params, dt))
    n = p.shape[1]
    rec = np.zeros((n, 10), dt)
    rect = np.zeros((n, 4), np.int32)
    vis = np.zeros(n, np.uint8)
    clamp = np.zeros(n, np.uint8)
    c = cam16(cam)
    o = optsv(opts)
    rc = getattr(lib(), "oracle_project_" + prec)(_ptr(p), n, sh_degree, _ptr(c), cam.width, cam.height, _ptr(o),
                                                   _ptr(rec), _ptr(rect), _ptr(vis), _ptr(clamp))
    assert rc == 0
    return dict(rec=rec, rect=rect, visible=vis, clamp=clamp)


def render(proj, cam, opts, target=None, mode=1, grads=True, prec="f32", want_last=False, want_sig=False,
           tile_mask=None, dldc_extra=None, l1_weight=1.0, want_tfinal=False, want_mag=False):
    """O7..O10 for one view.  target: [3,H,W] or None (forward only).
    tile_mask: None or [tiles] bool -- render only those tiles (others stay 0).
    dldc_extra: None or [3,H,W] -- another loss term's dL/dC added to the weighted L1 one.
    l1_weight: weight of the L1 term in the loss (and its gradient).
    want_tfinal: also return the per-pixel final transmittance ("t_final", [H, W]).
    want_mag: also return "grad2d_mag" [n, 9]: per entry the sum of the magnitudes of
    the terms grad2d sums (each term with its inner sums taken by absolute value),
    the scale of the comparison tolerance."""
    dt = _dt(prec)
    rec, rect, vis = proj["rec"], proj["rect"], proj["visible"]
    n = rec.shape[0]
    H, W = cam.height, cam.width
    img = np.zeros((3, H, W), dt)
    loss = np.zeros(1, np.float64)
    g2 = np.zeros((n, 9), np.float64) if (grads and target is not None) else None
    g2m = np.zeros((n, 9), np.float64) if (want_mag and g2 is not None) else None
    touched = np.zeros(n, np.uint8)
    counts = np.zeros(3, np.int64)
    last = np.zeros(H * W, np.int32) if want_last else None
    tfin = np.zeros(H * W, dt) if want_tfinal else None
    sig = np.zeros(1, np.uint64) if want_sig else None
    tgt = np.ascontiguousarray(np.asarray(target, dt)) if target is not None else None
    tm = np.ascontiguousarray(np.asarray(tile_mask, np.uint8)) if tile_mask is not None else None
    ex = np.ascontiguousarray(np.asarray(dldc_extra, dt)) if dldc_extra is not None else None
    rc = getattr(lib(), "oracle_render_" + prec)(_ptr(rec), _ptr(rect), _ptr(vis), n, W, H, _ptr(optsv(opts)), mode,
                                                  _ptr(tgt), _ptr(img), _ptr(loss), _ptr(g2), _ptr(touched),
                                                  _ptr(counts), _ptr(last), _ptr(sig), _ptr(tm),
                                                  _ptr(ex), float(l1_weight), _ptr(tfin), _ptr(g2m))
    assert rc == 0
    out = dict(image=img, loss=float(loss[0]) if target is not None else None, grad2d=g2, touched=touched,
               e_fwd=int(counts[0]), e_bwd=int(counts[1]), e_comp=int(counts[2]))
    if want_last:
        out["last"] = last.reshape(H, W)
    if want_sig:
        out["sig"] = int(sig[0])
    if want_tfinal:
        out["t_final"] = tfin.reshape(H, W)
    if g2m is not None:
        out["grad2d_mag"] = g2m
    return out


def vjp(params, sh_degree, cam, opts, grad2d, touched, clamp, grads=None, prec="f32"):
    """Projection VJP: accumulates d loss / d params ([P, n] fp64) for touched Gaussians."""
    dt = _dt(prec)
    p = np.ascontiguousarray(np.asarray(params, dt))
    P, n = p.shape
    if grads is None:
        grads = np.zeros((P, n), np.float64)
    rc = getattr(lib(), "oracle_vjp_" + prec)(_ptr(p), n, sh_degree, _ptr(cam16(cam)), cam.width, cam.height,
                                               _ptr(optsv(opts)), _ptr(np.ascontiguousarray(grad2d, np.float64)),
                                               _ptr(np.ascontiguousarray(touched, np.uint8)),
                                               _ptr(np.ascontiguousarray(clamp, np.uint8)), _ptr(grads))
    assert rc == 0
    return grads


def vjp_mag(params, sh_degree, cam, opts, grad2d_mag, touched, clamp, out=None):
    """Scale of the dense gradient's comparison tolerance, accumulated (+=) into
    ``out`` [P, n]: sum over the nine 2D gradient components k of
    |d param / d grad2d_k| * grad2d_mag[:, k].  The VJP is linear in grad2d, so
    each column's Jacobian row comes from one VJP call with only that column set."""
    P, n = np.shape(params)
    if out is None:
        out = np.zeros((P, n), np.float64)
    sel = np.flatnonzero(np.asarray(touched))
    p = np.ascontiguousarray(np.asarray(params, np.float32)[:, sel])
    m = np.asarray(grad2d_mag, np.float64)[sel]
    one = np.ones(sel.size, np.uint8)
    cl = np.ascontiguousarray(np.asarray(clamp, np.uint8)[sel])
    acc = np.zeros((P, sel.size), np.float64)
    for k in range(9):
        col = np.zeros((sel.size, 9), np.float64)
        col[:, k] = m[:, k]
        acc += np.abs(vjp(p, sh_degree, cam, opts, col, one, cl))
    out[:, sel] += acc
    return out


def tile_lists(proj, cam, prec="f32", budget=0):
    """Sorted per-tile candidate lists: (offsets[tiles+1], ids[I]); budget > 0: pruned lists."""
    rec, rect, vis = proj["rec"], proj["rect"], proj["visible"]
    n = rec.shape[0]
    tiles = ((cam.width + 15) // 16) * ((cam.height + 15) // 16)
    off = np.zeros(tiles + 1, np.int64)
    L = getattr(lib(), "oracle_tile_lists_" + prec)
    total = L(_ptr(rec), _ptr(rect), _ptr(vis), n, cam.width, cam.height, int(budget), _ptr(off), None)
    ids = np.zeros(max(total, 1), np.int64)
    total = L(_ptr(rec), _ptr(rect), _ptr(vis), n, cam.width, cam.height, int(budget), _ptr(off), _ptr(ids))
    assert total >= 0
    return off, ids[:total]


def compact(touched, prec="f32"):
    t = np.ascontiguousarray(touched, np.uint8)
    idx = np.zeros(max(t.size, 1), np.uint32)
    m = getattr(lib(), "oracle_compact_" + prec)(_ptr(t), t.size, _ptr(idx))
    return idx[:m]


def adam_dense_step(p, m, v, g, lr_rows, t, b1, b2, eps, prec="f32"):
    """One dense Adam step in place on [rows, n] arrays."""
    rows, n = p.shape
    getattr(lib(), "oracle_adam_dense_step_" + prec)(_ptr(p), _ptr(m), _ptr(v), _ptr(g), rows, n,
                                                     _ptr(np.ascontiguousarray(lr_rows, _dt(prec))), t, b1, b2, eps)


def adam_deferred(p, m, v, g, last_step, lr_rows, idx, t, b1, b2, eps, flush=False, prec="f32"):
    """Deferred Adam in place: listed Gaussians catch up and step; flush brings all to t."""
    rows, n = p.shape
    idx = np.ascontiguousarray(idx if idx is not None else np.zeros(0, np.uint32), np.uint32)
    getattr(lib(), "oracle_adam_deferred_" + prec)(_ptr(p), _ptr(m), _ptr(v), _ptr(g), _ptr(last_step), rows, n,
                                                   _ptr(np.ascontiguousarray(lr_rows, _dt(prec))), _ptr(idx), idx.size,
                                                   t, b1, b2, eps, 1 if flush else 0)


def train_step(scene, targets, state, t, lr_rows, betas, eps, mode=1, prec="f32"):
    """One full step O1..O12 over all views of ``scene`` (CPU baseline and parity reference).

    targets: [V,3,H,W].  state: dict(params, m, v, last_step) updated in place
    (fp32 arrays for prec f32).  lr_rows: one learning rate per parameter row.
    Returns dict with per-view outputs, the fp64 gradient sum and the union list.
    """
    from_params = state["params"]
    P, n = from_params.shape
    grads = np.zeros((P, n), np.float64)
    views = []
    for vi, cam in enumerate(scene.cameras):
        pr = project(from_params, scene.sh_degree, cam, scene.opts, prec=prec)
        rr = render(pr, cam, scene.opts, target=targets[vi], mode=mode, prec=prec)
        idx = compact(rr["touched"])
        vjp(from_params, scene.sh_degree, cam, scene.opts, rr["grad2d"], rr["touched"], pr["clamp"], grads, prec=prec)
        views.append(dict(proj=pr, render=rr, idx=idx))
    union = compact(np.any(np.stack([v["render"]["touched"] for v in views]), axis=0).astype(np.uint8))
    g = grads.astype(_dt(prec))
    lr = np.asarray(lr_rows, _dt(prec))
    adam_deferred(state["params"], state["m"], state["v"], g, state["last_step"], lr, union, t,
                  betas[0], betas[1], eps, prec=prec)
    return dict(views=views, grads=grads, union=union)


def render_subsets(proj, cam, opts, splits, prec="f32"):
    """Partial renders of disjoint depth slabs (Splaxel, English abstract: each part
    renders its local subset of Gaussians; the partial pixel values are composed).

    splits: ascending depths z_1 < ... < z_{S-1}; slab s holds the visible Gaussians
    with z_s <= depth < z_{s+1} (z_0 = -inf, z_S = +inf).  Each slab is rendered on
    its own with a zero background.  Returns a list of (C [3,H,W], T [H,W])."""
    z = np.concatenate([[-np.inf], np.asarray(splits, np.float64), [np.inf]])
    depth = proj["rec"][:, 9].astype(np.float64)
    parts = []
    for s in range(z.size - 1):
        sub = dict(proj)
        sub["visible"] = (proj["visible"].astype(bool) & (depth >= z[s]) & (depth < z[s + 1])).astype(np.uint8)
        out = render(sub, cam, dict(opts, bg=(0.0, 0.0, 0.0)), prec=prec, want_tfinal=True)
        parts.append((out["image"], out["t_final"]))
    return parts


def compose(parts, bg):
    """Front-to-back composition of partial renders, in fp64:
    C = sum_s (prod_{j<s} T_j) C_s + (prod_s T_s) bg, T = prod_s T_s."""
    C = np.zeros(parts[0][0].shape, np.float64)
    T = np.ones(parts[0][1].shape, np.float64)
    for Cs, Ts in parts:
        C += T[None] * Cs.astype(np.float64)
        T *= Ts.astype(np.float64)
    C += T[None] * np.asarray([float(np.float32(b)) for b in bg], np.float64)[:, None, None]
    return C, T
