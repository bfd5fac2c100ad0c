"""ctypes binding of the C ABI in ``include/gs.h`` (argument marshalling only).

Every function here has the name of the C entry point it calls and takes device
pointers as Python ints (``tensor.data_ptr()``), host structs for cameras and
options, and a stream handle (``torch.cuda.current_stream().cuda_stream``).
All computation happens in ``libgs_gb300.so``; if that library has not been
built, ``lib()`` raises -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libgs_gb300.so")
CHECKED_LIB_PATH = os.path.join(_HERE, "_build", "libgs_gb300_checked.so")

GS_OK, GS_ERR_INVALID_ARG, GS_ERR_CAPACITY, GS_ERR_CUDA, GS_ERR_TIMEOUT, GS_ERR_DEVICE = range(6)
GS_TILE = 16
GS_MAX_VIEWS = 32
GS_REC_FLOAT4 = 3
GS_GRAD2D_STRIDE = 12

EXPORTS = ("gs_project", "gs_bin_sort", "gs_raster_fused_fwd_bwd", "gs_grad_compact", "gs_adam_deferred",
           "gs_raster_forward_state", "gs_dssim_loss_grad", "gs_raster_backward_state", "gs_grad_compact_static",
           "gs_prune_tiles", "gs_split_ranges", "gs_compose", "gs_raster_work_counts", "gs_check_report",
           "gs_error_string", "gs_param_rows", "gs_param_stride", "gs_num_tiles", "gs_version")


class GsCamera(ctypes.Structure):
    _fields_ = [("R", ctypes.c_float * 9), ("t", ctypes.c_float * 3), ("fx", ctypes.c_float), ("fy", ctypes.c_float),
                ("cx", ctypes.c_float), ("cy", ctypes.c_float), ("width", ctypes.c_int32), ("height", ctypes.c_int32)]


class GsRenderOpts(ctypes.Structure):
    _fields_ = [("near_z", ctypes.c_float), ("lowpass", ctypes.c_float), ("alpha_min", ctypes.c_float),
                ("alpha_max", ctypes.c_float), ("t_min", ctypes.c_float), ("bg", ctypes.c_float * 3),
                ("exclude_crossing", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class GsProj(ctypes.Structure):
    _fields_ = [("rec", ctypes.c_void_p), ("depth", ctypes.c_void_p), ("rect", ctypes.c_void_p),
                ("tiles_touched", ctypes.c_void_p)]


class GsError(RuntimeError):
    def __init__(self, name, status, extra=""):
        self.status = status
        msg = lib().gs_error_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{name} failed: {msg} (status {status}){extra}")


_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_F = ctypes.c_float


def lib_path() -> str:
    """The library lib() loads: the bounds-checked build when the environment sets
    GS_CHECKED=1 (read once, at the first load), else the plain one."""
    return CHECKED_LIB_PATH if os.environ.get("GS_CHECKED", "") == "1" else LIB_PATH


def lib():
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library missing: {path}; build it with "
                               "`python -m differentiable_rasterizer_gb300.build`")
        L = ctypes.CDLL(path)
        L.gs_project.argtypes = [_P, _I64, _I32, _P, _I32, _P, ctypes.POINTER(GsProj), _P]
        L.gs_bin_sort.argtypes = [ctypes.POINTER(GsProj), _I64, _I32, _I32, _I32, _I64, _P, _P, _P,
                                  ctypes.POINTER(ctypes.c_int64), _P, ctypes.POINTER(ctypes.c_size_t), _P]
        L.gs_raster_fused_fwd_bwd.argtypes = [ctypes.POINTER(GsProj), _I64, _P, _P, _P, _I32, _P, _P, _P, _P, _P, _P,
                                              _P, _P, _I64, _P]
        L.gs_grad_compact.argtypes = [_P, _P, _P, _I64, _I32, _P, _I32, _P, _P, _P, _P, _P,
                                      ctypes.POINTER(ctypes.c_size_t), _P]
        L.gs_adam_deferred.argtypes = [_P, _P, _P, _P, _P, _I64, _I32, _P, _P, _I32, _P, _F, _F, _F, _I32, _P]
        L.gs_raster_forward_state.argtypes = [ctypes.POINTER(GsProj), _I64, _P, _P, _P, _I32, _P, _P, _P, _P, _P, _I64,
                                              _P, _P]
        L.gs_dssim_loss_grad.argtypes = [_P, _P, _I32, _I32, _I32, _F, _P, _P, _P]
        L.gs_raster_backward_state.argtypes = [ctypes.POINTER(GsProj), _I64, _P, _P, _P, _I32, _P, _P, _P, _P, _I64,
                                               _P, _P, _P, _P]
        L.gs_prune_tiles.argtypes = [ctypes.POINTER(GsProj), _I64, _I32, _I32, _I32, _I32, _P, _P, _P]
        L.gs_split_ranges.argtypes = [_P, _P, _I32, _I32, _I32, _I32, _P, _P, _P]
        L.gs_compose.argtypes = [_P, _P, _I32, _I32, _I32, _I32, _P, _P, _P, _P]
        L.gs_raster_work_counts.argtypes = [ctypes.POINTER(GsProj), _I64, _P, _P, _P, _I32, _P, _P, _P, _P, _P, _P,
                                            _P, _P, _I64, _P]
        for name in ("gs_project", "gs_bin_sort", "gs_raster_fused_fwd_bwd", "gs_grad_compact", "gs_adam_deferred",
                     "gs_raster_forward_state", "gs_dssim_loss_grad", "gs_raster_backward_state", "gs_prune_tiles",
                     "gs_split_ranges", "gs_compose", "gs_raster_work_counts"):
            getattr(L, name).restype = ctypes.c_int
        L.gs_check_report.argtypes = [_P, ctypes.POINTER(ctypes.c_int32)]
        L.gs_check_report.restype = ctypes.c_int
        L.gs_error_string.argtypes = [ctypes.c_int]
        L.gs_error_string.restype = ctypes.c_char_p
        L.gs_param_rows.argtypes = [_I32]
        L.gs_param_rows.restype = _I32
        L.gs_param_stride.argtypes = [_I32]
        L.gs_param_stride.restype = _I32
        L.gs_num_tiles.argtypes = [_I32, _I32]
        L.gs_num_tiles.restype = _I64
        L.gs_version.argtypes = []
        L.gs_version.restype = ctypes.c_char_p
        _lib = L
    return _lib


def _check(name, st, extra=""):
    if st != GS_OK:
        raise GsError(name, st, extra)


def cameras(cams) -> ctypes.Array:
    """Host array of gs_camera from objects with R, t, fx, fy, cx, cy, width, height."""
    arr = (GsCamera * len(cams))()
    for i, c in enumerate(cams):
        R = [float(x) for x in np.asarray(c.R, np.float32).reshape(9)]
        t = [float(x) for x in np.asarray(c.t, np.float32).reshape(3)]
        arr[i].R[:] = R
        arr[i].t[:] = t
        arr[i].fx, arr[i].fy, arr[i].cx, arr[i].cy = c.fx, c.fy, c.cx, c.cy
        arr[i].width, arr[i].height = c.width, c.height
    return arr


def render_opts(opts: dict) -> GsRenderOpts:
    o = GsRenderOpts()
    o.near_z, o.lowpass = opts["near_z"], opts["lowpass"]
    o.alpha_min, o.alpha_max, o.t_min = float(opts["alpha_min"]), opts["alpha_max"], opts["t_min"]
    o.bg[:] = [float(b) for b in opts["bg"]]
    o.exclude_crossing = int(opts.get("exclude_crossing", 0))
    return o


def proj_struct(rec, depth, rect, tiles_touched) -> GsProj:
    return GsProj(rec, depth, rect, tiles_touched)


def gs_project(params, n, sh_degree, cams, n_views, opts, proj, stream):
    _check("gs_project", lib().gs_project(params, n, sh_degree, cams, n_views, ctypes.byref(opts),
                                          ctypes.byref(proj), stream))


def gs_bin_sort_ws_bytes(n, n_views, width, height, capacity) -> int:
    sz = ctypes.c_size_t(0)
    cnt = ctypes.c_int64(0)
    _check("gs_bin_sort", lib().gs_bin_sort(None, n, n_views, width, height, capacity, None, None, None,
                                            ctypes.byref(cnt), None, ctypes.byref(sz), None))
    return sz.value


def gs_bin_sort(proj, n, n_views, width, height, capacity, keys, ids, tile_ranges, ws, ws_bytes, stream):
    """Returns (status, n_instances); CAPACITY is returned, not raised."""
    cnt = ctypes.c_int64(0)
    sz = ctypes.c_size_t(ws_bytes)
    st = lib().gs_bin_sort(ctypes.byref(proj), n, n_views, width, height, capacity, keys, ids, tile_ranges,
                           ctypes.byref(cnt), ws, ctypes.byref(sz), stream)
    if st not in (GS_OK, GS_ERR_CAPACITY):
        _check("gs_bin_sort", st)
    return st, cnt.value


def raster_bits_ws_words(n_instances, n_lists) -> int:
    """GS_RASTER_BITS_WS_WORDS: scratch words that cover n_instances entries in n_lists tile lists."""
    return (int(n_instances) + 32 * int(n_lists)) * 8


def gs_raster_fused_fwd_bwd(proj, n, tile_ranges, ids, cams, n_views, opts, target, image, loss, grad2d, touched,
                            eval_counts, stream, bits_ws=None, bits_ws_words=0):
    """bits_ws: None or a device pointer to bits_ws_words u32 of saved-pass-bits scratch."""
    _check("gs_raster_fused_fwd_bwd",
           lib().gs_raster_fused_fwd_bwd(ctypes.byref(proj), n, tile_ranges, ids, cams, n_views, ctypes.byref(opts),
                                         target, image, loss, grad2d, touched, eval_counts, bits_ws,
                                         int(bits_ws_words), stream))


GS_RASTER_WORK_COUNTERS = 10
RASTER_WORK_NAMES = ("pairs", "pair_exps", "composite_walks", "sparse_entries", "sparse_steps", "dense_entries",
                     "dense_steps", "chunks", "restaged_chunks", "recomputed_chunks")


def gs_raster_work_counts(proj, n, tile_ranges, ids, cams, n_views, opts, target, image, loss, grad2d, touched, work,
                          stream, bits_ws=None, bits_ws_words=0):
    _check("gs_raster_work_counts",
           lib().gs_raster_work_counts(ctypes.byref(proj), n, tile_ranges, ids, cams, n_views, ctypes.byref(opts),
                                       target, image, loss, grad2d, touched, work, bits_ws, int(bits_ws_words),
                                       stream))


CHECK_SITES = ("none", "bin_rect", "bin_slot", "sort_slot", "sort_id", "range", "raster_id", "prune_id",
               "compact_id", "adam_id")


def gs_check_report() -> dict:
    """Bounds-check report since the previous one (then reset): {"checked": bool,
    "failures": count, "site": name, "index": i, "bound": n}.  A DEVICE status
    (failed checks) is returned in the dict, not raised."""
    rep = (ctypes.c_uint64 * 4)()
    checked = ctypes.c_int32(0)
    st = lib().gs_check_report(rep, ctypes.byref(checked))
    if st not in (GS_OK, GS_ERR_DEVICE):
        _check("gs_check_report", st)
    idx = rep[2] - (1 << 64) if rep[2] >= (1 << 63) else rep[2]
    site = CHECK_SITES[rep[1]] if rep[1] < len(CHECK_SITES) else str(rep[1])
    return {"checked": bool(checked.value), "failures": int(rep[0]), "site": site, "index": int(idx),
            "bound": int(rep[3])}


def gs_prune_tiles(proj, n, n_views, width, height, budget, ids, tile_ranges, stream):
    _check("gs_prune_tiles", lib().gs_prune_tiles(ctypes.byref(proj), n, n_views, width, height, budget, ids,
                                                  tile_ranges, stream))


def gs_split_ranges(keys, tile_ranges, n_views, width, height, n_subsets, depth_splits, sub_ranges, stream):
    """depth_splits: host sequence [V][S-1] (converted to fp32)."""
    flat = [float(z) for row in depth_splits for z in row] if n_subsets > 1 else []
    arr = (ctypes.c_float * max(1, len(flat)))(*flat)
    _check("gs_split_ranges", lib().gs_split_ranges(keys, tile_ranges, n_views, width, height, n_subsets,
                                                    arr if flat else None, sub_ranges, stream))


def gs_compose(c_parts, t_parts, n_subsets, n_views, width, height, bg, image, t_final, stream):
    bga = (ctypes.c_float * 3)(*[float(b) for b in bg])
    _check("gs_compose", lib().gs_compose(c_parts, t_parts, n_subsets, n_views, width, height, bga, image, t_final,
                                          stream))


def gs_raster_forward_state(proj, n, tile_ranges, ids, cams, n_views, opts, image, t_final, last_idx, bits_ws,
                            bits_ws_words, eval_counts, stream):
    """bits_ws: None or a device pointer to bits_ws_words u32 (every chunk's pass bits are stored there)."""
    _check("gs_raster_forward_state",
           lib().gs_raster_forward_state(ctypes.byref(proj), n, tile_ranges, ids, cams, n_views, ctypes.byref(opts),
                                         image, t_final, last_idx, bits_ws, int(bits_ws_words), eval_counts, stream))


def gs_dssim_loss_grad(image, target, n_views, width, height, lam, loss, dldc, stream):
    _check("gs_dssim_loss_grad", lib().gs_dssim_loss_grad(image, target, n_views, width, height, lam, loss, dldc,
                                                          stream))


def gs_raster_backward_state(proj, n, tile_ranges, ids, cams, n_views, opts, t_final, last_idx, bits_ws,
                             bits_ws_words, dldc, grad2d, touched, stream):
    _check("gs_raster_backward_state",
           lib().gs_raster_backward_state(ctypes.byref(proj), n, tile_ranges, ids, cams, n_views, ctypes.byref(opts),
                                          t_final, last_idx, bits_ws, int(bits_ws_words), dldc, grad2d, touched,
                                          stream))


def gs_grad_compact_ws_bytes(n) -> int:
    sz = ctypes.c_size_t(0)
    _check("gs_grad_compact", lib().gs_grad_compact(None, None, None, n, 0, None, 1, None, None, None, None, None,
                                                    ctypes.byref(sz), None))
    return sz.value


def gs_grad_compact(grad2d, touched, params, n, sh_degree, cams, n_views, opts, idx, n_idx, grads, ws, ws_bytes,
                    stream):
    sz = ctypes.c_size_t(ws_bytes)
    _check("gs_grad_compact", lib().gs_grad_compact(grad2d, touched, params, n, sh_degree, cams, n_views,
                                                    ctypes.byref(opts), idx, n_idx, grads, ws, ctypes.byref(sz),
                                                    stream))


def gs_adam_deferred(params, grads, m, v, last_step, n, sh_degree, idx, n_idx, t, lr, beta1, beta2, eps, flush,
                     stream):
    lr_arr = (ctypes.c_float * 5)(*[float(x) for x in lr])
    _check("gs_adam_deferred", lib().gs_adam_deferred(params, grads, m, v, last_step, n, sh_degree, idx, n_idx, t,
                                                      lr_arr, beta1, beta2, eps, 1 if flush else 0, stream))


def gs_param_rows(sh_degree) -> int:
    return lib().gs_param_rows(sh_degree)


def gs_param_stride(sh_degree) -> int:
    return lib().gs_param_stride(sh_degree)


def gs_num_tiles(width, height) -> int:
    return lib().gs_num_tiles(width, height)


def gs_version() -> str:
    return lib().gs_version().decode()


def gs_grad_compact_static(grad2d, touched, params, n, sh_degree, cams, n_views, opts, idx, n_idx, grads, stream):
    """gs_grad_compact for callers that cannot allocate device memory: its scratch is a
    fixed array inside the library (at most GS_COMPACT_STATIC_MAX_N Gaussians)."""
    L = lib()
    f = L.gs_grad_compact_static
    if f.argtypes is None:
        f.argtypes = [_P, _P, _P, _I64, _I32, _P, _I32, _P, _P, _P, _P, _P]
        f.restype = ctypes.c_int
    _check("gs_grad_compact_static", f(grad2d, touched, params, n, sh_degree, cams, n_views, ctypes.byref(opts), idx,
                                       n_idx, grads, stream))
