"""Host-side checks of the C-ABI library (no GPU needed): it builds, loads, exports
every entry point that include/gs.h declares, answers workspace queries, and
rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from differentiable_rasterizer_gb300 import build, abi
    build.build()
    return abi.lib()


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "gs.h")).read()
    return sorted(set(re.findall(r"GS_API\s+[\w\s\*]*?\b(gs_\w+)\s*\(", text)))


def test_header_declares_the_five_calls():
    syms = _declared_symbols()
    for name in ("gs_project", "gs_bin_sort", "gs_raster_fused_fwd_bwd", "gs_grad_compact", "gs_adam_deferred"):
        assert name in syms


def test_library_exports_every_declared_symbol(L):
    for name in _declared_symbols():
        assert hasattr(L, name), name


def test_static_helpers(L):
    from differentiable_rasterizer_gb300 import abi
    assert abi.gs_param_rows(0) == 14 and abi.gs_param_rows(3) == 59 and abi.gs_param_rows(2) == -1
    assert abi.gs_param_stride(0) == 16 and abi.gs_param_stride(3) == 64 and abi.gs_param_stride(1) == -1
    assert abi.gs_num_tiles(1920, 1080) == 120 * 68
    assert abi.gs_num_tiles(64, 64) == 16
    assert "sm_103a" in abi.gs_version()
    assert L.gs_error_string(2) == b"instance capacity too small"


def test_workspace_queries(L):
    from differentiable_rasterizer_gb300 import abi
    a = abi.gs_bin_sort_ws_bytes(1000, 1, 64, 64, 4000)
    b = abi.gs_bin_sort_ws_bytes(1000, 1, 64, 64, 400000)
    assert 0 < a < b and a % 256 == 0
    assert abi.gs_grad_compact_ws_bytes(10 ** 6) >= 10 ** 6   # union flags
    assert abi.gs_grad_compact_ws_bytes(0) >= 0


def test_invalid_arguments_are_rejected_on_the_host(L):
    from differentiable_rasterizer_gb300 import abi, scenes
    sc = scenes.make_scene("tiny")
    cams = abi.cameras(sc.cameras)
    opts = abi.render_opts(sc.opts)
    proj = abi.GsProj(16, 16, 16, 16)
    # NULL params / bad degree / bad view count
    assert L.gs_project(None, 10, 0, cams, 1, ctypes.byref(opts), ctypes.byref(proj), None) == abi.GS_ERR_INVALID_ARG
    assert L.gs_project(16, 10, 2, cams, 1, ctypes.byref(opts), ctypes.byref(proj), None) == abi.GS_ERR_INVALID_ARG
    assert L.gs_project(16, 10, 0, cams, 0, ctypes.byref(opts), ctypes.byref(proj), None) == abi.GS_ERR_INVALID_ARG
    assert L.gs_project(16, 10, 0, cams, 33, ctypes.byref(opts), ctypes.byref(proj), None) == abi.GS_ERR_INVALID_ARG
    # mixed resolutions
    two = abi.cameras([sc.cameras[0], scenes.Camera(sc.cameras[0].R, sc.cameras[0].t, 64, 64, 32, 32, 64, 32)])
    assert L.gs_project(16, 10, 0, two, 2, ctypes.byref(opts), ctypes.byref(proj), None) == abi.GS_ERR_INVALID_ARG
    # misaligned record buffer
    bad = abi.GsProj(20, 16, 16, 16)
    assert L.gs_project(16, 10, 0, cams, 1, ctypes.byref(opts), ctypes.byref(bad), None) == abi.GS_ERR_INVALID_ARG
    # workspace too small
    cnt = ctypes.c_int64(0)
    sz = ctypes.c_size_t(8)
    assert L.gs_bin_sort(ctypes.byref(proj), 10, 1, 64, 64, 100, 16, 16, 16, ctypes.byref(cnt), 16,
                         ctypes.byref(sz), None) == abi.GS_ERR_INVALID_ARG
    # Adam: t must be >= 1
    lr = (ctypes.c_float * 5)(1, 1, 1, 1, 1)
    assert L.gs_adam_deferred(16, 16, 16, 16, 16, 10, 0, 16, 16, 0, lr, ctypes.c_float(0.9), ctypes.c_float(0.999),
                              ctypes.c_float(1e-8), 0, None) == abi.GS_ERR_INVALID_ARG
    # Adam: learning rates >= 0 and finite, 0 <= beta < 1, eps > 0
    for bad_lr, b1, b2, e in (((1, 1, -1e-3, 1, 1), 0.9, 0.999, 1e-8), ((1, 1, 1, float("inf"), 1), 0.9, 0.999, 1e-8),
                              ((1, 1, 1, 1, 1), 1.0, 0.999, 1e-8), ((1, 1, 1, 1, 1), 0.9, 0.999, 0.0)):
        lrb = (ctypes.c_float * 5)(*bad_lr)
        assert L.gs_adam_deferred(16, 16, 16, 16, 16, 10, 0, 16, 16, 1, lrb, ctypes.c_float(b1), ctypes.c_float(b2),
                                  ctypes.c_float(e), 0, None) == abi.GS_ERR_INVALID_ARG
    # raster with a target but no gradient buffers
    assert L.gs_raster_fused_fwd_bwd(ctypes.byref(proj), 10, 16, 16, cams, 1, ctypes.byref(opts), 16, 16, None, None,
                                     None, None, None, 0, None) == abi.GS_ERR_INVALID_ARG
    # saved-bits scratch: a pointer needs a positive size, a size is never negative
    for ws, words in ((16, 0), (None, -1), (16, -8)):
        assert L.gs_raster_fused_fwd_bwd(ctypes.byref(proj), 10, 16, 16, cams, 1, ctypes.byref(opts), None, 16, None,
                                         None, None, None, ws, words, None) == abi.GS_ERR_INVALID_ARG
    # forward with state: state buffers required; backward from state: dL/dC and gradient buffers required
    assert L.gs_raster_forward_state(ctypes.byref(proj), 10, 16, 16, cams, 1, ctypes.byref(opts), 16, None, 16, None,
                                     0, None, None) == abi.GS_ERR_INVALID_ARG
    for ws, words in ((16, 0), (None, -1)):   # the scratch: a pointer needs a size, no size is negative
        assert L.gs_raster_forward_state(ctypes.byref(proj), 10, 16, 16, cams, 1, ctypes.byref(opts), 16, 16, 16,
                                         ws, words, None, None) == abi.GS_ERR_INVALID_ARG
        assert L.gs_raster_backward_state(ctypes.byref(proj), 10, 16, 16, cams, 1, ctypes.byref(opts), 16, 16, ws,
                                          words, 16, 16, 16, None) == abi.GS_ERR_INVALID_ARG
    assert L.gs_raster_backward_state(ctypes.byref(proj), 10, 16, 16, cams, 1, ctypes.byref(opts), 16, 16, None,
                                      0, None, 16, 16, None) == abi.GS_ERR_INVALID_ARG
    assert L.gs_raster_backward_state(ctypes.byref(proj), 10, 16, 16, cams, 1, ctypes.byref(opts), 16, 16, None,
                                      0, 16, None, 16, None) == abi.GS_ERR_INVALID_ARG
    # pruning: budget >= 1
    assert L.gs_prune_tiles(ctypes.byref(proj), 10, 1, 64, 64, 0, 16, 16, None) == abi.GS_ERR_INVALID_ARG
    assert L.gs_prune_tiles(ctypes.byref(proj), 10, 1, 64, 64, 8, 16, None, None) == abi.GS_ERR_INVALID_ARG
    # partial render + compose: 1..8 slabs, positive ascending splits
    two = (ctypes.c_float * 2)(2.0, 1.0)
    assert L.gs_split_ranges(16, 16, 1, 64, 64, 3, two, 16, None) == abi.GS_ERR_INVALID_ARG
    neg = (ctypes.c_float * 1)(-1.0)
    assert L.gs_split_ranges(16, 16, 1, 64, 64, 2, neg, 16, None) == abi.GS_ERR_INVALID_ARG
    assert L.gs_split_ranges(16, 16, 1, 64, 64, 9, None, 16, None) == abi.GS_ERR_INVALID_ARG
    bg = (ctypes.c_float * 3)(0, 0, 0)
    assert L.gs_compose(16, 16, 0, 1, 64, 64, bg, 16, None, None) == abi.GS_ERR_INVALID_ARG
    assert L.gs_compose(16, 16, 2, 1, 64, 64, None, 16, None, None) == abi.GS_ERR_INVALID_ARG
    # D-SSIM: 0 <= lambda <= 1, at least one pixel and one view
    for lam, V, W, H in ((-0.1, 1, 8, 8), (1.5, 1, 8, 8), (float("nan"), 1, 8, 8), (0.2, 0, 8, 8), (0.2, 1, 0, 8),
                         (0.2, 33, 8, 8)):
        assert L.gs_dssim_loss_grad(16, 16, V, W, H, ctypes.c_float(lam), 16, 16, None) == abi.GS_ERR_INVALID_ARG
    assert L.gs_dssim_loss_grad(16, None, 1, 8, 8, ctypes.c_float(0.2), 16, 16, None) == abi.GS_ERR_INVALID_ARG


def test_binding_raises_without_the_library(tmp_path, monkeypatch):
    from differentiable_rasterizer_gb300 import abi
    monkeypatch.setattr(abi, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(abi, "_lib", None)
    with pytest.raises(RuntimeError, match="CUDA library missing"):
        abi.lib()


def test_every_entry_point_opens_an_nvtx_range_named_after_it():
    """Each C-ABI call that does device work starts with GS_NVTX_RANGE("<its name>"),
    so a profiler groups the kernels it launches under the call."""
    import glob
    csrc = os.path.join(ROOT, "differentiable_rasterizer_gb300", "csrc")
    seen = set()
    for path in glob.glob(os.path.join(csrc, "*.cu")):
        text = open(path).read()
        for m in re.finditer(r'extern "C" gs_status (gs_\w+)\(', text):
            body = text[text.index("\n{\n", m.end()) + 3:]
            first = body.lstrip().split("\n", 1)[0].strip()
            assert first == f'GS_NVTX_RANGE("{m.group(1)}");', (m.group(1), first)
            seen.add(m.group(1))
    declared = {s for s in _declared_symbols()}
    status_calls = {s for s in declared if s not in ("gs_error_string", "gs_param_rows", "gs_param_stride",
                                                     "gs_num_tiles", "gs_version")}
    assert status_calls <= seen, status_calls - seen


def test_checked_library_exports_every_declared_symbol(L):
    from differentiable_rasterizer_gb300 import build
    C = ctypes.CDLL(build.CHECKED_LIB)
    for name in _declared_symbols():
        assert hasattr(C, name), name


def test_check_report_on_the_host(L):
    """The plain build reports itself unchecked with a zero report and does no
    device work; both builds reject NULL outputs before touching the device."""
    from differentiable_rasterizer_gb300 import abi, build
    rep = (ctypes.c_uint64 * 4)(1, 2, 3, 4)
    chk = ctypes.c_int32(7)
    assert L.gs_check_report(rep, ctypes.byref(chk)) == abi.GS_OK
    assert chk.value == 0 and list(rep) == [0, 0, 0, 0]
    C = ctypes.CDLL(build.CHECKED_LIB)
    for lib in (L, C):
        assert lib.gs_check_report(None, ctypes.byref(chk)) == abi.GS_ERR_INVALID_ARG
        assert lib.gs_check_report(rep, None) == abi.GS_ERR_INVALID_ARG


def test_check_sites_agree_between_header_binding_and_kernels():
    """The binding's site names follow gs.h's gs_check_site enum in order, and every
    declared site is tested somewhere in the kernels and only declared sites are."""
    import glob
    from differentiable_rasterizer_gb300 import abi
    text = open(os.path.join(ROOT, "include", "gs.h")).read()
    body = text[text.index("typedef enum gs_check_site"):]
    body = body[:body.index("} gs_check_site;")]
    decl = re.findall(r"GS_CHECK_(\w+)\s*=\s*(\d+)", body)
    assert [int(v) for _, v in decl] == list(range(len(decl)))
    assert tuple(name.lower() for name, _ in decl) == abi.CHECK_SITES
    used = set()
    for path in glob.glob(os.path.join(ROOT, "differentiable_rasterizer_gb300", "csrc", "*.cu")):
        used |= set(re.findall(r"GS_IN_RANGE\([^;]*?GS_CHECK_(\w+)\)", open(path).read(), re.S))
    assert used == {name for name, _ in decl if name != "NONE"}, used
