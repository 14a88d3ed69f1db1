"""The C ABI without a GPU: the library builds and loads, exports every
function include/gs2d.h declares, sizes workspaces, and rejects bad
arguments on the host before touching CUDA (these calls never reach the
device, so they run on a machine without one)."""
import ctypes as C
import os
import re

import pytest

from raster_gaussian_02_b300 import build as lib_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gs2d.h")


@pytest.fixture(scope="module")
def gs2d():
    lib_build.build()
    from raster_gaussian_02_b300 import gs2d as g
    g.lib()
    return g


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"GS2D_API\s+[\w\s\*]+?\b(gs2d_\w+)\s*\(", text)


def test_header_declares_the_five_calls():
    names = declared_functions()
    for n in ("gs2d_project", "gs2d_bin_and_sort", "gs2d_render_fwd", "gs2d_render_bwd",
              "gs2d_loss_l2"):
        assert n in names


def test_library_exports_every_declared_symbol(gs2d):
    lib = C.CDLL(gs2d.LIB_PATH)
    names = declared_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), n


def test_nm_shows_only_the_abi(gs2d):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", gs2d.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    gs = {e for e in exported if e.startswith("gs2d_")}
    assert gs == set(declared_functions())


def test_checked_build_exports_the_same_abi(gs2d):
    """libgs2d_checked.so (GS2D_CHECKS) builds and exports exactly the
    declared functions; the normal build answers the check-word call with
    GS2D_ERR_UNSUPPORTED without touching CUDA."""
    import subprocess
    path = lib_build.build(checked=True)
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True,
                         check=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l and " gs2d_" in l}
    assert exported == set(declared_functions())
    st, word = gs2d.gs2d_debug_check_word()
    assert (st, word) == (gs2d.GS2D_ERR_UNSUPPORTED, 0)
    assert gs2d.lib().gs2d_debug_check_word(None, 0) == gs2d.GS2D_ERR_INVALID_ARG


def test_status_strings(gs2d):
    for s in range(7):
        assert gs2d.status_string(s) != "unknown status"
    assert gs2d.status_string(99) == "unknown status"


def test_workspace_size(gs2d):
    cfg = gs2d.make_config(768, 512)
    a = gs2d.gs2d_workspace_size(cfg, 50_000, 200_000)
    b = gs2d.gs2d_workspace_size(cfg, 50_000, 400_000)
    assert 0 < a < b
    assert gs2d.gs2d_workspace_size(cfg, 0, 0) >= 16384
    comp = gs2d.make_config(768, 512, gs2d.GS2D_MODE_COMPOSITE)
    # per pair, composite needs more (64-bit keys, 12-float partials)
    ca, cb = (gs2d.gs2d_workspace_size(comp, 50_000, k) for k in (200_000, 400_000))
    assert cb - ca > b - a
    bad = [gs2d.gs2d_config(0, 512, 16, 0, 3.0, 1e-4), gs2d.gs2d_config(768, 512, 8, 0, 3.0, 1e-4),
           gs2d.gs2d_config(768, 512, 16, 2, 3.0, 1e-4), gs2d.gs2d_config(768, 512, 16, 0, 0.0, 1e-4),
           gs2d.gs2d_config(768, 512, 16, 0, float("nan"), 1e-4),
           gs2d.gs2d_config(40000, 512, 16, 0, 3.0, 1e-4),
           gs2d.gs2d_config(768, 512, 16, 1, 3.0, 2.0),
           gs2d.gs2d_config(768, 512, 16, 0, 3.0, 1e-4, 2),
           gs2d.gs2d_config(768, 512, 16, 0, 3.0, 1e-4, 0, -1.0),
           gs2d.gs2d_config(768, 512, 16, 0, 3.0, 1e-4, 0, float("inf"))]
    for c in bad:
        assert gs2d.gs2d_workspace_size(c, 10, 10) == 0
    assert gs2d.gs2d_workspace_size(cfg, -1, 10) == 0
    sr = gs2d.make_config(768, 512, param=gs2d.GS2D_PARAM_SCALE_ROT)
    assert gs2d.gs2d_workspace_size(sr, 50_000, 200_000) == a
    assert gs2d.gs2d_workspace_size(cfg, 10, 1 << 30) == 0


def test_host_checks_reject_bad_arguments(gs2d):
    """Every one of these returns GS2D_ERR_INVALID_ARG on the host."""
    L = gs2d.lib()
    INVALID = gs2d.GS2D_ERR_INVALID_ARG
    good = gs2d.make_config(64, 64)
    bad = gs2d.gs2d_config(64, 64, 8, 0, 3.0, 1e-4)
    fake = C.c_void_p(0x10000)       # 16-byte aligned, never dereferenced
    odd = C.c_void_p(0x10004)        # 4-byte aligned only
    null = None
    # project
    assert L.gs2d_project(C.byref(bad), 4, fake, fake, fake, null, null, fake, fake, fake, null) == INVALID
    assert L.gs2d_project(C.byref(good), -1, fake, fake, fake, null, null, fake, fake, fake, null) == INVALID
    assert L.gs2d_project(C.byref(good), 4, null, fake, fake, null, null, fake, fake, fake, null) == INVALID
    assert L.gs2d_project(C.byref(good), 4, fake, fake, fake, null, null, odd, fake, fake, null) == INVALID
    assert L.gs2d_project(C.byref(good), 4, fake, fake, fake, null, null, fake, odd, fake, null) == INVALID
    comp = gs2d.make_config(64, 64, gs2d.GS2D_MODE_COMPOSITE)
    assert L.gs2d_project(C.byref(comp), 4, fake, fake, fake, null, fake, fake, fake, fake, null) == INVALID
    assert L.gs2d_project(None, 4, fake, fake, fake, null, null, fake, fake, fake, null) == INVALID
    # n == 0 is a no-op that succeeds without touching anything
    assert L.gs2d_project(C.byref(good), 0, null, null, null, null, null, null, null, null, null) == 0
    # bin_and_sort
    assert L.gs2d_bin_and_sort(C.byref(good), 4, fake, fake, fake, 10, None, fake, fake, null, null) == INVALID
    assert L.gs2d_bin_and_sort(C.byref(good), 4, fake, fake, fake, -1, None, fake, fake, fake, null) == INVALID
    assert L.gs2d_bin_and_sort(C.byref(good), 4, fake, fake, fake, 1 << 30, None, fake, fake, fake, null) == INVALID
    assert L.gs2d_bin_and_sort(C.byref(good), 4, fake, fake, fake, 10, None, odd, fake, fake, null) == INVALID
    assert L.gs2d_bin_and_sort(C.byref(good), 4, fake, fake, fake, 10, None, fake, null, fake, null) == INVALID
    assert L.gs2d_bin_and_sort(C.byref(good), 4, null, fake, fake, 10, None, fake, fake, fake, null) == INVALID
    # project_bin_and_sort: (xy shape rgb depth opacity rec rect count) cap pairs_out (ranges gid ws)
    pb = L.gs2d_project_bin_and_sort
    assert pb(C.byref(bad), 4, fake, fake, fake, null, null, fake, fake, fake, 10, None, fake, fake, fake, null) == INVALID
    assert pb(C.byref(good), 4, null, fake, fake, null, null, fake, fake, fake, 10, None, fake, fake, fake, null) == INVALID
    assert pb(C.byref(good), 4, fake, fake, fake, null, null, odd, fake, fake, 10, None, fake, fake, fake, null) == INVALID
    assert pb(C.byref(comp), 4, fake, fake, fake, null, fake, fake, fake, fake, 10, None, fake, fake, fake, null) == INVALID
    assert pb(C.byref(good), 4, fake, fake, fake, null, null, fake, fake, fake, -1, None, fake, fake, fake, null) == INVALID
    assert pb(C.byref(good), 4, fake, fake, fake, null, null, fake, fake, fake, 10, None, fake, fake, odd, null) == INVALID
    assert pb(C.byref(good), 4, fake, fake, fake, null, null, fake, fake, fake, 10, None, fake, null, fake, null) == INVALID
    # render_fwd: (rec ranges gid bg image t_final last workspace)
    assert L.gs2d_render_fwd(C.byref(good), 4, fake, fake, fake, null, null, null, null, null, null) == INVALID
    assert L.gs2d_render_fwd(C.byref(good), 4, odd, fake, fake, null, fake, null, null, null, null) == INVALID
    assert L.gs2d_render_fwd(C.byref(bad), 4, fake, fake, fake, null, fake, null, null, null, null) == INVALID
    assert L.gs2d_render_fwd(C.byref(good), 4, fake, fake, fake, null, fake, null, null, odd, null) == INVALID
    # loss
    assert L.gs2d_loss_l2(0, 64, fake, fake, fake, fake, fake, null) == INVALID
    assert L.gs2d_loss_l2(64, 64, fake, null, fake, fake, fake, null) == INVALID
    assert L.gs2d_loss_l2(64, 64, fake, fake, fake, fake, null, null) == INVALID
    assert L.gs2d_loss_l2(64, 64, fake, fake, fake, fake, odd, null) == INVALID
    # render_bwd: composite needs t_final and last
    args = [fake] * 16
    args[6] = null  # t_final
    assert L.gs2d_render_bwd(C.byref(comp), 4, *args, null) == INVALID
    args = [fake] * 16
    args[0] = null  # shape
    assert L.gs2d_render_bwd(C.byref(good), 4, *args, null) == INVALID
    args = [fake] * 16
    args[14] = C.c_void_p(0x10002)  # d_xy_abs misaligned
    assert L.gs2d_render_bwd(C.byref(good), 4, *args, null) == INVALID
    # fused fwd + L2 + bwd: target, loss and workspace are required
    # (shape rec rect ranges gid bg target image loss dxy dshape drgb dop dbg dabs ws)
    args = [fake] * 16
    args[6] = null  # target
    assert L.gs2d_render_fwd_bwd_l2(C.byref(good), 4, *args, null) == INVALID
    args = [fake] * 16
    args[8] = null  # loss
    assert L.gs2d_render_fwd_bwd_l2(C.byref(good), 4, *args, null) == INVALID
    args = [fake] * 16
    args[15] = odd  # workspace
    assert L.gs2d_render_fwd_bwd_l2(C.byref(good), 4, *args, null) == INVALID
    args = [fake] * 16
    args[3] = odd  # tile_ranges
    assert L.gs2d_render_fwd_bwd_l2(C.byref(good), 4, *args, null) == INVALID
    assert L.gs2d_render_fwd_bwd_l2(C.byref(bad), 4, *([fake] * 16), null) == INVALID
    # merge: sum mode only, max_merges >= 0, a 256-byte aligned workspace
    margs = [fake] * 7
    assert L.gs2d_merge(C.byref(comp), 4, *margs, 1, fake, fake, fake, None, fake, null) == INVALID
    assert L.gs2d_merge(C.byref(good), 4, *margs, -1, fake, fake, fake, None, fake, null) == INVALID
    assert L.gs2d_merge(C.byref(good), 4, *margs, 1, fake, fake, fake, None, C.c_void_p(0x10010),
                        null) == INVALID
    assert L.gs2d_merge(C.byref(good), 4, *margs, 1, null, fake, fake, None, fake, null) == INVALID
    assert gs2d.gs2d_merge_workspace_size(-1) == 0
    assert gs2d.gs2d_merge_workspace_size(1000) > gs2d.gs2d_merge_workspace_size(10) > 0
    # adam: step >= 1, lr >= 0 and finite, betas in [0, 1), eps > 0, width 1..16, arrays non-NULL
    ok = gs2d.gs2d_adam(0.01, 0.9, 0.999, 1e-8, 1)
    for o in (gs2d.gs2d_adam(0.01, 0.9, 0.999, 1e-8, 0), gs2d.gs2d_adam(-1.0, 0.9, 0.999, 1e-8, 1),
              gs2d.gs2d_adam(float("nan"), 0.9, 0.999, 1e-8, 1), gs2d.gs2d_adam(0.01, 1.0, 0.999, 1e-8, 1),
              gs2d.gs2d_adam(0.01, 0.9, -0.5, 1e-8, 1), gs2d.gs2d_adam(0.01, 0.9, 0.999, 0.0, 1)):
        assert L.gs2d_adam_step(C.byref(o), 4, 2, fake, fake, fake, fake, null, null) == INVALID
    assert L.gs2d_adam_step(None, 4, 2, fake, fake, fake, fake, null, null) == INVALID
    assert L.gs2d_adam_step(C.byref(ok), 0, 2, fake, fake, fake, fake, null, null) == gs2d.GS2D_OK  # nothing to do
    assert L.gs2d_adam_step(C.byref(ok), -1, 2, fake, fake, fake, fake, null, null) == INVALID
    assert L.gs2d_adam_step(C.byref(ok), 4, 0, fake, fake, fake, fake, null, null) == INVALID
    assert L.gs2d_adam_step(C.byref(ok), 4, 17, fake, fake, fake, fake, null, null) == INVALID
    assert L.gs2d_adam_step(C.byref(ok), 4, 2, fake, null, fake, fake, null, null) == INVALID
    assert L.gs2d_adam_step(C.byref(ok), 4, 2, fake, fake, fake, C.c_void_p(0x10002), null, null) == INVALID
    # read_status
    assert L.gs2d_read_status(None, None, None, None) == INVALID
    assert L.gs2d_read_status(odd, None, None, None) == INVALID


def test_probe_library_builds_and_checks_arguments():
    """libgs2d_probe.so (the FP32 / SFU throughput probes behind the
    roofline's peaks) exports exactly what include/gs2d_probe.h declares and
    rejects bad arguments on the host (status 1, nothing launched)."""
    import subprocess
    path = lib_build.build_probe()
    text = open(os.path.join(ROOT, "include", "gs2d_probe.h")).read()
    declared = set(re.findall(r"GS2D_PROBE_API\s+[\w\s\*]+?\b(gs2d_\w+)\s*\(", text))
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True,
                         check=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l and " gs2d_" in l}
    assert exported == declared == {"gs2d_probe_fp32_fma", "gs2d_probe_ex2"}
    L = C.CDLL(path)
    L.gs2d_probe_fp32_fma.argtypes = [C.c_void_p, C.c_int32, C.c_int32, C.c_float, C.c_float, C.c_void_p]
    L.gs2d_probe_ex2.argtypes = [C.c_void_p, C.c_int32, C.c_int32, C.c_void_p]
    fake = C.c_void_p(0x10000)
    assert L.gs2d_probe_fp32_fma(None, 8, 16, 1.0, 0.0, None) == 1
    assert L.gs2d_probe_fp32_fma(fake, 0, 16, 1.0, 0.0, None) == 1
    assert L.gs2d_probe_fp32_fma(fake, 8, 0, 1.0, 0.0, None) == 1
    assert L.gs2d_probe_ex2(fake, 70000, 16, None) == 1
    assert L.gs2d_probe_ex2(fake, 8, (1 << 20) + 1, None) == 1


def test_trace_rejects_bad_arguments_on_the_host(gs2d):
    """gs2d_trace_begin checks its arguments before anything else; with no
    trace active gs2d_trace_end returns 0 and no kernel has a name.  None of
    this reaches CUDA."""
    L = gs2d.lib()
    assert L.gs2d_trace_begin(None, 1) == gs2d.GS2D_ERR_INVALID_ARG
    fake = (C.c_void_p * 4)(1, 2, 3, 4)  # never dereferenced: rejected first
    assert L.gs2d_trace_begin(fake, 0) == gs2d.GS2D_ERR_INVALID_ARG
    assert L.gs2d_trace_begin(fake, 4097) == gs2d.GS2D_ERR_INVALID_ARG
    holes = (C.c_void_p * 4)(1, None, 3, 4)
    assert L.gs2d_trace_begin(holes, 2) == gs2d.GS2D_ERR_INVALID_ARG
    assert gs2d.gs2d_trace_end() == 0
    assert gs2d.gs2d_trace_kernel_name(0) is None
    assert gs2d.gs2d_trace_kernel_name(-1) is None
