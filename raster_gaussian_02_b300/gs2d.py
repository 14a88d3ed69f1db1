"""Python binding of the gs2d C ABI (include/gs2d.h).

Argument marshalling only: each function below has the C entry point's name,
checks that the torch tensors it is given are CUDA, contiguous and of the
right dtype, and passes their device pointers and the current CUDA stream to
libgs2d.so.  Every step of the rasterizer runs in the library's kernels;
there is no fallback.  If the library is missing the first call raises.

`Rasterizer` strings the calls together for a fixed configuration, owning
the torch buffers they need.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# GS2D_CHECKED=1 loads the bounds-checked build instead (same ABI; see
# gs2d_debug_check_word), for debugging and the checked-build tests.
CHECKED = os.environ.get("GS2D_CHECKED", "0") == "1"
LIB_PATH = os.path.join(_HERE, "libgs2d_checked.so" if CHECKED else "libgs2d.so")

(GS2D_OK, GS2D_ERR_INVALID_ARG, GS2D_ERR_CAPACITY, GS2D_ERR_CUDA, GS2D_ERR_TIMEOUT, GS2D_ERR_OVERFLOW,
 GS2D_ERR_UNSUPPORTED) = range(7)
GS2D_MODE_SUM, GS2D_MODE_COMPOSITE = 0, 1
GS2D_PARAM_CHOLESKY, GS2D_PARAM_SCALE_ROT = 0, 1
GS2D_FLAG_CAPACITY, GS2D_FLAG_OVERFLOW, GS2D_FLAG_TIMEOUT = 1, 2, 4
RECORD_BYTES = 48
TILE = 16


class gs2d_config(C.Structure):
    _fields_ = [("width", C.c_int32), ("height", C.c_int32), ("tile", C.c_int32),
                ("mode", C.c_int32), ("cutoff_sigma", C.c_float), ("t_min", C.c_float),
                ("param", C.c_int32), ("scale", C.c_float)]


def make_config(width: int, height: int, mode: int = GS2D_MODE_SUM, cutoff_sigma: float = 3.0,
                t_min: float = 1e-4, param: int = GS2D_PARAM_CHOLESKY,
                scale: float = 1.0) -> gs2d_config:
    """scale: output pixels per unit of xy and shape (render at any resolution)."""
    return gs2d_config(int(width), int(height), TILE, int(mode), float(cutoff_sigma), float(t_min),
                       int(param), float(scale))


class gs2d_adam(C.Structure):
    _fields_ = [("lr", C.c_float), ("beta1", C.c_float), ("beta2", C.c_float), ("eps", C.c_float),
                ("step", C.c_int32)]


class Gs2dError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_string(status)} (status {status})")
        self.status = status


_lib = None
_p = C.c_void_p
_cfgp = C.POINTER(gs2d_config)


def lib() -> C.CDLL:
    """The loaded libgs2d.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"gs2d CUDA library not built: {LIB_PATH} is missing "
                               "(run raster_gaussian_02_b300/build.py"
                               + (" --checked)" if CHECKED else ")"))
        L = C.CDLL(LIB_PATH)
        L.gs2d_workspace_size.argtypes = [_cfgp, C.c_int32, C.c_int64]
        L.gs2d_workspace_size.restype = C.c_size_t
        L.gs2d_project.argtypes = [_cfgp, C.c_int32] + [_p] * 8 + [_p]
        L.gs2d_project.restype = C.c_int
        L.gs2d_bin_and_sort.argtypes = [_cfgp, C.c_int32, _p, _p, _p, C.c_int64,
                                        C.POINTER(C.c_int64), _p, _p, _p, _p]
        L.gs2d_bin_and_sort.restype = C.c_int
        L.gs2d_project_bin_and_sort.argtypes = ([_cfgp, C.c_int32] + [_p] * 8 +
                                                [C.c_int64, C.POINTER(C.c_int64)] + [_p] * 3 + [_p])
        L.gs2d_project_bin_and_sort.restype = C.c_int
        L.gs2d_render_fwd.argtypes = [_cfgp, C.c_int32] + [_p] * 8 + [_p]
        L.gs2d_render_fwd.restype = C.c_int
        L.gs2d_loss_l2.argtypes = [C.c_int32, C.c_int32] + [_p] * 5 + [_p]
        L.gs2d_loss_l2.restype = C.c_int
        L.gs2d_render_bwd.argtypes = [_cfgp, C.c_int32] + [_p] * 16 + [_p]
        L.gs2d_render_bwd.restype = C.c_int
        L.gs2d_render_fwd_bwd_l2.argtypes = [_cfgp, C.c_int32] + [_p] * 16 + [_p]
        L.gs2d_render_fwd_bwd_l2.restype = C.c_int
        L.gs2d_merge_workspace_size.argtypes = [C.c_int32]
        L.gs2d_merge_workspace_size.restype = C.c_size_t
        L.gs2d_merge.argtypes = [_cfgp, C.c_int32] + [_p] * 7 + [C.c_int32] + [_p] * 5 + [_p]
        L.gs2d_merge.restype = C.c_int
        L.gs2d_adam_step.argtypes = [C.POINTER(gs2d_adam), C.c_int32, C.c_int32] + [_p] * 5 + [_p]
        L.gs2d_adam_step.restype = C.c_int
        L.gs2d_loss_l2_noalloc.argtypes = [C.c_int32, C.c_int32] + [_p] * 4 + [_p]
        L.gs2d_loss_l2_noalloc.restype = C.c_int
        L.gs2d_read_status.argtypes = [_p, C.POINTER(C.c_int64), C.POINTER(C.c_uint32), _p]
        L.gs2d_read_status.restype = C.c_int
        L.gs2d_status_string.argtypes = [C.c_int]
        L.gs2d_status_string.restype = C.c_char_p
        L.gs2d_debug_check_word.argtypes = [C.POINTER(C.c_uint32), C.c_int32]
        L.gs2d_debug_check_word.restype = C.c_int
        L.gs2d_trace_begin.argtypes = [C.POINTER(C.c_void_p), C.c_int32]
        L.gs2d_trace_begin.restype = C.c_int
        L.gs2d_trace_end.argtypes = []
        L.gs2d_trace_end.restype = C.c_int32
        L.gs2d_trace_kernel_name.argtypes = [C.c_int32]
        L.gs2d_trace_kernel_name.restype = C.c_char_p
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().gs2d_status_string(int(status)).decode()


def check(status: int, where: str) -> None:
    if status != GS2D_OK:
        raise Gs2dError(status, where)


def _stream(stream=None) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _ptr(t, dtype=None, what="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{what}: expected a torch tensor")
    if not t.is_cuda:
        raise ValueError(f"{what}: must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what}: must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{what}: expected {dtype}, got {t.dtype}")
    return t.data_ptr()


_f32, _i32, _u8 = torch.float32, torch.int32, torch.uint8


# --------------------------------------------------------- the C entry points

def gs2d_workspace_size(cfg: gs2d_config, n: int, pair_capacity: int) -> int:
    return int(lib().gs2d_workspace_size(C.byref(cfg), int(n), int(pair_capacity)))


def gs2d_project(cfg, n, xy, shape, rgb, depth, opacity, rec, rect, count, stream=None) -> int:
    return lib().gs2d_project(C.byref(cfg), int(n), _ptr(xy, _f32, "xy"), _ptr(shape, _f32, "shape"),
                              _ptr(rgb, _f32, "rgb"), _ptr(depth, _f32, "depth"),
                              _ptr(opacity, _f32, "opacity"), _ptr(rec, None, "rec"),
                              _ptr(rect, _i32, "rect"), _ptr(count, _i32, "count"), _stream(stream))


def gs2d_bin_and_sort(cfg, n, rec, rect, count, pair_capacity, pairs_out, tile_ranges, sorted_gid,
                      workspace, stream=None) -> int:
    """pairs_out: None (no wait) or a ctypes.c_int64 that receives P."""
    po = C.byref(pairs_out) if pairs_out is not None else None
    return lib().gs2d_bin_and_sort(C.byref(cfg), int(n), _ptr(rec, None, "rec"),
                                   _ptr(rect, _i32, "rect"), _ptr(count, _i32, "count"),
                                   int(pair_capacity), po, _ptr(tile_ranges, _i32, "tile_ranges"),
                                   _ptr(sorted_gid, _i32, "sorted_gid"),
                                   _ptr(workspace, None, "workspace"), _stream(stream))


def gs2d_project_bin_and_sort(cfg, n, xy, shape, rgb, depth, opacity, rec, rect, count,
                              pair_capacity, pairs_out, tile_ranges, sorted_gid, workspace,
                              stream=None) -> int:
    """gs2d_project then gs2d_bin_and_sort in one call (pairs_out as there)."""
    po = C.byref(pairs_out) if pairs_out is not None else None
    return lib().gs2d_project_bin_and_sort(
        C.byref(cfg), int(n), _ptr(xy, _f32, "xy"), _ptr(shape, _f32, "shape"),
        _ptr(rgb, _f32, "rgb"), _ptr(depth, _f32, "depth"), _ptr(opacity, _f32, "opacity"),
        _ptr(rec, None, "rec"), _ptr(rect, _i32, "rect"), _ptr(count, _i32, "count"),
        int(pair_capacity), po, _ptr(tile_ranges, _i32, "tile_ranges"),
        _ptr(sorted_gid, _i32, "sorted_gid"), _ptr(workspace, None, "workspace"), _stream(stream))


def gs2d_render_fwd(cfg, n, rec, tile_ranges, sorted_gid, background, image, t_final, last,
                    workspace=None, stream=None) -> int:
    return lib().gs2d_render_fwd(C.byref(cfg), int(n), _ptr(rec, None, "rec"),
                                 _ptr(tile_ranges, _i32, "tile_ranges"),
                                 _ptr(sorted_gid, _i32, "sorted_gid"),
                                 _ptr(background, _f32, "background"), _ptr(image, _f32, "image"),
                                 _ptr(t_final, _f32, "t_final"), _ptr(last, _i32, "last"),
                                 _ptr(workspace, None, "workspace"), _stream(stream))


def gs2d_loss_l2(height, width, image, target, loss, d_image, workspace, stream=None) -> int:
    return lib().gs2d_loss_l2(int(height), int(width), _ptr(image, _f32, "image"),
                              _ptr(target, _f32, "target"), _ptr(loss, _f32, "loss"),
                              _ptr(d_image, _f32, "d_image"), _ptr(workspace, None, "workspace"),
                              _stream(stream))


def gs2d_loss_l2_noalloc(height, width, image, target, loss, d_image, stream=None) -> int:
    """The L2 loss without a workspace (for callers that cannot allocate;
    the library keeps the reduction's partial sums in its own fixed 4 KiB
    device array, shared by every call on the device)."""
    return lib().gs2d_loss_l2_noalloc(int(height), int(width), _ptr(image, _f32, "image"),
                                      _ptr(target, _f32, "target"), _ptr(loss, _f32, "loss"),
                                      _ptr(d_image, _f32, "d_image"), _stream(stream))


def gs2d_render_bwd(cfg, n, shape, rec, rect, tile_ranges, sorted_gid, background, t_final, last,
                    d_image, d_xy, d_shape, d_rgb, d_opacity, d_background, workspace,
                    stream=None, d_xy_abs=None) -> int:
    return lib().gs2d_render_bwd(
        C.byref(cfg), int(n), _ptr(shape, _f32, "shape"), _ptr(rec, None, "rec"),
        _ptr(rect, _i32, "rect"), _ptr(tile_ranges, _i32, "tile_ranges"),
        _ptr(sorted_gid, _i32, "sorted_gid"), _ptr(background, _f32, "background"),
        _ptr(t_final, _f32, "t_final"), _ptr(last, _i32, "last"), _ptr(d_image, _f32, "d_image"),
        _ptr(d_xy, _f32, "d_xy"), _ptr(d_shape, _f32, "d_shape"), _ptr(d_rgb, _f32, "d_rgb"),
        _ptr(d_opacity, _f32, "d_opacity"), _ptr(d_background, _f32, "d_background"),
        _ptr(d_xy_abs, _f32, "d_xy_abs"), _ptr(workspace, None, "workspace"), _stream(stream))


def gs2d_render_fwd_bwd_l2(cfg, n, shape, rec, rect, tile_ranges, sorted_gid, background, target,
                           image, loss, d_xy, d_shape, d_rgb, d_opacity, d_background, workspace,
                           stream=None, d_xy_abs=None) -> int:
    return lib().gs2d_render_fwd_bwd_l2(
        C.byref(cfg), int(n), _ptr(shape, _f32, "shape"), _ptr(rec, None, "rec"),
        _ptr(rect, _i32, "rect"), _ptr(tile_ranges, _i32, "tile_ranges"),
        _ptr(sorted_gid, _i32, "sorted_gid"), _ptr(background, _f32, "background"),
        _ptr(target, _f32, "target"), _ptr(image, _f32, "image"), _ptr(loss, _f32, "loss"),
        _ptr(d_xy, _f32, "d_xy"), _ptr(d_shape, _f32, "d_shape"), _ptr(d_rgb, _f32, "d_rgb"),
        _ptr(d_opacity, _f32, "d_opacity"), _ptr(d_background, _f32, "d_background"),
        _ptr(d_xy_abs, _f32, "d_xy_abs"), _ptr(workspace, None, "workspace"), _stream(stream))


def gs2d_merge_workspace_size(n: int) -> int:
    return int(lib().gs2d_merge_workspace_size(int(n)))


def gs2d_merge(cfg, n, xy, shape, rgb, rec, count, tile_ranges, sorted_gid, max_merges, out_xy,
               out_shape, out_rgb, merges_out, merge_workspace, stream=None) -> int:
    return lib().gs2d_merge(
        C.byref(cfg), int(n), _ptr(xy, _f32, "xy"), _ptr(shape, _f32, "shape"), _ptr(rgb, _f32, "rgb"),
        _ptr(rec, None, "rec"), _ptr(count, _i32, "count"), _ptr(tile_ranges, _i32, "tile_ranges"),
        _ptr(sorted_gid, _i32, "sorted_gid"), int(max_merges), _ptr(out_xy, _f32, "out_xy"),
        _ptr(out_shape, _f32, "out_shape"), _ptr(out_rgb, _f32, "out_rgb"),
        None if merges_out is None else C.byref(merges_out),
        _ptr(merge_workspace, None, "merge_workspace"), _stream(stream))


def gs2d_adam_step(opt: gs2d_adam, n, width, param, grad, exp_avg, exp_avg_sq, count=None,
                   stream=None) -> int:
    return lib().gs2d_adam_step(
        C.byref(opt), int(n), int(width), _ptr(param, _f32, "param"), _ptr(grad, _f32, "grad"),
        _ptr(exp_avg, _f32, "exp_avg"), _ptr(exp_avg_sq, _f32, "exp_avg_sq"),
        _ptr(count, _i32, "count"), _stream(stream))


def adam_step(param, grad, exp_avg, exp_avg_sq, step, lr, beta1=0.9, beta2=0.999, eps=1e-8,
              count=None, stream=None) -> None:
    """Selective Adam step in place on a [n, width] parameter tensor and its
    two moment tensors (rows with count == 0 untouched when count is given)."""
    n = param.shape[0]
    width = 1 if param.dim() == 1 else int(param[0].numel())
    for t, what in ((grad, "grad"), (exp_avg, "exp_avg"), (exp_avg_sq, "exp_avg_sq")):
        if t.shape != param.shape:
            raise ValueError(f"{what}: shape {tuple(t.shape)} != param {tuple(param.shape)}")
    if count is not None and count.numel() < n:
        raise ValueError("count: fewer entries than parameter rows")
    opt = gs2d_adam(float(lr), float(beta1), float(beta2), float(eps), int(step))
    check(gs2d_adam_step(opt, n, width, param, grad, exp_avg, exp_avg_sq, count, stream),
          "gs2d_adam_step")


def gs2d_read_status(workspace, stream=None):
    """Waits for the stream; returns (status, pairs, flags)."""
    pairs, flags = C.c_int64(0), C.c_uint32(0)
    st = lib().gs2d_read_status(_ptr(workspace, None, "workspace"), C.byref(pairs),
                                C.byref(flags), _stream(stream))
    return st, pairs.value, flags.value


def gs2d_debug_check_word(clear: bool = True):
    """Synchronizes the device; returns (status, word): the bounds-check bits
    set since the last clear (checked build), or GS2D_ERR_UNSUPPORTED."""
    w = C.c_uint32(0)
    st = lib().gs2d_debug_check_word(C.byref(w), 1 if clear else 0)
    return st, w.value


def gs2d_trace_begin(events, max_kernels: int) -> int:
    """events: a ctypes array of 2 * max_kernels cudaEvent_t handles."""
    return lib().gs2d_trace_begin(events, int(max_kernels))


def gs2d_trace_end() -> int:
    return int(lib().gs2d_trace_end())


def gs2d_trace_kernel_name(k: int):
    name = lib().gs2d_trace_kernel_name(int(k))
    return None if name is None else name.decode()


class KernelTrace:
    """Per-kernel device times of the library calls made inside a `with`
    block (gs2d_trace_begin / gs2d_trace_end), on `device`.  Works eagerly
    and under CUDA-graph capture; after a graph replay, durations() gives
    that replay's times.

        tr = KernelTrace(64)
        with tr:
            ...library calls...
        torch.cuda.synchronize()
        tr.durations()   # [(kernel name, ms), ...] in launch order
    """

    def __init__(self, max_kernels: int = 256, device=None):
        self.max_kernels = int(max_kernels)
        self.events = []
        with torch.cuda.device(device):
            s = torch.cuda.current_stream()
            for _ in range(2 * self.max_kernels):
                e = torch.cuda.Event(enable_timing=True)
                e.record(s)  # creates the underlying CUDA event
                self.events.append(e)
            torch.cuda.synchronize()
        self._arr = (C.c_void_p * len(self.events))(*[e.cuda_event for e in self.events])
        self.names = []
        self.launched = 0

    def __enter__(self):
        check(gs2d_trace_begin(self._arr, self.max_kernels), "gs2d_trace_begin")
        return self

    def __exit__(self, *exc):
        self.launched = gs2d_trace_end()
        k = min(self.launched, self.max_kernels)
        self.names = [gs2d_trace_kernel_name(i) for i in range(k)]
        return False

    def durations(self):
        """[(name, ms)] of the traced kernels; synchronize first."""
        return [(n, self.events[2 * i].elapsed_time(self.events[2 * i + 1]))
                for i, n in enumerate(self.names)]


# ------------------------------------------------------------- convenience

class Rasterizer:
    """Buffers and call sequence for one configuration and Gaussian count.

    project -> bin_and_sort -> render_fwd [-> loss_l2 -> render_bwd].
    All tensors live on `device`; nothing here computes, it only allocates
    and calls the library.
    """

    def __init__(self, width, height, n, mode=GS2D_MODE_SUM, cutoff_sigma=3.0, t_min=1e-4,
                 pair_capacity=None, device="cuda", param=GS2D_PARAM_CHOLESKY, scale=1.0):
        self.cfg = make_config(width, height, mode, cutoff_sigma, t_min, param, scale)
        self.width, self.height, self.n, self.mode = int(width), int(height), int(n), int(mode)
        self.device = torch.device(device)
        self.num_tiles = ((width + TILE - 1) // TILE) * ((height + TILE - 1) // TILE)
        d = self.device
        self.rec = torch.empty(max(n, 1) * RECORD_BYTES, dtype=_u8, device=d)
        self.rect = torch.empty((max(n, 1), 4), dtype=_i32, device=d)
        self.count = torch.empty(max(n, 1), dtype=_i32, device=d)
        self.tile_ranges = torch.empty((self.num_tiles, 2), dtype=_i32, device=d)
        self.image = torch.empty((3, height, width), dtype=_f32, device=d)
        comp = mode == GS2D_MODE_COMPOSITE
        self.t_final = torch.empty((height, width), dtype=_f32, device=d) if comp else None
        self.last = torch.empty((height, width), dtype=_i32, device=d) if comp else None
        self.loss = torch.empty(1, dtype=_f32, device=d)
        self.d_image = torch.empty((3, height, width), dtype=_f32, device=d)
        self.d_xy = torch.empty((max(n, 1), 2), dtype=_f32, device=d)
        self.d_shape = torch.empty((max(n, 1), 3), dtype=_f32, device=d)
        self.d_rgb = torch.empty((max(n, 1), 3), dtype=_f32, device=d)
        self.d_opacity = torch.empty(max(n, 1), dtype=_f32, device=d) if comp else None
        self.d_background = torch.empty(3, dtype=_f32, device=d) if comp else None
        self.d_xy_abs = None  # allocated on the first backward that asks for absgrad
        self.pairs = None
        self._alloc_pairs(int(pair_capacity) if pair_capacity is not None else 4 * max(n, 1))

    def _alloc_pairs(self, cap):
        self.capacity = int(cap)
        self.sorted_gid = torch.empty(max(self.capacity, 1), dtype=_i32, device=self.device)
        ws = gs2d_workspace_size(self.cfg, self.n, self.capacity)
        if ws == 0:
            raise ValueError("invalid configuration for gs2d_workspace_size")
        self.workspace = torch.empty(ws, dtype=_u8, device=self.device)

    def project(self, xy, shape, rgb, depth=None, opacity=None):
        self.xy, self.shape, self.rgb, self.depth, self.opacity = xy, shape, rgb, depth, opacity
        check(gs2d_project(self.cfg, self.n, xy, shape, rgb, depth, opacity, self.rec, self.rect,
                           self.count), "gs2d_project")

    def bin_and_sort(self, sync: bool = True, grow: bool = True):
        """sync=True reads P back (and, with grow, reallocates and retries on
        a capacity miss); sync=False leaves everything on the device."""
        if not sync:
            check(gs2d_bin_and_sort(self.cfg, self.n, self.rec, self.rect, self.count,
                                    self.capacity, None, self.tile_ranges, self.sorted_gid,
                                    self.workspace), "gs2d_bin_and_sort")
            return None
        while True:
            P = C.c_int64(0)
            st = gs2d_bin_and_sort(self.cfg, self.n, self.rec, self.rect, self.count,
                                   self.capacity, P, self.tile_ranges, self.sorted_gid,
                                   self.workspace)
            if st == GS2D_ERR_CAPACITY and grow:
                self._alloc_pairs(int(P.value * 1.25) + 1024)
                continue
            check(st, "gs2d_bin_and_sort")
            self.pairs = int(P.value)
            return self.pairs

    def project_bin_and_sort(self, xy, shape, rgb, depth=None, opacity=None, sync: bool = True,
                             grow: bool = True):
        """project() and bin_and_sort() in one library call (same results)."""
        self.xy, self.shape, self.rgb, self.depth, self.opacity = xy, shape, rgb, depth, opacity
        while True:
            P = C.c_int64(0) if sync else None
            st = gs2d_project_bin_and_sort(self.cfg, self.n, xy, shape, rgb, depth, opacity,
                                           self.rec, self.rect, self.count, self.capacity, P,
                                           self.tile_ranges, self.sorted_gid, self.workspace)
            if sync and st == GS2D_ERR_CAPACITY and grow:
                self._alloc_pairs(int(P.value * 1.25) + 1024)
                continue
            check(st, "gs2d_project_bin_and_sort")
            if sync:
                self.pairs = int(P.value)
                return self.pairs
            return None

    def render_fwd(self, background=None):
        self.background = background
        check(gs2d_render_fwd(self.cfg, self.n, self.rec, self.tile_ranges, self.sorted_gid,
                              background, self.image, self.t_final, self.last, self.workspace),
              "gs2d_render_fwd")
        return self.image

    def loss_l2(self, target):
        check(gs2d_loss_l2(self.height, self.width, self.image, target, self.loss, self.d_image,
                           self.workspace), "gs2d_loss_l2")
        return self.loss

    def _absgrad_out(self, absgrad):
        if not absgrad:
            return None
        if self.d_xy_abs is None:
            self.d_xy_abs = torch.empty((max(self.n, 1), 2), dtype=_f32, device=self.device)
        return self.d_xy_abs

    def render_bwd(self, d_image=None, absgrad=False):
        d_image = self.d_image if d_image is None else d_image
        check(gs2d_render_bwd(self.cfg, self.n, self.shape, self.rec, self.rect, self.tile_ranges,
                              self.sorted_gid, self.background, self.t_final, self.last, d_image,
                              self.d_xy, self.d_shape, self.d_rgb, self.d_opacity,
                              self.d_background, self.workspace,
                              d_xy_abs=self._absgrad_out(absgrad)), "gs2d_render_bwd")

    def render_fwd_bwd_l2(self, target, background=None, write_image=True, absgrad=False):
        """Fused forward + L2 loss + backward: composite, one per-tile kernel
        and the gather; sum, the forward with the loss folded in, the pair
        backward and the gather.  Fills loss and the d_* gradients, and the
        image unless write_image is False; d_image (sum mode: kept in the
        workspace instead), t_final and last are not written."""
        self.background = background
        check(gs2d_render_fwd_bwd_l2(self.cfg, self.n, self.shape, self.rec, self.rect,
                                     self.tile_ranges, self.sorted_gid, background, target,
                                     self.image if write_image else None, self.loss, self.d_xy,
                                     self.d_shape, self.d_rgb, self.d_opacity, self.d_background,
                                     self.workspace, d_xy_abs=self._absgrad_out(absgrad)),
              "gs2d_render_fwd_bwd_l2")
        return self.loss

    def step(self, xy, shape, rgb, target, depth=None, opacity=None, background=None, sync=False,
             fused=False):
        """One pass of the whole path: project, bin and sort, forward, L2
        loss, backward (fused=True: projection and binning in one call, and
        forward, loss and backward in another).  Returns the device loss
        tensor."""
        if fused:
            self.project_bin_and_sort(xy, shape, rgb, depth, opacity, sync=sync)
            return self.render_fwd_bwd_l2(target, background)
        self.project(xy, shape, rgb, depth, opacity)
        self.bin_and_sort(sync=sync)
        self.render_fwd(background)
        self.loss_l2(target)
        self.render_bwd()
        return self.loss

    def merge(self, max_merges: int):
        """One round of the moment-matching merge of the parameters last
        projected and binned (sum mode).  Returns (xy, shape, rgb) of the
        merged set as new tensors and the number of pairs merged."""
        n = self.n
        d = self.device
        out_xy = torch.empty((max(n, 1), 2), dtype=_f32, device=d)
        out_shape = torch.empty((max(n, 1), 3), dtype=_f32, device=d)
        out_rgb = torch.empty((max(n, 1), 3), dtype=_f32, device=d)
        ws = torch.empty(gs2d_merge_workspace_size(n), dtype=_u8, device=d)
        m = C.c_int32(0)
        check(gs2d_merge(self.cfg, n, self.xy, self.shape, self.rgb, self.rec, self.count,
                         self.tile_ranges, self.sorted_gid, max_merges, out_xy, out_shape, out_rgb,
                         m, ws), "gs2d_merge")
        k = n - m.value
        return out_xy[:k], out_shape[:k], out_rgb[:k], m.value

    def records(self):
        """The projected records decoded into named tensors (for tests)."""
        f = self.rec.view(torch.float32).view(-1, 12)[: self.n]
        u = self.rec.view(torch.int32).view(-1, 12)[: self.n]
        return dict(mean=f[:, 0:2], conic=f[:, 2:5], rgb=f[:, 5:8],
                    box_x=u[:, 8], box_y=u[:, 9], opacity=f[:, 10], depth=f[:, 11])
