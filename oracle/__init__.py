"""Python face of the CPU oracle (test infrastructure, not product code).

Only the test suite, the package's smoke check and the benchmark's CPU
baseline leg import this package.  It wraps oracle/libgs2d_oracle.so (plain
C, fp64 values, FP32 touch decisions) with numpy arrays and shares nothing
with the CUDA library or its Python binding.

The parameters of a scene are FP32 (what a caller stores); the oracle takes
its touch decisions from those FP32 values and evaluates every weight,
colour and gradient in double from the same values widened to double.
Finite-difference checks perturb the double copies while the FP32 mask data
stays fixed, which is the "mask held constant" reading of the gradient.
"""
from __future__ import annotations

import ctypes as C
import dataclasses
import os

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(_build.build())
        _declare(_lib)
    return _lib


_omp = None


def omp_lib():
    """The multi-threaded timing driver (libgs2d_oracle_omp.so): the same
    per-pixel functions, tile rows spread over OpenMP threads."""
    global _omp
    if _omp is None:
        _omp = C.CDLL(_build.build_omp())
        _declare(_omp)
        cfgp = C.POINTER(RefCfg)
        _omp.gs2dref_omp_threads.argtypes = [_i32]
        _omp.gs2dref_omp_threads.restype = _i32
        _omp.gs2dref_omp_render_fwd.argtypes = [cfgp] + [_p] * 14
        _omp.gs2dref_omp_render_fwd.restype = _i64
        _omp.gs2dref_omp_render_bwd.argtypes = [cfgp, _i32] + [_p] * 19 + [_i64]
        _omp.gs2dref_omp_render_bwd.restype = None
    return _omp


def omp_threads(want: int = 0) -> int:
    """Sets (want > 0) and returns the thread count of the OpenMP driver."""
    return int(omp_lib().gs2dref_omp_threads(int(want)))


class use_library:
    """Context manager that points this module at another build of the
    oracle source (the mutation tests plant mistakes in copies of it)."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        self.saved = lib()
        _lib = C.CDLL(self.path)
        _declare(_lib)
        return _lib

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


class RefCfg(C.Structure):
    _fields_ = [("width", C.c_int32), ("height", C.c_int32), ("tile", C.c_int32),
                ("mode", C.c_int32), ("cutoff_sigma", C.c_float), ("t_min", C.c_float),
                ("param", C.c_int32), ("scale", C.c_float)]


SUM, COMPOSITE = 0, 1
# Shape parameters per Gaussian: a Cholesky factor (l11, l21, l22) or a scale
# and rotation angle (s_x, s_y, theta).
CHOLESKY, SCALE_ROT = 0, 1

_p = C.c_void_p
_i32, _i64 = C.c_int32, C.c_int64


def _declare(L):
    cfgp = C.POINTER(RefCfg)
    L.gs2dref_num_tiles.argtypes = [cfgp]
    L.gs2dref_num_tiles.restype = _i32
    L.gs2dref_project.argtypes = [cfgp, _i32] + [_p] * 9
    L.gs2dref_project.restype = _i32
    L.gs2dref_bin.argtypes = [cfgp, _i32, _p, _p, _p, _p, _p]
    L.gs2dref_bin.restype = _i64
    L.gs2dref_render_fwd.argtypes = [cfgp] + [_p] * 14
    L.gs2dref_render_fwd.restype = _i64
    L.gs2dref_render_pixels.argtypes = [cfgp] + [_p] * 11 + [_i64] + [_p] * 4
    L.gs2dref_render_pixels.restype = None
    L.gs2dref_render_brute.argtypes = [cfgp, _i32] + [_p] * 12
    L.gs2dref_render_brute.restype = None
    L.gs2dref_merge.argtypes = [cfgp, _i32] + [_p] * 6 + [_i32] + [_p] * 4
    L.gs2dref_merge.restype = _i32
    L.gs2dref_merge_cost.argtypes = [cfgp, _i32] + [_p] * 5
    L.gs2dref_merge_cost.restype = None
    L.gs2dref_sincos_f32.argtypes = [_i32, _p, _p, _p]
    L.gs2dref_sincos_f32.restype = None
    L.gs2dref_loss_l2.argtypes = [_i32, _i32, _p, _p, _p]
    L.gs2dref_loss_l2.restype = C.c_double
    L.gs2dref_render_bwd.argtypes = [cfgp, _i32] + [_p] * 19
    L.gs2dref_render_bwd.restype = None
    L.gs2dref_render_bwd_gaussians.argtypes = [cfgp, _i32] + [_p] * 12 + [_p, _i32] + [_p] * 5
    L.gs2dref_render_bwd_gaussians.restype = None


@dataclasses.dataclass
class Config:
    width: int
    height: int
    mode: int = SUM
    cutoff_sigma: float = 3.0
    t_min: float = 1e-4
    tile: int = 16
    param: int = CHOLESKY
    scale: float = 1.0  # output pixels per unit of xy and shape

    def c(self) -> RefCfg:
        return RefCfg(self.width, self.height, self.tile, self.mode, self.cutoff_sigma, self.t_min,
                      self.param, self.scale)

    @property
    def tiles_x(self) -> int:
        return (self.width + self.tile - 1) // self.tile

    @property
    def tiles_y(self) -> int:
        return (self.height + self.tile - 1) // self.tile

    @property
    def num_tiles(self) -> int:
        return self.tiles_x * self.tiles_y


def _ptr(a):
    return None if a is None else a.ctypes.data


def _f32(a, shape=None):
    if a is None:
        return None
    a = np.ascontiguousarray(a, dtype=np.float32)
    if shape is not None:
        a = a.reshape(shape)
    return a


def _f64(a, shape=None):
    if a is None:
        return None
    a = np.ascontiguousarray(a, dtype=np.float64)
    if shape is not None:
        a = a.reshape(shape)
    return a


@dataclasses.dataclass
class Projection:
    conic: np.ndarray   # [n,3] float32 (A, B, C) of the inverse covariance
    aabb: np.ndarray    # [n,4] int32 pixel box (x0, y0, x1, y1), inclusive
    rect: np.ndarray    # [n,4] int32 tile rectangle (tx0, ty0, tx1, ty1), inclusive
    count: np.ndarray   # [n] int32 tiles touched, 0 when culled
    valid: int


def project(cfg: Config, xy, chol, rgb, depth=None, opacity=None) -> Projection:
    n = int(np.asarray(xy).reshape(-1, 2).shape[0])
    xy, chol, rgb = _f32(xy, (n, 2)), _f32(chol, (n, 3)), _f32(rgb, (n, 3))
    depth, opacity = _f32(depth), _f32(opacity)
    if cfg.mode == COMPOSITE and (depth is None or opacity is None):
        raise ValueError("composite mode needs depth and opacity")
    conic = np.zeros((n, 3), np.float32)
    aabb = np.zeros((n, 4), np.int32)
    rect = np.zeros((n, 4), np.int32)
    count = np.zeros((n,), np.int32)
    c = cfg.c()
    valid = lib().gs2dref_project(C.byref(c), n, _ptr(xy), _ptr(chol), _ptr(rgb), _ptr(depth),
                                  _ptr(opacity), _ptr(conic), _ptr(aabb), _ptr(rect), _ptr(count))
    return Projection(conic, aabb, rect, count, int(valid))


def sincos_f32(theta):
    """(sin, cos) of FP32 angles by the FP32 sequence the scale-rotation mask
    data use."""
    th = _f32(theta).ravel()
    sn, cs = np.zeros_like(th), np.zeros_like(th)
    lib().gs2dref_sincos_f32(int(th.size), _ptr(th), _ptr(sn), _ptr(cs))
    return sn, cs


def bin_tiles(cfg: Config, proj: Projection, depth=None):
    """Returns (ranges[T,2] int32, sorted_gid[P] int32)."""
    n = proj.count.shape[0]
    depth = _f32(depth)
    c = cfg.c()
    P = lib().gs2dref_bin(C.byref(c), n, _ptr(proj.rect), _ptr(proj.count), _ptr(depth), None, None)
    ranges = np.zeros((cfg.num_tiles, 2), np.int32)
    sorted_gid = np.zeros((max(P, 1),), np.int32)
    lib().gs2dref_bin(C.byref(c), n, _ptr(proj.rect), _ptr(proj.count), _ptr(depth), _ptr(ranges),
                      _ptr(sorted_gid))
    return ranges, sorted_gid[:P]


class Scene:
    """One scene: FP32 parameters, their projection and tile lists, and the
    double copies used for values (which finite differences may perturb)."""

    def __init__(self, cfg: Config, xy, chol, rgb, depth=None, opacity=None, background=None):
        self.cfg = cfg
        n = int(np.asarray(xy).reshape(-1, 2).shape[0])
        self.n = n
        self.xy_f = _f32(xy, (n, 2))
        self.chol_f = _f32(chol, (n, 3))
        self.rgb_f = _f32(rgb, (n, 3))
        self.depth_f = _f32(depth)
        self.opacity_f = _f32(opacity)
        self.bg_f = _f32(background) if background is not None else np.zeros(3, np.float32)
        self.proj = project(cfg, self.xy_f, self.chol_f, self.rgb_f, self.depth_f, self.opacity_f)
        self.ranges, self.sorted_gid = bin_tiles(cfg, self.proj, self.depth_f)
        self.reset_values()

    def reset_values(self):
        self.xy = self.xy_f.astype(np.float64)
        self.chol = self.chol_f.astype(np.float64)
        self.rgb = self.rgb_f.astype(np.float64)
        self.opacity = (self.opacity_f.astype(np.float64) if self.opacity_f is not None
                        else np.zeros(self.n, np.float64))
        self.bg = self.bg_f.astype(np.float64)

    @property
    def num_pairs(self) -> int:
        return int(self.sorted_gid.shape[0])

    def _common(self):
        return (_ptr(self.xy), _ptr(self.chol), _ptr(self.rgb), _ptr(self.opacity), _ptr(self.bg),
                _ptr(self.xy_f), _ptr(self.proj.conic), _ptr(self.proj.aabb))

    def _lists(self):
        # keep a non-empty buffer alive for the C side even when P == 0
        if self.sorted_gid.size == 0:
            self._sg_keep = np.zeros(1, np.int32)
            return _ptr(self.ranges), _ptr(self._sg_keep)
        return _ptr(self.ranges), _ptr(self.sorted_gid)

    def render(self, omp: bool = False):
        """Full image: returns dict(image[3,H,W], t_final[H,W], last[H,W], margin[H,W], masked).
        omp: through the OpenMP timing driver (same per-pixel functions)."""
        H, W = self.cfg.height, self.cfg.width
        img = np.zeros((3, H, W), np.float64)
        tf = np.zeros((H, W), np.float64)
        last = np.zeros((H, W), np.int32)
        margin = np.zeros((H, W), np.float64)
        c = self.cfg.c()
        fn = omp_lib().gs2dref_omp_render_fwd if omp else lib().gs2dref_render_fwd
        masked = fn(C.byref(c), *self._common(), *self._lists(), _ptr(img), _ptr(tf), _ptr(last),
                    _ptr(margin))
        return dict(image=img, t_final=tf, last=last, margin=margin, masked=int(masked))

    def render_pixels(self, pix):
        """Forward at linear pixel indices pix (i*W + j)."""
        pix = np.ascontiguousarray(pix, dtype=np.int64)
        m = pix.shape[0]
        out = np.zeros((m, 3), np.float64)
        tf = np.zeros(m, np.float64)
        last = np.zeros(m, np.int32)
        margin = np.zeros(m, np.float64)
        c = self.cfg.c()
        lib().gs2dref_render_pixels(C.byref(c), *self._common(), *self._lists(), _ptr(pix), m,
                                    _ptr(out), _ptr(tf), _ptr(last), _ptr(margin))
        return dict(rgb=out, t_final=tf, last=last, margin=margin)

    def render_brute(self):
        H, W = self.cfg.height, self.cfg.width
        img = np.zeros((3, H, W), np.float64)
        tf = np.zeros((H, W), np.float64)
        depth = self.depth_f if self.depth_f is not None else np.zeros(self.n, np.float32)
        c = self.cfg.c()
        lib().gs2dref_render_brute(C.byref(c), self.n, *self._common(), _ptr(self.proj.count),
                                   _ptr(depth), _ptr(img), _ptr(tf))
        return dict(image=img, t_final=tf)

    def render_bwd(self, d_image, omp: bool = False):
        """omp: through the OpenMP timing driver (same per-pixel functions,
        per-thread accumulators summed in thread order)."""
        d_image = _f64(d_image, (3, self.cfg.height, self.cfg.width))
        n = self.n
        dxy = np.zeros((n, 2)); dchol = np.zeros((n, 3)); drgb = np.zeros((n, 3))
        dop = np.zeros(n); dbg = np.zeros(3); dconic = np.zeros((n, 3)); dabs = np.zeros((n, 2))
        c = self.cfg.c()
        args = (C.byref(c), n, *self._common(), _ptr(self.proj.count), *self._lists(), _ptr(d_image),
                _ptr(dxy), _ptr(dchol), _ptr(drgb), _ptr(dop), _ptr(dbg), _ptr(dconic), _ptr(dabs))
        if omp:
            omp_lib().gs2dref_omp_render_bwd(*args, 0)
        else:
            lib().gs2dref_render_bwd(*args)
        return dict(xy=dxy, chol=dchol, rgb=drgb, opacity=dop, background=dbg, conic=dconic,
                    xy_abs=dabs)

    def render_bwd_gaussians(self, d_image, gids):
        d_image = _f64(d_image, (3, self.cfg.height, self.cfg.width))
        gids = np.ascontiguousarray(gids, dtype=np.int32)
        m = gids.shape[0]
        dxy = np.zeros((m, 2)); dchol = np.zeros((m, 3)); drgb = np.zeros((m, 3)); dop = np.zeros(m)
        dabs = np.zeros((m, 2))
        c = self.cfg.c()
        lib().gs2dref_render_bwd_gaussians(C.byref(c), self.n, *self._common(),
                                           _ptr(self.proj.count), *self._lists(), _ptr(d_image),
                                           _ptr(gids), m, _ptr(dxy), _ptr(dchol), _ptr(drgb),
                                           _ptr(dop), _ptr(dabs))
        return dict(xy=dxy, chol=dchol, rgb=drgb, opacity=dop, xy_abs=dabs)


def loss_l2(image, target):
    """Returns (loss, d_image) in double: loss = mean over 3HW of (C - target)^2."""
    image = _f64(image)
    target = _f64(target)
    if image.shape != target.shape or image.ndim != 3 or image.shape[0] != 3:
        raise ValueError("image and target must both be [3,H,W]")
    _, h, w = image.shape
    d = np.zeros_like(image)
    loss = lib().gs2dref_loss_l2(h, w, _ptr(image), _ptr(target), _ptr(d))
    return float(loss), d


def merge(cfg: Config, xy, shape, rgb, max_merges: int, with_partners: bool = False):
    """One round of the moment-matching merge (sum mode).  Returns
    (xy, shape, rgb) of the merged set (FP32) and the number of merges (and,
    with_partners, each input's merged partner if it was the pair's lower
    index, else -1)."""
    if cfg.mode != SUM:
        raise ValueError("the merge is defined for the accumulated sum")
    n = int(np.asarray(xy).reshape(-1, 2).shape[0])
    xy, shape, rgb = _f32(xy, (n, 2)), _f32(shape, (n, 3)), _f32(rgb, (n, 3))
    proj = project(cfg, xy, shape, rgb)
    ranges, sorted_gid = bin_tiles(cfg, proj)
    sg = sorted_gid if sorted_gid.size else np.zeros(1, np.int32)
    oxy, osh, orgb = np.zeros_like(xy), np.zeros_like(shape), np.zeros_like(rgb)
    partner = np.zeros(max(n, 1), np.int32)
    m = lib().gs2dref_merge(C.byref(cfg.c()), n, _ptr(xy), _ptr(shape), _ptr(rgb), _ptr(proj.count),
                            _ptr(ranges), _ptr(sg), int(max_merges), _ptr(oxy), _ptr(osh), _ptr(orgb),
                            _ptr(partner))
    k = n - m
    out = (oxy[:k], osh[:k], orgb[:k], int(m))
    return out + (partner[:n],) if with_partners else out


def merge_cost(cfg: Config, xa, sha, xb, shb):
    """The merge's pairing cost (FP32) of the k-th Gaussian of (xa, sha)
    against the k-th of (xb, shb), shapes in cfg.param's parameters."""
    xa = _f32(xa, (-1, 2))
    m = xa.shape[0]
    xb, sha, shb = _f32(xb, (m, 2)), _f32(sha, (m, 3)), _f32(shb, (m, 3))
    out = np.zeros(max(m, 1), np.float32)
    lib().gs2dref_merge_cost(C.byref(cfg.c()), m, _ptr(xa), _ptr(sha), _ptr(xb), _ptr(shb), _ptr(out))
    return out[:m]


def step(cfg: Config, xy, chol, rgb, target, depth=None, opacity=None, background=None,
         omp: bool = False):
    """One pass of the whole path on the CPU: project, bin, render, L2 loss,
    backward.  Returns (scene, forward dict, loss, d_image, gradient dict).
    omp: render and backward through the OpenMP timing driver."""
    s = Scene(cfg, xy, chol, rgb, depth, opacity, background)
    fwd = s.render(omp=omp)
    loss, dimg = loss_l2(fwd["image"], target)
    grads = s.render_bwd(dimg, omp=omp)
    return s, fwd, loss, dimg, grads


def adam_step(param, grad, exp_avg, exp_avg_sq, step: int, lr: float, beta1: float = 0.9,
              beta2: float = 0.999, eps: float = 1e-8, count=None):
    """One selective Adam step on row-aligned state (DrawingWithGaussians
    README, MLX-specific notes: the COLMAP trainer carries row-aligned
    optimizer state for its selective Adam).  The pages name the optimizer
    and give no formula; this is Adam as Kingma and Ba define it, in the
    order they state it, in double:
        m_t = beta1 m_{t-1} + (1 - beta1) g_t
        v_t = beta2 v_{t-1} + (1 - beta2) g_t^2
        mhat = m_t / (1 - beta1^t),  vhat = v_t / (1 - beta2^t)
        p_t = p_{t-1} - lr mhat / (sqrt(vhat) + eps)
    param, grad, exp_avg, exp_avg_sq: [n, width] (or [n]); count: [n] or
    None.  Selective: rows with count == 0 keep p, m and v.  Returns new
    (param, exp_avg, exp_avg_sq) as float64 arrays; the inputs are left as
    they are."""
    p = np.array(param, np.float64, copy=True)
    g = np.asarray(grad, np.float64)
    m = np.array(exp_avg, np.float64, copy=True)
    v = np.array(exp_avg_sq, np.float64, copy=True)
    if not (p.shape == g.shape == m.shape == v.shape):
        raise ValueError("param, grad and both moments must have one shape")
    if step < 1:
        raise ValueError("step counts from 1")
    rows = np.ones(p.shape[0], bool) if count is None else np.asarray(count)[: p.shape[0]] != 0
    m_new = beta1 * m + (1.0 - beta1) * g
    v_new = beta2 * v + (1.0 - beta2) * g * g
    mhat = m_new / (1.0 - beta1 ** step)
    vhat = v_new / (1.0 - beta2 ** step)
    p_new = p - lr * mhat / (np.sqrt(vhat) + eps)
    sel = rows.reshape((-1,) + (1,) * (p.ndim - 1))
    return np.where(sel, p_new, p), np.where(sel, m_new, m), np.where(sel, v_new, v)
