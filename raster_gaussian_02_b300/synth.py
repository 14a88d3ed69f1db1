"""Seeded synthetic inputs for the 2D Gaussian-splatting rasterizer.

This module only draws inputs: target images and Gaussian parameters with the
shapes, sizes and distributions of the workloads the rasterizer is measured
on.  It holds none of the rasterizer's arithmetic and imports neither the
CUDA library nor the oracle, so both sides can be fed the same arrays.

The image-fitting pages measure on photographs (the Kodak set at 768x512 and
DIV2K).  Those are not available here; the procedural targets below stand in
for their shape: smooth regions plus hard edges, values in [0, 1].

All arrays are float32, C-contiguous:
  xy [N,2] pixel units, chol [N,3] = the shape parameters: (l11, l21, l22) of
  the lower-triangular Cholesky factor, or (s_x, s_y, theta) for workloads
  with param == SCALE_ROT; rgb [N,3], depth [N], opacity [N], background
  [3], target [3,H,W] planar.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

SUM, COMPOSITE = 0, 1
CHOLESKY, SCALE_ROT = 0, 1  # what a workload's shape parameters are


# ---------------------------------------------------------------- targets --

def target_blobs(h: int, w: int, rng: np.random.Generator, n_blobs: int = 20) -> np.ndarray:
    """Sum of isotropic blobs (centre uniform over the image, sigma U(4,16) px,
    colour U(0,1)), divided by its maximum so that it lies in [0, 1]."""
    yy, xx = np.mgrid[0:h, 0:w].astype(np.float64) + 0.5
    img = np.zeros((3, h, w), np.float64)
    for _ in range(n_blobs):
        cx, cy = rng.uniform(0, w), rng.uniform(0, h)
        s = rng.uniform(4.0, 16.0)
        col = rng.uniform(0.0, 1.0, size=3)
        g = np.exp(-((xx - cx) ** 2 + (yy - cy) ** 2) / (2 * s * s))
        img += col[:, None, None] * g[None]
    img /= max(img.max(), 1e-12)
    return img.astype(np.float32)


def _value_noise(h: int, w: int, spacing: float, rng: np.random.Generator) -> np.ndarray:
    gh = int(math.ceil(h / spacing)) + 2
    gw = int(math.ceil(w / spacing)) + 2
    lat = rng.random((gh, gw))
    ys = (np.arange(h) + 0.5) / spacing
    xs = (np.arange(w) + 0.5) / spacing
    iy = np.floor(ys).astype(np.int64)
    ix = np.floor(xs).astype(np.int64)
    fy = ys - iy
    fx = xs - ix
    sy = fy * fy * (3 - 2 * fy)
    sx = fx * fx * (3 - 2 * fx)
    v00 = lat[iy][:, ix]
    v01 = lat[iy][:, ix + 1]
    v10 = lat[iy + 1][:, ix]
    v11 = lat[iy + 1][:, ix + 1]
    top = v00 + (v01 - v00) * sx[None, :]
    bot = v10 + (v11 - v10) * sx[None, :]
    return top + (bot - top) * sy[:, None]


def _fill_polygon(mask_out: np.ndarray, vx: np.ndarray, vy: np.ndarray):
    """Even-odd fill of a polygon, sampled at pixel centres, inside its box."""
    h, w = mask_out.shape
    x0 = max(int(np.floor(vx.min())), 0)
    x1 = min(int(np.ceil(vx.max())), w - 1)
    y0 = max(int(np.floor(vy.min())), 0)
    y1 = min(int(np.ceil(vy.max())), h - 1)
    if x0 > x1 or y0 > y1:
        return
    py, px = np.mgrid[y0:y1 + 1, x0:x1 + 1].astype(np.float64) + 0.5
    inside = np.zeros(px.shape, bool)
    m = len(vx)
    for k in range(m):
        xa, ya = vx[k], vy[k]
        xb, yb = vx[(k + 1) % m], vy[(k + 1) % m]
        crosses = (ya > py) != (yb > py)
        with np.errstate(divide="ignore", invalid="ignore"):
            xint = xa + (py - ya) * (xb - xa) / (yb - ya)
        inside ^= crosses & (px < xint)
    mask_out[y0:y1 + 1, x0:x1 + 1] |= inside


def target_noise_polygons(h: int, w: int, rng: np.random.Generator, lattice_scale: float = 1.0,
                          n_polygons: int = 30) -> np.ndarray:
    """Five-octave value noise per channel (finest lattice 8 px times
    lattice_scale, each coarser octave doubles the spacing, amplitude halves
    from coarse to fine: persistence 0.5, smoothstep interpolation), with 30
    opaque star-shaped polygons of 3-8 vertices and uniform colours painted
    on top, clamped to [0, 1]."""
    img = np.zeros((3, h, w), np.float64)
    for ch in range(3):
        acc = np.zeros((h, w))
        norm = 0.0
        for o in range(5):
            spacing = 8.0 * lattice_scale * (2 ** (4 - o))
            amp = 0.5 ** o
            acc += amp * _value_noise(h, w, spacing, rng)
            norm += amp
        img[ch] = acc / norm
    r_max = 0.2 * min(h, w)
    for _ in range(n_polygons):
        nv = int(rng.integers(3, 9))
        cx, cy = rng.uniform(0, w), rng.uniform(0, h)
        R = rng.uniform(0.15, 1.0) * r_max
        ang = np.sort(rng.uniform(0, 2 * np.pi, size=nv))
        rad = R * rng.uniform(0.3, 1.0, size=nv)
        vx = cx + rad * np.cos(ang)
        vy = cy + rad * np.sin(ang)
        m = np.zeros((h, w), bool)
        _fill_polygon(m, vx, vy)
        col = rng.uniform(0.0, 1.0, size=3)
        img[:, m] = col[:, None]
    return np.clip(img, 0.0, 1.0).astype(np.float32)


def _sobel_magnitude(img: np.ndarray) -> np.ndarray:
    lum = 0.299 * img[0] + 0.587 * img[1] + 0.114 * img[2]
    p = np.pad(lum.astype(np.float64), 1, mode="edge")
    gx = (p[:-2, 2:] + 2 * p[1:-1, 2:] + p[2:, 2:]) - (p[:-2, :-2] + 2 * p[1:-1, :-2] + p[2:, :-2])
    gy = (p[2:, :-2] + 2 * p[2:, 1:-1] + p[2:, 2:]) - (p[:-2, :-2] + 2 * p[:-2, 1:-1] + p[:-2, 2:])
    return np.hypot(gx, gy)


# -------------------------------------------------------------- gaussians --

def positions_uniform(n: int, h: int, w: int, rng: np.random.Generator) -> np.ndarray:
    return np.stack([rng.uniform(0, w, n), rng.uniform(0, h, n)], 1).astype(np.float32)


def positions_by_gradient(n: int, target: np.ndarray, rng: np.random.Generator) -> np.ndarray:
    """Pixel drawn with probability proportional to (Sobel luminance magnitude
    + 0.1 * its mean), plus a U(0,1) sub-pixel offset (the density-weighted
    initialisation idea of the FlashImgs README, Training Features)."""
    _, h, w = target.shape
    mag = _sobel_magnitude(target)
    wgt = (mag + 0.1 * mag.mean()).ravel()
    wgt = wgt / wgt.sum()
    idx = rng.choice(h * w, size=n, p=wgt)
    i, j = np.divmod(idx, w)
    x = j + rng.uniform(0, 1, n)
    y = i + rng.uniform(0, 1, n)
    return np.stack([x, y], 1).astype(np.float32)


def cholesky_uniform(n: int, diag: tuple, offdiag_sigma: float, rng: np.random.Generator) -> np.ndarray:
    a = rng.uniform(diag[0], diag[1], n)
    c = rng.uniform(diag[0], diag[1], n)
    b = rng.normal(0.0, offdiag_sigma, n)
    return np.stack([a, b, c], 1).astype(np.float32)


def cholesky_heavy_tail(n: int, rng: np.random.Generator, median: float = 1.5,
                        log_sigma: float = 1.41, s_max: float = 40.0) -> np.ndarray:
    """Log-normal major scale (median 1.5 px, about 1% at the 40 px cap),
    minor scale = major * U(0.3,1), rotation U(0, pi); the covariance
    R diag(s1^2, s2^2) R^T is handed over as its Cholesky factor."""
    s1 = np.minimum(s_max, np.exp(rng.normal(math.log(median), log_sigma, n)))
    s2 = s1 * rng.uniform(0.3, 1.0, n)
    th = rng.uniform(0.0, np.pi, n)
    cs, sn = np.cos(th), np.sin(th)
    sxx = cs * cs * s1 * s1 + sn * sn * s2 * s2
    sxy = cs * sn * (s1 * s1 - s2 * s2)
    syy = sn * sn * s1 * s1 + cs * cs * s2 * s2
    a = np.sqrt(sxx)
    b = sxy / a
    c = np.sqrt(np.maximum(syy - b * b, 1e-12))
    return np.stack([a, b, c], 1).astype(np.float32)


def scale_rot_heavy_tail(n: int, rng: np.random.Generator, median: float = 1.5,
                         log_sigma: float = 1.41, s_max: float = 40.0) -> np.ndarray:
    """The draws of cholesky_heavy_tail handed over as they are:
    (s_x, s_y, theta) = (major, minor, rotation)."""
    s1 = np.minimum(s_max, np.exp(rng.normal(math.log(median), log_sigma, n)))
    s2 = s1 * rng.uniform(0.3, 1.0, n)
    th = rng.uniform(0.0, np.pi, n)
    return np.stack([s1, s2, th], 1).astype(np.float32)


def scale_rot_uniform(n: int, scale, rng: np.random.Generator) -> np.ndarray:
    """(s_x, s_y, theta): scales U(scale) px with random signs (the
    covariance does not depend on them), theta U(-pi, pi)."""
    lo, hi = scale
    sx = rng.uniform(lo, hi, n) * rng.choice([-1.0, 1.0], n)
    sy = rng.uniform(lo, hi, n) * rng.choice([-1.0, 1.0], n)
    th = rng.uniform(-np.pi, np.pi, n)
    return np.stack([sx, sy, th], 1).astype(np.float32)


# -------------------------------------------------------------- workloads --

@dataclasses.dataclass
class Workload:
    name: str
    width: int
    height: int
    mode: int
    xy: np.ndarray
    chol: np.ndarray
    rgb: np.ndarray
    target: np.ndarray | None
    depth: np.ndarray | None = None
    opacity: np.ndarray | None = None
    background: np.ndarray | None = None
    cutoff_sigma: float = 3.0
    t_min: float = 1e-4
    param: int = CHOLESKY
    scale: float = 1.0  # render scale: output pixels per unit of xy and shape

    @property
    def n(self) -> int:
        return int(self.xy.shape[0])


def _rgb(n, rng):
    return rng.uniform(0.0, 1.0, (n, 3)).astype(np.float32)


def small_64x64(seed: int = 1000, n: int = 1000) -> Workload:
    """64x64 blob target; 1,000 Gaussians, xy uniform, diag U(0.5,3) px,
    off-diagonal N(0,0.5), rgb U(0,1); accumulated sum."""
    rng = np.random.default_rng(seed)
    h = w = 64
    tgt = target_blobs(h, w, rng)
    return Workload("small_64x64_1k", w, h, SUM, positions_uniform(n, h, w, rng),
                    cholesky_uniform(n, (0.5, 3.0), 0.5, rng), _rgb(n, rng), tgt)


def image_768x512(seed: int = 2000, n: int = 50_000) -> Workload:
    """768x512 noise+polygon target; 50,000 Gaussians placed by gradient
    magnitude, diag U(0.7,2.5) px, off-diagonal N(0,0.5), rgb U(0,1)."""
    rng = np.random.default_rng(seed)
    h, w = 512, 768
    tgt = target_noise_polygons(h, w, rng)
    return Workload(f"image_768x512_{n // 1000}k", w, h, SUM, positions_by_gradient(n, tgt, rng),
                    cholesky_uniform(n, (0.7, 2.5), 0.5, rng), _rgb(n, rng), tgt)


def heavy_2048x1360(seed: int = 3000, n: int = 300_000) -> Workload:
    """2048x1360 target (lattice scaled by 2048/768); 300,000 rotated
    Gaussians with heavy-tailed sizes, placed by gradient magnitude."""
    rng = np.random.default_rng(seed)
    h, w = 1360, 2048
    tgt = target_noise_polygons(h, w, rng, lattice_scale=2048 / 768)
    return Workload("heavy_2048x1360_300k", w, h, SUM, positions_by_gradient(n, tgt, rng),
                    cholesky_heavy_tail(n, rng), _rgb(n, rng), tgt)


def heavy_1024x680(seed: int = 3000, n: int = 75_000) -> Workload:
    """A quarter of heavy_2048x1360 (half the width and height, a quarter of
    the Gaussians; the same target lattice, density and size distribution),
    small enough for profiler captures of the same kernels."""
    rng = np.random.default_rng(seed)
    h, w = 680, 1024
    tgt = target_noise_polygons(h, w, rng, lattice_scale=2048 / 768)
    return Workload("heavy_1024x680_75k", w, h, SUM, positions_by_gradient(n, tgt, rng),
                    cholesky_heavy_tail(n, rng), _rgb(n, rng), tgt)


def image_768x512_sr(seed: int = 2000, n: int = 50_000) -> Workload:
    """The 768x512 workload with scale-rotation shapes: scales U(0.7,2.5) px,
    rotation U(-pi, pi)."""
    rng = np.random.default_rng(seed)
    h, w = 512, 768
    tgt = target_noise_polygons(h, w, rng)
    return Workload(f"image_768x512_{n // 1000}k_sr", w, h, SUM, positions_by_gradient(n, tgt, rng),
                    scale_rot_uniform(n, (0.7, 2.5), rng), _rgb(n, rng), tgt, param=SCALE_ROT)


def heavy_2048x1360_sr(seed: int = 3000, n: int = 300_000) -> Workload:
    """heavy_2048x1360 with the same draws given as (scale, rotation)."""
    rng = np.random.default_rng(seed)
    h, w = 1360, 2048
    tgt = target_noise_polygons(h, w, rng, lattice_scale=2048 / 768)
    return Workload("heavy_2048x1360_300k_sr", w, h, SUM, positions_by_gradient(n, tgt, rng),
                    scale_rot_heavy_tail(n, rng), _rgb(n, rng), tgt, param=SCALE_ROT)


def composite_768x512(seed: int = 4000, n: int = 50_000) -> Workload:
    """The 768x512 workload, alpha-composited: depth U(0,1), opacity
    sigmoid(N(0,1)), background U(0,1)^3."""
    base = image_768x512(seed, n)
    rng = np.random.default_rng(seed + 1)
    depth = rng.uniform(0.0, 1.0, n).astype(np.float32)
    opacity = (1.0 / (1.0 + np.exp(-rng.normal(0.0, 1.0, n)))).astype(np.float32)
    bg = rng.uniform(0.0, 1.0, 3).astype(np.float32)
    return dataclasses.replace(base, name=f"composite_768x512_{n // 1000}k", mode=COMPOSITE,
                               depth=depth, opacity=opacity, background=bg)


def render_uniform(width: int, height: int, n: int, seed: int = 5000, with_target: bool = False) -> Workload:
    """Forward-only throughput scene: xy uniform, diag U(0.5,4) px,
    off-diagonal N(0,0.5), rgb U(0,1)."""
    rng = np.random.default_rng(seed)
    tgt = target_blobs(height, width, rng) if with_target else None
    return Workload(f"render_{width}x{height}_{n}", width, height, SUM,
                    positions_uniform(n, height, width, rng),
                    cholesky_uniform(n, (0.5, 4.0), 0.5, rng), _rgb(n, rng), tgt)


def render_4096x4096(seed: int = 5000, n: int = 2_000_000) -> Workload:
    return render_uniform(4096, 4096, n, seed)


def render_2048x2048(seed: int = 5000, n: int = 500_000) -> Workload:
    """A quarter of the 4096x4096 render scene (same density and sizes), small
    enough for profiler captures."""
    return render_uniform(2048, 2048, n, seed)


def random_scene(width: int, height: int, n: int, seed: int, mode: int = SUM,
                 diag=(0.5, 3.0), offdiag_sigma: float = 0.5, margin: float = 0.0,
                 param: int = CHOLESKY) -> Workload:
    """Small random scene for parity and edge cases; `margin` px of the
    positions may fall outside the image.  param == SCALE_ROT draws the
    scales from `diag` instead of the Cholesky diagonal."""
    rng = np.random.default_rng(seed)
    xy = np.stack([rng.uniform(-margin, width + margin, n),
                   rng.uniform(-margin, height + margin, n)], 1).astype(np.float32)
    if param == SCALE_ROT:
        chol = scale_rot_uniform(n, diag, rng)
    else:
        chol = cholesky_uniform(n, diag, offdiag_sigma, rng)
        # random signs on the diagonal: L L^T does not depend on them
        chol[:, 0] *= rng.choice([-1.0, 1.0], n).astype(np.float32)
        chol[:, 2] *= rng.choice([-1.0, 1.0], n).astype(np.float32)
    rgb = _rgb(n, rng)
    tgt = rng.uniform(0.0, 1.0, (3, height, width)).astype(np.float32)
    wl = Workload(f"random_{width}x{height}_{n}", width, height, mode, xy, chol, rgb, tgt,
                  param=param)
    if mode == COMPOSITE:
        wl.depth = rng.uniform(0.0, 1.0, n).astype(np.float32)
        wl.opacity = (1.0 / (1.0 + np.exp(-rng.normal(0.0, 1.0, n)))).astype(np.float32)
        wl.background = rng.uniform(0.0, 1.0, 3).astype(np.float32)
    return wl


def d_image(height: int, width: int, seed: int, scale: float = 1.0) -> np.ndarray:
    """A seeded upstream gradient dL/dC [3,H,W] for backward-only checks."""
    rng = np.random.default_rng(seed)
    return (scale * rng.normal(0.0, 1.0, (3, height, width))).astype(np.float32)


WORKLOADS = {
    "small_64x64_1k": small_64x64,
    "image_768x512_50k": image_768x512,
    "heavy_2048x1360_300k": heavy_2048x1360,
    "heavy_1024x680_75k": heavy_1024x680,
    "image_768x512_50k_sr": image_768x512_sr,
    "heavy_2048x1360_300k_sr": heavy_2048x1360_sr,
    "composite_768x512_50k": composite_768x512,
    "render_4096x4096_2m": render_4096x4096,
    "render_2048x2048_500k": render_2048x2048,
}
