"""Pins of the oracle's render scale (any-resolution rendering, CPU only).

With s output pixels per unit, the mean and the lengths of the shape are
multiplied by s: areas grow by s^2 and peaks keep the colour.  Pinned by the
lattice-sum integral (2 pi |ac| s^2), the peak of a Gaussian whose scaled
mean falls on a pixel centre, equality with parameters scaled beforehand,
and central differences of the loss with respect to the unscaled
parameters (including absgrad)."""
import math

import numpy as np
import pytest

import oracle
from raster_gaussian_02_b300 import synth

from test_oracle_pins import _fd_check


def one(w, h, xy, shape, rgb, scale, k=3.0, param=oracle.CHOLESKY):
    cfg = oracle.Config(w, h, oracle.SUM, cutoff_sigma=k, param=param, scale=scale)
    return oracle.Scene(cfg, np.array([xy], np.float32), np.array([shape], np.float32),
                        np.array([rgb], np.float32))


@pytest.mark.parametrize("s", [1.0, 1.75, 3.0])
def test_integral_scales_with_area(s):
    a, b, c = 1.6, 0.4, 1.3
    size = int(60 * s)
    img = one(size, size, [30.0, 30.0], [a, b, c], [1, 1, 1], s, k=20.0).render()["image"]
    a32, c32 = np.float32(a), np.float32(c)
    assert img[0].sum() == pytest.approx(2 * math.pi * float(a32) * float(c32) * s * s, rel=1e-6)


@pytest.mark.parametrize("s", [0.5, 2.0, 4.0])
def test_peak_keeps_the_colour(s):
    # scaled mean s * mu on the centre of pixel (10, 12)
    mu = [12.5 / s, 10.5 / s]
    img = one(32, 32, mu, [1.5, 0.0, 1.5], [0.3, 0.6, 0.9], s).render()["image"]
    want = np.array([0.3, 0.6, 0.9], np.float32).astype(np.float64)
    np.testing.assert_allclose(img[:, 10, 12], want, rtol=1e-15)


@pytest.mark.parametrize("param", [oracle.CHOLESKY, oracle.SCALE_ROT])
def test_same_as_prescaled_parameters(param):
    wl = synth.random_scene(40, 30, 200, seed=97, diag=(0.5, 3.0), param=param)
    s = np.float32(2.5)
    big = oracle.Config(100, 75, oracle.SUM, param=param, scale=float(s))
    one_ = oracle.Config(100, 75, oracle.SUM, param=param)
    shape = wl.chol.copy()
    shape[:, :2] *= s
    if param == oracle.CHOLESKY:
        shape[:, 2] *= s
    a = oracle.Scene(big, wl.xy, wl.chol, wl.rgb)
    b = oracle.Scene(one_, wl.xy * s, shape, wl.rgb)
    assert np.array_equal(a.proj.conic, b.proj.conic)
    assert np.array_equal(a.proj.aabb, b.proj.aabb)
    # values: the double path scales the exact FP32 inputs, the prescaled
    # scene their FP32-rounded products
    np.testing.assert_allclose(a.render()["image"], b.render()["image"], rtol=2e-6, atol=1e-12)


def test_zero_scale_means_one():
    wl = synth.random_scene(40, 30, 100, seed=101)
    a = oracle.Scene(oracle.Config(40, 30, scale=0.0), wl.xy, wl.chol, wl.rgb)
    b = oracle.Scene(oracle.Config(40, 30, scale=1.0), wl.xy, wl.chol, wl.rgb)
    assert np.array_equal(a.render()["image"], b.render()["image"])


@pytest.mark.parametrize("param,mode", [(oracle.CHOLESKY, oracle.SUM), (oracle.SCALE_ROT, oracle.SUM),
                                        (oracle.CHOLESKY, oracle.COMPOSITE)])
def test_gradients_by_central_differences(param, mode):
    wl = synth.random_scene(20, 16, 40, seed=103, mode=mode, diag=(0.6, 2.5), param=param)
    cfg = oracle.Config(50, 40, mode, param=param, scale=2.5)
    s = oracle.Scene(cfg, wl.xy, wl.chol, wl.rgb, wl.depth, wl.opacity, wl.background)
    tgt = synth.random_scene(50, 40, 1, seed=7).target.astype(np.float64)
    names = ["xy", "chol", "rgb"] + (["opacity"] if mode == oracle.COMPOSITE else [])
    _fd_check(s, tgt, names)


def test_absgrad_scales():
    """absgrad at scale s: per-pixel central differences with respect to the
    unscaled mean."""
    wl = synth.random_scene(16, 12, 20, seed=107, diag=(0.6, 2.0))
    cfg = oracle.Config(48, 36, oracle.SUM, scale=3.0)
    s = oracle.Scene(cfg, wl.xy, wl.chol, wl.rgb)
    tgt = synth.random_scene(48, 36, 1, seed=9).target.astype(np.float64)
    _, dimg = oracle.loss_l2(s.render()["image"], tgt)
    g = s.render_bwd(dimg)
    for gi in np.nonzero(s.proj.count > 0)[0][:6]:
        for d in range(2):
            base = s.xy[gi, d]
            h = 1e-6
            s.xy[gi, d] = base + h
            lp = ((s.render()["image"] - tgt) ** 2).sum(0)
            s.xy[gi, d] = base - h
            lm = ((s.render()["image"] - tgt) ** 2).sum(0)
            s.xy[gi, d] = base
            fd = np.abs((lp - lm) / (2 * h)).sum() / (3 * 48 * 36)
            assert fd == pytest.approx(g["xy_abs"][gi, d], rel=1e-5, abs=1e-12)
