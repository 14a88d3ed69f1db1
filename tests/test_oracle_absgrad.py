"""Pins of the oracle's absgrad output (CPU only).

absgrad of a Gaussian = (sum over pixels p of |dL_p/dmu_x|, same for mu_y),
L_p being pixel p's term of the L2 loss (its three channels together), so
that the per-pixel contributions cannot cancel.  Pinned against central
differences of every pixel's loss term, the triangle inequality against the
plain mean gradient, the cancellation in a symmetric scene, and the two
backward traversals agreeing.
"""
import numpy as np
import pytest

import oracle
from raster_gaussian_02_b300 import synth


def scene_of(wl, **kw):
    cfg = oracle.Config(wl.width, wl.height, wl.mode, param=wl.param, **kw)
    return oracle.Scene(cfg, wl.xy, wl.chol, wl.rgb, wl.depth, wl.opacity, wl.background)


def pixel_losses(s, target):
    img = s.render()["image"]
    H, W = s.cfg.height, s.cfg.width
    return ((img - target) ** 2).sum(0) / (3 * H * W)


@pytest.mark.parametrize("mode,param", [(oracle.SUM, oracle.CHOLESKY),
                                        (oracle.COMPOSITE, oracle.CHOLESKY),
                                        (oracle.SUM, oracle.SCALE_ROT)])
def test_absgrad_by_per_pixel_central_differences(mode, param):
    wl = synth.random_scene(24, 20, 30, seed=71, mode=mode, diag=(1.0, 4.0), param=param)
    s = scene_of(wl)
    tgt = wl.target.astype(np.float64)
    _, dimg = oracle.loss_l2(s.render()["image"], tgt)
    g = s.render_bwd(dimg)
    valid = np.nonzero(s.proj.count > 0)[0]
    scale = np.abs(g["xy_abs"]).max()
    for gi in valid[:12]:
        for d in range(2):
            base = s.xy[gi, d]
            h = 1e-5 * max(1.0, abs(base))
            s.xy[gi, d] = base + h
            lp = pixel_losses(s, tgt)
            s.xy[gi, d] = base - h
            lm = pixel_losses(s, tgt)
            s.xy[gi, d] = base
            fd = np.abs((lp - lm) / (2 * h)).sum()
            assert abs(fd - g["xy_abs"][gi, d]) <= 1e-6 * scale + 1e-14, (gi, d, fd, g["xy_abs"][gi, d])


def test_triangle_inequality_and_culled_zero():
    wl = synth.random_scene(48, 40, 300, seed=73, diag=(0.5, 5.0), margin=10)
    s = scene_of(wl)
    _, dimg = oracle.loss_l2(s.render()["image"], wl.target.astype(np.float64))
    g = s.render_bwd(dimg)
    assert np.all(g["xy_abs"] >= np.abs(g["xy"]) - 1e-15)
    assert np.all(g["xy_abs"][s.proj.count == 0] == 0)
    assert (g["xy_abs"] > 1.5 * np.abs(g["xy"])).mean() > 0.3  # contributions do cancel


def test_symmetric_scene_cancels_only_the_plain_gradient():
    """One isotropic Gaussian centred on a pixel centre, target zero: the
    per-pixel contributions are odd in dx, so the mean gradient is 0 while
    absgrad is positive."""
    cfg = oracle.Config(33, 33, oracle.SUM)
    s = oracle.Scene(cfg, np.array([[16.5, 16.5]], np.float32), np.array([[3.0, 0.0, 3.0]], np.float32),
                     np.array([[0.2, 0.5, 0.9]], np.float32))
    _, dimg = oracle.loss_l2(s.render()["image"], np.zeros((3, 33, 33)))
    g = s.render_bwd(dimg)
    assert np.all(np.abs(g["xy"][0]) < 1e-15)
    assert np.all(g["xy_abs"][0] > 1e-6)
    assert g["xy_abs"][0, 0] == pytest.approx(g["xy_abs"][0, 1], rel=1e-12)


@pytest.mark.parametrize("mode", [oracle.SUM, oracle.COMPOSITE])
def test_two_traversals_agree(mode):
    wl = synth.random_scene(45, 38, 150, seed=79, mode=mode, diag=(0.5, 5.0))
    s = scene_of(wl)
    dimg = synth.d_image(38, 45, seed=5).astype(np.float64)
    full = s.render_bwd(dimg)
    part = s.render_bwd_gaussians(dimg, np.arange(wl.n, dtype=np.int32))
    np.testing.assert_allclose(part["xy_abs"], full["xy_abs"], rtol=1e-10,
                               atol=1e-12 * np.abs(full["xy_abs"]).max())
