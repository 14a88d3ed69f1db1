"""Pins of the oracle's scale-rotation parameterization (CPU only).

Shape parameters (s_x, s_y, theta) give Sigma = R(theta) diag(s_x^2, s_y^2)
R(theta)^T.  The oracle is tied to: scipy's normal density with Sigma formed
here by numpy, the FP32 inverse covariance against that Sigma, the theta = 0
case against the Cholesky path, the symmetries of the parameterization
(swapping the axes with a quarter turn, the sign of a scale), and central
finite differences for the gradients with respect to (s_x, s_y, theta).
"""
import math

import numpy as np
import pytest
from scipy.stats import multivariate_normal

import oracle
from raster_gaussian_02_b300 import synth

from test_oracle_pins import _fd_check


def sigma_of(sh):
    """Sigma [.., 2, 2] in double from (s_x, s_y, theta) rows."""
    sh = np.atleast_2d(np.asarray(sh, np.float64))
    c, s = np.cos(sh[:, 2]), np.sin(sh[:, 2])
    R = np.stack([np.stack([c, -s], -1), np.stack([s, c], -1)], -2)
    D = np.zeros((len(sh), 2, 2))
    D[:, 0, 0] = sh[:, 0] ** 2
    D[:, 1, 1] = sh[:, 1] ** 2
    return R @ D @ np.transpose(R, (0, 2, 1))


def scene(w, h, xy, shape, rgb, k=3.0, mode=oracle.SUM, param=oracle.SCALE_ROT, **kw):
    cfg = oracle.Config(w, h, mode, cutoff_sigma=k, param=param)
    return oracle.Scene(cfg, np.asarray(xy, np.float32).reshape(-1, 2),
                        np.asarray(shape, np.float32).reshape(-1, 3),
                        np.asarray(rgb, np.float32).reshape(-1, 3), **kw)


def scene_of(wl, **kw):
    cfg = oracle.Config(wl.width, wl.height, wl.mode, param=wl.param, **kw)
    return oracle.Scene(cfg, wl.xy, wl.chol, wl.rgb, wl.depth, wl.opacity, wl.background)


def test_fp32_sincos_accuracy():
    """The FP32 sin/cos of the mask data against libm in double: within
    4e-7 absolute for |theta| <= 1000 (a few FP32 ulp of 1), s^2 + c^2 = 1
    to 1e-6, exact at 0, and the quadrant signs right."""
    rng = np.random.default_rng(1)
    th = np.concatenate([np.linspace(-10, 10, 20001), rng.uniform(-1000, 1000, 20000),
                         np.array([0.0, np.pi / 2, np.pi, -np.pi, 3 * np.pi / 2])]).astype(np.float32)
    sn, cs = oracle.sincos_f32(th)
    t64 = th.astype(np.float64)
    assert np.abs(sn - np.sin(t64)).max() <= 4e-7
    assert np.abs(cs - np.cos(t64)).max() <= 4e-7
    assert np.abs(sn.astype(np.float64) ** 2 + cs.astype(np.float64) ** 2 - 1).max() <= 1e-6
    z_s, z_c = oracle.sincos_f32(np.zeros(1, np.float32))
    assert z_s[0] == 0.0 and z_c[0] == 1.0


def test_large_angles_are_culled():
    s = scene(32, 32, [[16, 16], [16, 16]], [[3, 2, 65536.0], [3, 2, 65537.0]], [[1, 1, 1]] * 2)
    assert list(s.proj.count > 0) == [True, False]


def test_single_gaussian_matches_library_density():
    """Every pixel of a rotated anisotropic Gaussian against scipy's density
    of Sigma (numpy, from the FP32 parameters) scaled to a unit peak; pixels
    outside q <= 9 are zero."""
    rng = np.random.default_rng(17)
    for trial in range(20):
        sh = np.array([rng.uniform(0.6, 4.0), rng.uniform(0.6, 4.0), rng.uniform(-4, 4)],
                      np.float32)
        mu = rng.uniform(8, 24, 2)
        s = scene(32, 32, mu, sh, [1.0, 0.5, 0.25])
        img = s.render()["image"]
        Sigma = sigma_of(sh.astype(np.float64))[0]
        mvn = multivariate_normal(mean=s.xy_f[0].astype(np.float64), cov=Sigma)
        yy, xx = np.mgrid[0:32, 0:32]
        pts = np.stack([xx.ravel() + 0.5, yy.ravel() + 0.5], 1)
        dens = mvn.pdf(pts).reshape(32, 32) * 2 * math.pi * math.sqrt(np.linalg.det(Sigma))
        d = pts - s.xy_f[0].astype(np.float64)
        q = np.einsum("ni,ij,nj->n", d, np.linalg.inv(Sigma), d).reshape(32, 32)
        inside = img[0] > 0
        assert np.all(inside[q < 9 * (1 - 1e-5)]), trial
        assert not np.any(inside[q > 9 * (1 + 1e-5)]), trial
        np.testing.assert_allclose(img[0][inside], dens[inside], rtol=1e-9, atol=0)
        np.testing.assert_allclose(img[2][inside], 0.25 * dens[inside], rtol=1e-9, atol=0)


def test_inverse_covariance_fp32():
    """FP32 (A, B, C) times Sigma (numpy, double) is the identity to FP32
    rounding."""
    wl = synth.random_scene(64, 64, 500, seed=23, diag=(0.3, 6.0), param=synth.SCALE_ROT)
    s = scene_of(wl)
    Sigma = sigma_of(wl.chol)
    A, B, Cc = s.proj.conic.astype(np.float64).T
    Q = np.stack([np.stack([A, B], -1), np.stack([B, Cc], -1)], -2)
    err = np.abs(Q @ Sigma - np.eye(2)).max(axis=(1, 2))
    assert np.all(err <= 1e-6 * np.linalg.cond(Sigma))


def test_pixel_box_is_the_ellipse_box():
    """Box ends recomputed in double from Sigma_xx, Sigma_yy (numpy), except
    where a double end lies within 1e-4 of an integer."""
    wl = synth.random_scene(100, 70, 3000, seed=29, diag=(0.2, 6.0), margin=15,
                            param=synth.SCALE_ROT)
    s = scene_of(wl)
    Sg = sigma_of(wl.chol)
    mx, my = wl.xy[:, 0].astype(np.float64), wl.xy[:, 1].astype(np.float64)
    rx, ry = 3 * np.sqrt(Sg[:, 0, 0]), 3 * np.sqrt(Sg[:, 1, 1])
    lo_x, hi_x, lo_y, hi_y = mx - rx - 0.5, mx + rx - 0.5, my - ry - 0.5, my + ry - 0.5
    x0, x1, y0, y1 = np.ceil(lo_x), np.floor(hi_x), np.ceil(lo_y), np.floor(hi_y)
    nonempty = (x0 <= x1) & (y0 <= y1) & (x0 <= 99) & (x1 >= 0) & (y0 <= 69) & (y1 >= 0)
    near = lambda v: np.abs(v - np.round(v)) < 1e-4
    ok = ~(near(lo_x) | near(hi_x) | near(lo_y) | near(hi_y))
    valid = s.proj.count > 0
    assert np.array_equal(valid[ok], nonempty[ok])
    m = ok & nonempty
    bb = s.proj.aabb
    assert np.array_equal(bb[m, 0], np.maximum(x0[m], 0))
    assert np.array_equal(bb[m, 2], np.minimum(x1[m], 99))
    assert np.array_equal(bb[m, 1], np.maximum(y0[m], 0))
    assert np.array_equal(bb[m, 3], np.minimum(y1[m], 69))


def test_zero_rotation_equals_cholesky():
    """theta = 0: Sigma = diag(s_x^2, s_y^2) = L L^T with L = [[s_x, 0],
    [0, s_y]]; both paths give the same FP32 conic, pixel box and image."""
    rng = np.random.default_rng(3)
    n = 200
    xy = rng.uniform(0, 48, (n, 2)).astype(np.float32)
    sc = rng.uniform(0.4, 5.0, (n, 2)).astype(np.float32)
    rgb = rng.uniform(0, 1, (n, 3)).astype(np.float32)
    sr = np.stack([sc[:, 0], sc[:, 1], np.zeros(n, np.float32)], 1)
    ch = np.stack([sc[:, 0], np.zeros(n, np.float32), sc[:, 1]], 1)
    a = scene(48, 40, xy, sr, rgb)
    b = scene(48, 40, xy, ch, rgb, param=oracle.CHOLESKY)
    assert np.array_equal(a.proj.conic, b.proj.conic)  # -0 == +0 for the zero B
    assert np.array_equal(a.proj.aabb, b.proj.aabb)
    np.testing.assert_allclose(a.render()["image"], b.render()["image"], rtol=1e-13, atol=1e-15)


def test_symmetries():
    """(s_y, s_x, theta + pi/2) is the same covariance as (s_x, s_y, theta);
    the sign of a scale does not matter (bit for bit)."""
    rng = np.random.default_rng(5)
    n = 100
    xy = rng.uniform(8, 56, (n, 2)).astype(np.float32)
    sh = synth.scale_rot_uniform(n, (1.0, 4.0), rng)
    sh[:, :2] = np.abs(sh[:, :2])
    rgb = rng.uniform(0, 1, (n, 3)).astype(np.float32)
    quarter = np.stack([sh[:, 1], sh[:, 0], sh[:, 2] + np.float32(np.pi / 2)], 1)
    # a wide cutoff keeps the FP32 mask edge where the weight is ~e^-200
    a = scene(64, 64, xy, sh, rgb, k=20.0).render()["image"]
    b = scene(64, 64, xy, quarter, rgb, k=20.0).render()["image"]
    np.testing.assert_allclose(a, b, rtol=1e-5, atol=1e-9)
    flipped = sh * np.array([-1.0, 1.0, 1.0], np.float32)
    c = scene(64, 64, xy, flipped, rgb).render()["image"]
    d = scene(64, 64, xy, sh, rgb).render()["image"]
    assert np.array_equal(c, d)


def test_same_covariance_as_cholesky_factor():
    """Any (s_x, s_y, theta) against the Cholesky factor of the same Sigma
    (numpy, double, then FP32): images agree to the FP32 rounding of the
    parameters (wide cutoff, so that the two FP32 masks agree)."""
    rng = np.random.default_rng(9)
    n = 150
    xy = rng.uniform(8, 56, (n, 2)).astype(np.float32)
    sh = synth.scale_rot_uniform(n, (0.8, 4.0), rng)
    rgb = rng.uniform(0, 1, (n, 3)).astype(np.float32)
    L = np.linalg.cholesky(sigma_of(sh.astype(np.float64)))
    ch = np.stack([L[:, 0, 0], L[:, 1, 0], L[:, 1, 1]], 1).astype(np.float32)
    a = scene(64, 64, xy, sh, rgb, k=20.0).render()["image"]
    b = scene(64, 64, xy, ch, rgb, k=20.0, param=oracle.CHOLESKY).render()["image"]
    np.testing.assert_allclose(a, b, rtol=2e-5, atol=1e-9)


def test_sum_gradients_by_central_differences():
    wl = synth.random_scene(40, 32, 60, seed=47, diag=(0.8, 4.0), param=synth.SCALE_ROT)
    s = scene_of(wl)
    _fd_check(s, wl.target.astype(np.float64), ["xy", "chol", "rgb"])


def test_composite_gradients_by_central_differences():
    wl = synth.random_scene(40, 32, 60, seed=53, mode=oracle.COMPOSITE, diag=(0.8, 4.0),
                            param=synth.SCALE_ROT)
    s = scene_of(wl)
    _fd_check(s, wl.target.astype(np.float64), ["xy", "chol", "rgb", "opacity", "bg"])


@pytest.mark.parametrize("mode", [oracle.SUM, oracle.COMPOSITE])
def test_tiled_equals_brute_force(mode):
    wl = synth.random_scene(40, 33, 64, seed=59, mode=mode, diag=(0.5, 5.0), param=synth.SCALE_ROT)
    s = scene_of(wl)
    tiled = s.render()["image"]
    brute = s.render_brute()["image"]
    np.testing.assert_allclose(tiled, brute, rtol=1e-12, atol=1e-12)
