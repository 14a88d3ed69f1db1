"""Pins of the CPU oracle to things other than itself (CPU only).

The pages print no worked example of a render or a gradient, so the oracle
is tied to: hand-derived closed forms (tests/golden), an independent library
evaluation of the Gaussian (scipy's multivariate normal density and numpy's
matrix inverse), the lattice-sum identity for the integral of a Gaussian,
brute force without tiles, invariants of the sum form, the algebra of
front-to-back compositing, and central finite differences for every
gradient.  Each is chosen so that a plausible slip (a dropped factor 1/2, a
wrong sign of the off-diagonal term, a transposed Cholesky factor, a missed
tile, a wrong chain-rule term) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
from scipy.stats import multivariate_normal

import oracle
from raster_gaussian_02_b300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")


def scene_of(wl, **kw):
    cfg = oracle.Config(wl.width, wl.height, wl.mode, **kw)
    return oracle.Scene(cfg, wl.xy, wl.chol, wl.rgb, wl.depth, wl.opacity, wl.background)


def one_gaussian(w, h, xy, chol, rgb, k=3.0):
    cfg = oracle.Config(w, h, oracle.SUM, cutoff_sigma=k)
    return oracle.Scene(cfg, np.array([xy], np.float32), np.array([chol], np.float32),
                        np.array([rgb], np.float32))


# ------------------------------------------------------------ closed forms --

def test_golden_single_gaussian_values():
    gold = json.load(open(GOLDEN))
    for case in gold["single"]:
        s = one_gaussian(case["width"], case["height"], case["xy"], case["chol"], case["rgb"])
        img = s.render()["image"]
        i, j = case["pixel"]
        want = case.get("value_rgb", [case.get("value")] * 3)
        want = np.array(want) * (np.array(case["rgb"]) if "value" in case else 1.0)
        np.testing.assert_allclose(img[:, i, j], want, rtol=1e-15, atol=1e-15, err_msg=case["name"])


def test_golden_composite_values():
    gold = json.load(open(GOLDEN))
    for case in gold["composite"]:
        cfg = oracle.Config(case["width"], case["height"], oracle.COMPOSITE)
        s = oracle.Scene(cfg, case["xy"], case["chol"], case["rgb"], case["depth"],
                         case["opacity"], case["background"])
        out = s.render()
        i, j = case["pixel"]
        np.testing.assert_allclose(out["image"][:, i, j], case["value_rgb"], rtol=1e-15, atol=1e-15,
                                   err_msg=case["name"])
        assert out["t_final"][i, j] == pytest.approx(case["t_final"], rel=1e-15)
        assert out["last"][i, j] == 2


def test_single_gaussian_matches_library_density():
    """Every pixel of a random anisotropic Gaussian against scipy's normal
    density scaled by 2*pi*sqrt(det Sigma) (so that the peak is 1), with
    Sigma = L L^T formed by numpy; pixels outside q <= 9 must be zero."""
    rng = np.random.default_rng(7)
    for trial in range(20):
        a, c = rng.uniform(0.7, 4.0, 2) * rng.choice([-1, 1], 2)
        b = rng.normal(0, 1.5)
        mu = rng.uniform(5, 27, 2)
        L = np.array([[a, 0.0], [b, c]], np.float32).astype(np.float64)
        s = one_gaussian(32, 32, mu, [a, b, c], [1.0, 0.5, 0.25])
        img = s.render()["image"]
        Sigma = L @ L.T
        mvn = multivariate_normal(mean=s.xy_f[0].astype(np.float64), cov=Sigma)
        yy, xx = np.mgrid[0:32, 0:32]
        pts = np.stack([xx.ravel() + 0.5, yy.ravel() + 0.5], 1)
        dens = mvn.pdf(pts).reshape(32, 32) * 2 * math.pi * math.sqrt(np.linalg.det(Sigma))
        d = pts - s.xy_f[0].astype(np.float64)
        q = np.einsum("ni,ij,nj->n", d, np.linalg.inv(Sigma), d).reshape(32, 32)
        inside = img[0] > 0
        clear_in = q < 9 * (1 - 1e-6)
        clear_out = q > 9 * (1 + 1e-6)
        assert np.all(inside[clear_in]), trial
        assert not np.any(inside[clear_out]), trial
        np.testing.assert_allclose(img[0][inside], dens[inside], rtol=1e-9, atol=0)
        np.testing.assert_allclose(img[1][inside], 0.5 * dens[inside], rtol=1e-9, atol=0)
        np.testing.assert_allclose(img[2][inside], 0.25 * dens[inside], rtol=1e-9, atol=0)


def test_integral_equals_2pi_det_L():
    """With a wide cutoff (k=20) and sigma >= 1, the pixel-lattice sum of
    exp(-q/2) equals the integral 2*pi*|a c| up to terms of order
    exp(-2 pi^2 sigma_min^2) (Poisson summation), far below 1e-6."""
    rng = np.random.default_rng(11)
    for _ in range(8):
        a, c = rng.uniform(1.2, 3.0, 2)
        b = rng.normal(0, 0.7)
        mu = rng.uniform(60, 68, 2)
        s = one_gaussian(128, 128, mu, [a, b, c], [1.0, 1.0, 1.0], k=20.0)
        total = s.render()["image"][0].sum()
        a32, c32 = np.float32(a), np.float32(c)
        assert total == pytest.approx(2 * math.pi * abs(float(a32) * float(c32)), rel=1e-6)


def test_mass_inside_three_sigma():
    """At k=3 the touched mass approaches (1 - e^-4.5) 2 pi s^2 for an
    isotropic Gaussian; the lattice count of the disc's rim limits the
    agreement to about a percent at s = 6."""
    s_ = 6.0
    s = one_gaussian(64, 64, [32.0, 32.0], [s_, 0.0, s_], [1, 1, 1])
    total = s.render()["image"][0].sum()
    assert total == pytest.approx((1 - math.exp(-4.5)) * 2 * math.pi * s_ * s_, rel=0.02)


def test_inverse_covariance_fp32():
    """The FP32 inverse covariance times Sigma = L L^T (numpy, double) is the
    identity to FP32 rounding."""
    wl = synth.random_scene(64, 64, 500, seed=3, diag=(0.3, 5.0), offdiag_sigma=2.0)
    s = scene_of(wl)
    L = np.zeros((wl.n, 2, 2))
    L[:, 0, 0] = wl.chol[:, 0]
    L[:, 1, 0] = wl.chol[:, 1]
    L[:, 1, 1] = wl.chol[:, 2]
    Sigma = L @ np.transpose(L, (0, 2, 1))
    A, B, Cc = s.proj.conic.astype(np.float64).T
    Q = np.stack([np.stack([A, B], -1), np.stack([B, Cc], -1)], -2)
    I = Q @ Sigma
    cond = np.linalg.cond(Sigma)
    err = np.abs(I - np.eye(2)).max(axis=(1, 2))
    assert np.all(err <= 1e-6 * cond)


def test_isotropic_peak_is_colour():
    for s_ in (0.5, 1.0, 3.7):
        s = one_gaussian(16, 16, [7.5, 9.5], [s_, 0.0, s_], [0.3, 0.6, 0.9])
        img = s.render()["image"]
        np.testing.assert_array_equal(img[:, 9, 7], np.array([0.3, 0.6, 0.9], np.float32))


# --------------------------------------------------------------- the box --

def test_pixel_box_formula():
    """The pixel box is the tight box of the 3-sigma ellipse, clipped to the
    image: its ends are recomputed here in double from Sigma = L L^T; the two
    may differ only where the double end lies within 1e-4 of an integer."""
    wl = synth.random_scene(100, 70, 3000, seed=5, diag=(0.2, 6.0), offdiag_sigma=2.0, margin=15)
    s = scene_of(wl)
    L = wl.chol.astype(np.float64)
    Sxx = L[:, 0] ** 2
    Syy = L[:, 1] ** 2 + L[:, 2] ** 2
    mx, my = wl.xy[:, 0].astype(np.float64), wl.xy[:, 1].astype(np.float64)
    lo_x = mx - 3 * np.sqrt(Sxx) - 0.5
    hi_x = mx + 3 * np.sqrt(Sxx) - 0.5
    lo_y = my - 3 * np.sqrt(Syy) - 0.5
    hi_y = my + 3 * np.sqrt(Syy) - 0.5
    x0, x1 = np.ceil(lo_x), np.floor(hi_x)
    y0, y1 = np.ceil(lo_y), np.floor(hi_y)
    nonempty = (x0 <= x1) & (y0 <= y1) & (x0 <= 99) & (x1 >= 0) & (y0 <= 69) & (y1 >= 0)
    near = lambda v: np.abs(v - np.round(v)) < 1e-4
    amb = near(lo_x) | near(hi_x) | near(lo_y) | near(hi_y)
    ok = ~amb
    valid = s.proj.count > 0
    assert np.array_equal(valid[ok], nonempty[ok])
    m = ok & nonempty
    bb = s.proj.aabb
    assert np.array_equal(bb[m, 0], np.maximum(x0[m], 0))
    assert np.array_equal(bb[m, 1], np.maximum(y0[m], 0))
    assert np.array_equal(bb[m, 2], np.minimum(x1[m], 99))
    assert np.array_equal(bb[m, 3], np.minimum(y1[m], 69))
    assert np.array_equal(s.proj.rect[valid], bb[valid] // 16)
    cnt = (s.proj.rect[:, 2] - s.proj.rect[:, 0] + 1) * (s.proj.rect[:, 3] - s.proj.rect[:, 1] + 1)
    assert np.array_equal(s.proj.count[valid], cnt[valid])


def test_every_touched_pixel_lies_in_box():
    wl = synth.random_scene(48, 40, 400, seed=9, diag=(0.3, 4.0), offdiag_sigma=1.5, margin=5)
    s = scene_of(wl)
    yy, xx = np.mgrid[0:40, 0:48]
    pts = np.stack([xx.ravel() + 0.5, yy.ravel() + 0.5], 1)
    for g in np.nonzero(s.proj.count)[0][:150]:
        L = np.array([[wl.chol[g, 0], 0], [wl.chol[g, 1], wl.chol[g, 2]]], np.float64)
        d = pts - wl.xy[g].astype(np.float64)
        q = np.einsum("ni,ij,nj->n", d, np.linalg.inv(L @ L.T), d)
        inner = q < 9 * (1 - 1e-5)
        bb = s.proj.aabb[g]
        px, py = xx.ravel()[inner], yy.ravel()[inner]
        assert np.all((px >= bb[0]) & (px <= bb[2]) & (py >= bb[1]) & (py <= bb[3]))


# -------------------------------------------------------------- tile lists --

@pytest.mark.parametrize("mode", [oracle.SUM, oracle.COMPOSITE])
def test_tile_lists_by_brute_force(mode):
    """Each tile's list re-derived by testing every Gaussian's pixel box
    against the tile's pixel square; order ascending index (sum) or
    ascending (depth, index) (composite)."""
    wl = synth.random_scene(75, 50, 300, seed=21, mode=mode, diag=(0.5, 8.0), margin=10)
    s = scene_of(wl)
    cfg = s.cfg
    assert s.num_pairs == int(s.proj.count.sum())
    for ty in range(cfg.tiles_y):
        for tx in range(cfg.tiles_x):
            t = ty * cfg.tiles_x + tx
            a, b = s.ranges[t]
            got = s.sorted_gid[a:b]
            X0, X1, Y0, Y1 = 16 * tx, 16 * tx + 15, 16 * ty, 16 * ty + 15
            bb = s.proj.aabb
            hit = (s.proj.count > 0) & (bb[:, 0] <= X1) & (bb[:, 2] >= X0) & (bb[:, 1] <= Y1) & (bb[:, 3] >= Y0)
            want = np.nonzero(hit)[0]
            if mode == oracle.COMPOSITE:
                want = sorted(want, key=lambda g: (wl.depth[g], g))
            assert list(got) == list(want), (tx, ty)
    assert s.ranges[0, 0] == 0 and np.all(s.ranges[1:, 0] == s.ranges[:-1, 1])


# ----------------------------------------------------------- brute force --

@pytest.mark.parametrize("w,h,n", [(8, 8, 5), (17, 13, 24), (40, 33, 64), (64, 64, 64), (1, 1, 3)])
@pytest.mark.parametrize("mode", [oracle.SUM, oracle.COMPOSITE])
def test_tiled_equals_brute_force(w, h, n, mode):
    wl = synth.random_scene(w, h, n, seed=w * 100 + h + n, mode=mode, diag=(0.3, 6.0), margin=4)
    s = scene_of(wl)
    tiled = s.render()
    brute = s.render_brute()
    np.testing.assert_allclose(tiled["image"], brute["image"], rtol=0, atol=1e-12)
    if mode == oracle.COMPOSITE:
        np.testing.assert_allclose(tiled["t_final"], brute["t_final"], rtol=0, atol=1e-12)


def test_sampled_pixels_equal_full_render():
    wl = synth.random_scene(50, 37, 200, seed=4, mode=oracle.COMPOSITE, diag=(0.5, 5.0))
    s = scene_of(wl)
    full = s.render()
    pix = np.random.default_rng(0).choice(50 * 37, 300, replace=False)
    part = s.render_pixels(pix)
    np.testing.assert_array_equal(part["rgb"], full["image"].reshape(3, -1)[:, pix].T)
    np.testing.assert_array_equal(part["last"], full["last"].ravel()[pix])
    np.testing.assert_array_equal(part["t_final"], full["t_final"].ravel()[pix])


# ------------------------------------------------------------- invariants --

def test_sum_is_order_independent():
    wl = synth.random_scene(48, 48, 120, seed=13, diag=(0.5, 5.0))
    s0 = scene_of(wl)
    perm = np.random.default_rng(1).permutation(wl.n)
    wl2 = synth.Workload(wl.name, wl.width, wl.height, wl.mode, wl.xy[perm], wl.chol[perm],
                         wl.rgb[perm], wl.target)
    s1 = scene_of(wl2)
    np.testing.assert_allclose(s0.render()["image"], s1.render()["image"], rtol=0, atol=1e-12)


def test_composite_depends_on_depth_order():
    """Swapping the depths of two overlapping Gaussians changes the
    composite image, exactly as swapping their colours and opacities."""
    xy = np.array([[8.0, 8.0], [9.0, 8.5]], np.float32)
    chol = np.array([[2.0, 0.3, 1.5], [1.5, -0.2, 2.0]], np.float32)
    rgb = np.array([[1, 0, 0], [0, 1, 0]], np.float32)
    op = np.array([0.7, 0.6], np.float32)
    bg = np.array([0.1, 0.2, 0.3], np.float32)
    cfg = oracle.Config(16, 16, oracle.COMPOSITE)
    a = oracle.Scene(cfg, xy, chol, rgb, np.array([0.1, 0.2], np.float32), op, bg).render()["image"]
    b = oracle.Scene(cfg, xy, chol, rgb, np.array([0.2, 0.1], np.float32), op, bg).render()["image"]
    assert np.abs(a - b).max() > 0.05
    c = oracle.Scene(cfg, xy[::-1].copy(), chol[::-1].copy(), rgb[::-1].copy(),
                     np.array([0.1, 0.2], np.float32), op[::-1].copy(), bg).render()["image"]
    np.testing.assert_allclose(b, c, rtol=0, atol=1e-15)


def test_composite_special_cases():
    cfg = oracle.Config(8, 8, oracle.COMPOSITE)
    bg = np.array([0.2, 0.4, 0.6], np.float32)
    xy = np.array([[3.5, 3.5]], np.float32)
    chol = np.array([[1.0, 0.0, 1.0]], np.float32)
    rgb = np.array([[0.9, 0.5, 0.1]], np.float32)
    for o in (0.0, 0.3, 0.99):
        s = oracle.Scene(cfg, xy, chol, rgb, np.array([0.5], np.float32), np.array([o], np.float32), bg)
        out = s.render()
        o64 = float(np.float32(o))
        np.testing.assert_allclose(out["image"][:, 3, 3],
                                   rgb[0].astype(np.float64) * o64 + (1 - o64) * bg.astype(np.float64),
                                   rtol=1e-15, atol=1e-15)
    # a pixel that no Gaussian touches shows the background, T_final = 1
    np.testing.assert_allclose(out["image"][:, 7, 0], bg.astype(np.float64), rtol=0, atol=0)
    assert out["t_final"][7, 0] == 1.0 and out["last"][7, 0] == 0


def test_composite_early_termination():
    """Three nearly opaque Gaussians on one pixel centre: after two the
    transmittance is about 1e-8 < t_min, so the third is never processed."""
    cfg = oracle.Config(8, 8, oracle.COMPOSITE, t_min=1e-4)
    n = 3
    xy = np.tile(np.array([[4.5, 4.5]], np.float32), (n, 1))
    chol = np.tile(np.array([[1.0, 0.0, 1.0]], np.float32), (n, 1))
    rgb = np.array([[1, 0, 0], [0, 1, 0], [0, 0, 1]], np.float32)
    op = np.full(n, 0.9999, np.float32)
    s = oracle.Scene(cfg, xy, chol, rgb, np.array([0.1, 0.2, 0.3], np.float32), op,
                     np.zeros(3, np.float32))
    out = s.render()
    o = float(np.float32(0.9999))
    assert out["last"][4, 4] == 2
    assert out["t_final"][4, 4] == pytest.approx((1 - o) ** 2, rel=1e-12)
    np.testing.assert_allclose(out["image"][:, 4, 4], [o, o * (1 - o), 0.0], rtol=1e-12, atol=0)


def test_culling():
    """Non-finite parameters, a zero diagonal, a Gaussian entirely off the
    image and (composite) an opacity outside [0,1) are culled: no tiles,
    no pixels, zero gradient."""
    xy = np.array([[4, 4], [np.nan, 3], [4, 4], [4, 4], [-50, 4], [4, 4], [4, 4]], np.float32)
    chol = np.array([[1, 0, 1], [1, 0, 1], [0, 0.5, 1], [1, 0.5, 0], [1, 0, 1], [1, np.inf, 1],
                     [1, 0, 1]], np.float32)
    rgb = np.ones((7, 3), np.float32)
    depth = np.linspace(0, 1, 7).astype(np.float32)
    op = np.array([0.5, 0.5, 0.5, 0.5, 0.5, 0.5, 1.0], np.float32)
    for mode in (oracle.SUM, oracle.COMPOSITE):
        cfg = oracle.Config(8, 8, mode)
        s = oracle.Scene(cfg, xy, chol, rgb, depth, op, np.zeros(3, np.float32))
        want_valid = [True, False, False, False, False, False, mode == oracle.SUM]
        assert list(s.proj.count > 0) == want_valid
        g = s.render_bwd(np.ones((3, 8, 8)))
        assert np.all(g["xy"][~np.array(want_valid)] == 0)
        assert np.all(g["chol"][~np.array(want_valid)] == 0)


# -------------------------------------------------------------- gradients --

def _flat_loss(s, target):
    out = s.render()
    loss, _ = oracle.loss_l2(out["image"], target)
    return loss


def _fd_check(s, target, names, h_rel=1e-5, rtol=1e-6, n_probe=40, seed=0):
    out = s.render()
    loss, dimg = oracle.loss_l2(out["image"], target)
    g = s.render_bwd(dimg)
    rng = np.random.default_rng(seed)
    valid = np.nonzero(s.proj.count > 0)[0]
    last0 = out["last"].copy()
    for name in names:
        arr = getattr(s, name)
        grad = g["background" if name == "bg" else name]
        scale = np.abs(grad).max()
        idxs = [()] if name == "bg" else None
        probes = range(3) if name == "bg" else rng.choice(valid, min(n_probe, len(valid)), replace=False)
        for p in probes:
            cols = [p] if arr.ndim == 1 else [(p, d) for d in range(arr.shape[1])]
            for ix in cols:
                base = arr[ix]
                h = h_rel * max(1.0, abs(base))
                arr[ix] = base + h
                lp = _flat_loss(s, target)
                arr[ix] = base - h
                lm = _flat_loss(s, target)
                arr[ix] = base
                fd = (lp - lm) / (2 * h)
                assert abs(fd - grad[ix]) <= rtol * scale + 1e-14, (name, ix, fd, grad[ix], scale)
    # the early-termination decisions did not move under the perturbations
    assert np.array_equal(s.render()["last"], last0)


def test_sum_gradients_by_central_differences():
    wl = synth.random_scene(40, 32, 60, seed=31, diag=(0.8, 4.0))
    s = scene_of(wl)
    _fd_check(s, wl.target.astype(np.float64), ["xy", "chol", "rgb"])


def test_composite_gradients_by_central_differences():
    wl = synth.random_scene(40, 32, 60, seed=37, mode=oracle.COMPOSITE, diag=(0.8, 4.0))
    s = scene_of(wl)
    _fd_check(s, wl.target.astype(np.float64), ["xy", "chol", "rgb", "opacity", "bg"])


def test_composite_gradients_with_termination():
    """Dense opaque stack so that many pixels stop early; the decisions are
    held fixed and the gradients still match central differences."""
    wl = synth.random_scene(24, 24, 120, seed=41, mode=oracle.COMPOSITE, diag=(2.0, 5.0))
    wl.opacity = np.full(wl.n, 0.97, np.float32)
    s = scene_of(wl)
    out = s.render()
    assert (out["t_final"] < 1e-4).mean() > 0.2
    _fd_check(s, wl.target.astype(np.float64), ["xy", "chol", "rgb", "opacity", "bg"], n_probe=25)


def test_loss_gradient_by_central_differences():
    rng = np.random.default_rng(2)
    img = rng.normal(size=(3, 5, 7))
    tgt = rng.normal(size=(3, 5, 7))
    loss, d = oracle.loss_l2(img, tgt)
    assert loss == pytest.approx(((img - tgt) ** 2).mean(), rel=1e-14)
    for ix in [(0, 0, 0), (1, 3, 4), (2, 4, 6)]:
        h = 1e-6
        e = img.copy(); e[ix] += h
        lp, _ = oracle.loss_l2(e, tgt)
        e[ix] -= 2 * h
        lm, _ = oracle.loss_l2(e, tgt)
        assert (lp - lm) / (2 * h) == pytest.approx(d[ix], rel=1e-7)


@pytest.mark.parametrize("mode", [oracle.SUM, oracle.COMPOSITE])
def test_two_backward_traversals_agree(mode):
    """Pixel-major and Gaussian-major traversals of the backward give the
    same gradients."""
    wl = synth.random_scene(45, 38, 150, seed=43, mode=mode, diag=(0.5, 5.0))
    s = scene_of(wl)
    dimg = synth.d_image(38, 45, seed=5).astype(np.float64)
    full = s.render_bwd(dimg)
    gids = np.arange(wl.n, dtype=np.int32)
    part = s.render_bwd_gaussians(dimg, gids)
    for k in ("xy", "chol", "rgb", "opacity"):
        np.testing.assert_allclose(part[k], full[k], rtol=1e-10, atol=1e-12 * np.abs(full[k]).max())
