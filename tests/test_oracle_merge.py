"""Pins of the oracle's moment-matching merge (CPU only).

Pinned by: identical twins merging into one Gaussian of twice the colour
with the image unchanged; the mass, centroid and second moments of the
rendered image (lattice sums at a wide cutoff) preserved by a merge; the
per-channel masses preserved for coloured pairs; every merged pair being a
mutual nearest-neighbour pair under the stated cost (brute force over the
candidate lists); the merge count; both parameterizations giving the same
merged covariance; pass-through of culled Gaussians and of max_merges = 0.
The pairing cost itself is pinned by its closed forms (isotropic and
axis-aligned pairs, a rotated pair along and across its axes) and by
double-precision linear algebra on random pairs.
"""
import numpy as np
import pytest

import oracle
from raster_gaussian_02_b300 import synth


def render(cfg, xy, shape, rgb):
    return oracle.Scene(cfg, xy, shape, rgb).render()["image"]


def moments(img):
    """Mass, centroid and central second moments of one channel of an image
    (lattice sums at the pixel centres)."""
    h, w = img.shape
    yy, xx = np.mgrid[0:h, 0:w] + 0.5
    m = img.sum()
    cx, cy = (img * xx).sum() / m, (img * yy).sum() / m
    sxx = (img * (xx - cx) ** 2).sum() / m
    sxy = (img * (xx - cx) * (yy - cy)).sum() / m
    syy = (img * (yy - cy) ** 2).sum() / m
    return np.array([m, cx, cy, sxx, sxy, syy])


def test_identical_twins():
    cfg = oracle.Config(64, 64)
    xy = np.array([[30.3, 31.7], [30.3, 31.7], [10.0, 50.0]], np.float32)
    sh = np.array([[2.0, 0.7, 1.5], [2.0, 0.7, 1.5], [1.0, 0.0, 1.0]], np.float32)
    rgb = np.array([[0.2, 0.4, 0.6], [0.2, 0.4, 0.6], [1, 1, 1]], np.float32)
    oxy, osh, orgb, m = oracle.merge(cfg, xy, sh, rgb, 10)
    assert m == 1
    np.testing.assert_array_equal(oxy[0], xy[0])
    np.testing.assert_allclose(osh[0], sh[0], rtol=1e-6)
    np.testing.assert_allclose(orgb[0], 2 * rgb[0], rtol=1e-6)
    np.testing.assert_allclose(render(cfg, oxy, osh, orgb), render(cfg, xy, sh, rgb), rtol=1e-5, atol=1e-9)


@pytest.mark.parametrize("param", [oracle.CHOLESKY, oracle.SCALE_ROT])
def test_moments_of_the_image_are_kept(param):
    """A gray pair far from the borders, wide cutoff: the merged Gaussian's
    image has the pair's mass, centroid and second moments."""
    cfg = oracle.Config(96, 96, cutoff_sigma=20.0, param=param)
    xy = np.array([[46.0, 47.5], [49.5, 45.0]], np.float32)
    if param == oracle.SCALE_ROT:
        sh = np.array([[3.0, 1.8, 0.4], [2.2, 2.9, -1.1]], np.float32)
    else:
        sh = np.array([[3.0, 0.8, 1.7], [2.2, -0.9, 2.6]], np.float32)
    rgb = np.array([[0.7, 0.7, 0.7], [0.3, 0.3, 0.3]], np.float32)
    oxy, osh, orgb, m = oracle.merge(cfg, xy, sh, rgb, 1)
    assert m == 1
    a = moments(render(cfg, xy, sh, rgb)[0])
    b = moments(render(cfg, oxy, osh, orgb)[0])
    np.testing.assert_allclose(b, a, rtol=2e-5, atol=2e-5)


def test_channel_masses_are_kept():
    cfg = oracle.Config(96, 96, cutoff_sigma=20.0)
    xy = np.array([[46.0, 47.5], [49.5, 45.0]], np.float32)
    sh = np.array([[3.0, 0.8, 1.7], [2.2, -0.9, 2.6]], np.float32)
    rgb = np.array([[0.9, 0.1, 0.5], [0.2, 0.8, 0.5]], np.float32)
    oxy, osh, orgb, m = oracle.merge(cfg, xy, sh, rgb, 1)
    np.testing.assert_allclose(render(cfg, oxy, osh, orgb).sum((1, 2)),
                               render(cfg, xy, sh, rgb).sum((1, 2)), rtol=1e-5)


def sigma(param, sh):
    sh = sh.astype(np.float64)
    if param == oracle.SCALE_ROT:
        sn, cs = oracle.sincos_f32(sh[:, 2].astype(np.float32))
        c, s = cs.astype(np.float64), sn.astype(np.float64)
        x2, y2 = sh[:, 0] ** 2, sh[:, 1] ** 2
        return np.stack([c * c * x2 + s * s * y2, c * s * (x2 - y2), s * s * x2 + c * c * y2], 1)
    a, b, c = sh.T
    return np.stack([a * a, a * b, b * b + c * c], 1)


def test_merge_cost_closed_forms():
    """The pairing cost d^T M^-1 d with M the mean of the two covariances,
    against its closed forms: two isotropic Gaussians of scale s at distance
    d give d^2/s^2 in any direction; scales s1 and s2 give 2 d^2/(s1^2 + s2^2);
    two axis-aligned Gaussians diag(sx^2, sy^2) give dx^2/sx^2 + dy^2/sy^2;
    a rotated pair gives d^2/sx^2 along its major axis and d^2/sy^2 across
    it; coincident means cost 0."""
    ch = oracle.Config(64, 64)
    cases = []  # (xa, shape a, xb, shape b, expected)
    for s, d, ang in ((1.0, 2.0, 0.0), (2.5, 3.0, 0.7), (0.8, 0.5, 2.0), (4.0, 10.0, -1.2)):
        dx, dy = d * np.cos(ang), d * np.sin(ang)
        cases.append(((10.0, 20.0), (s, 0.0, s), (10.0 + dx, 20.0 + dy), (s, 0.0, s), d * d / (s * s)))
    for s1, s2, d in ((1.0, 3.0, 2.0), (0.6, 2.2, 1.3)):
        cases.append(((5.0, 5.0), (s1, 0.0, s1), (5.0, 5.0 + d), (s2, 0.0, s2),
                      2 * d * d / (s1 * s1 + s2 * s2)))
    for sx, sy, dx, dy in ((2.0, 0.5, 1.5, 0.25), (1.2, 3.1, -2.0, 4.0)):
        cases.append(((30.0, 30.0), (sx, 0.0, sy), (30.0 + dx, 30.0 + dy), (sx, 0.0, sy),
                      dx * dx / (sx * sx) + dy * dy / (sy * sy)))
    cases.append(((7.0, 9.0), (1.5, 0.4, 2.0), (7.0, 9.0), (0.9, -0.3, 1.1), 0.0))
    xa, sa, xb, sb, want = (np.array(v, np.float64) for v in zip(*cases))
    got = oracle.merge_cost(ch, xa, sa, xb, sb).astype(np.float64)
    np.testing.assert_allclose(got, want, rtol=2e-6, atol=0)
    # rotated pair (scale-rotation shapes): along the major axis, then across it
    sr = oracle.Config(64, 64, param=oracle.SCALE_ROT)
    th, sx, sy, d = 0.6, 3.0, 1.0, 2.0
    sn, cs = (float(v[0]) for v in oracle.sincos_f32(np.array([th], np.float32)))
    xa = np.array([[20.0, 20.0], [20.0, 20.0]])
    xb = xa + d * np.array([[cs, sn], [-sn, cs]])
    shp = np.array([[sx, sy, th], [sx, sy, th]])
    got = oracle.merge_cost(sr, xa, shp, xb, shp).astype(np.float64)
    np.testing.assert_allclose(got, [d * d / (sx * sx), d * d / (sy * sy)], rtol=1e-5)


def test_merge_cost_against_linear_algebra():
    """Random pairs: the FP32 cost against d^T M^-1 d solved in double by
    numpy, M = (Sigma_a + Sigma_b) / 2 with Sigma = L L^T (Cholesky) or
    R diag(s^2) R^T (scale-rotation), within FP32 rounding of the inputs."""
    rng = np.random.default_rng(12)
    m = 400
    for param in (oracle.CHOLESKY, oracle.SCALE_ROT):
        cfg = oracle.Config(64, 64, param=param)
        xa = rng.uniform(0, 64, (m, 2))
        xb = xa + rng.normal(0, 3, (m, 2))
        if param == oracle.CHOLESKY:
            sa = np.stack([rng.uniform(0.5, 3, m), rng.normal(0, 0.5, m), rng.uniform(0.5, 3, m)], 1)
            sb = np.stack([rng.uniform(0.5, 3, m), rng.normal(0, 0.5, m), rng.uniform(0.5, 3, m)], 1)
        else:
            sa = np.stack([rng.uniform(0.5, 3, m), rng.uniform(0.5, 3, m), rng.uniform(-3, 3, m)], 1)
            sb = np.stack([rng.uniform(0.5, 3, m), rng.uniform(0.5, 3, m), rng.uniform(-3, 3, m)], 1)
        sa, sb = sa.astype(np.float32), sb.astype(np.float32)
        got = oracle.merge_cost(cfg, xa, sa, xb, sb).astype(np.float64)

        def cov(sh):
            sh = sh.astype(np.float64)
            if param == oracle.CHOLESKY:
                L = np.zeros((m, 2, 2))
                L[:, 0, 0], L[:, 1, 0], L[:, 1, 1] = sh[:, 0], sh[:, 1], sh[:, 2]
                return L @ np.transpose(L, (0, 2, 1))
            c, s = np.cos(sh[:, 2]), np.sin(sh[:, 2])
            R = np.stack([np.stack([c, -s], -1), np.stack([s, c], -1)], -2)
            D = np.zeros((m, 2, 2))
            D[:, 0, 0], D[:, 1, 1] = sh[:, 0] ** 2, sh[:, 1] ** 2
            return R @ D @ np.transpose(R, (0, 2, 1))
        M = 0.5 * (cov(sa) + cov(sb))
        d = (xa.astype(np.float32) - xb.astype(np.float32)).astype(np.float64)
        want = np.einsum("ki,ki->k", d, np.linalg.solve(M, d[..., None])[..., 0])
        np.testing.assert_allclose(got, want, rtol=2e-4, atol=1e-5)


@pytest.mark.parametrize("param", [oracle.CHOLESKY, oracle.SCALE_ROT])
def test_pairs_are_mutual_nearest_neighbours(param):
    wl = synth.random_scene(64, 48, 500, seed=131, diag=(0.5, 4.0), margin=3, param=param)
    cfg = oracle.Config(64, 48, param=param)
    s = oracle.Scene(cfg, wl.xy, wl.chol, wl.rgb)
    valid = s.proj.count > 0

    def cost(i, j):
        # the pairing cost, pinned by test_merge_cost_closed_forms
        return float(oracle.merge_cost(cfg, wl.xy[[i]], wl.chol[[i]], wl.xy[[j]], wl.chol[[j]])[0])

    nn = np.full(wl.n, -1)
    for i in np.nonzero(valid)[0]:
        px = min(max(int(np.floor(wl.xy[i, 0])), 0), 63)
        py = min(max(int(np.floor(wl.xy[i, 1])), 0), 47)
        t = (py // 16) * cfg.tiles_x + px // 16
        cands = [j for j in s.sorted_gid[s.ranges[t, 0]:s.ranges[t, 1]] if j != i]
        if cands:
            cs = [(cost(i, j), j) for j in cands]
            nn[i] = min(cs)[1]
    mutual = [i for i in range(wl.n) if nn[i] > i and nn[nn[i]] == i]
    for k in (5, len(mutual) // 2, 10 ** 6):
        _, _, _, m, partner = oracle.merge(cfg, wl.xy, wl.chol, wl.rgb, k, with_partners=True)
        assert m == min(k, len(mutual))
        got = np.nonzero(partner >= 0)[0]
        assert set(got) <= set(mutual)
        assert all(partner[i] == nn[i] for i in got)
    assert len(mutual) > 20


def test_parameterizations_merge_to_the_same_covariance():
    rng = np.random.default_rng(4)
    n = 300
    xy = rng.uniform(4, 60, (n, 2)).astype(np.float32)
    sr = synth.scale_rot_uniform(n, (0.8, 3.5), rng)
    S = sigma(oracle.SCALE_ROT, sr)
    L = np.linalg.cholesky(np.stack([np.stack([S[:, 0], S[:, 1]], -1), np.stack([S[:, 1], S[:, 2]], -1)], -2))
    ch = np.stack([L[:, 0, 0], L[:, 1, 0], L[:, 1, 1]], 1).astype(np.float32)
    rgb = rng.uniform(0, 1, (n, 3)).astype(np.float32)
    a = oracle.merge(oracle.Config(64, 64, param=oracle.SCALE_ROT), xy, sr, rgb, 60, with_partners=True)
    b = oracle.merge(oracle.Config(64, 64, param=oracle.CHOLESKY), xy, ch, rgb, 60, with_partners=True)
    same = np.nonzero((a[4] >= 0) & (a[4] == b[4]))[0]
    assert len(same) > 30
    # positions of the merged Gaussians in the outputs: index minus the drops before it
    def slot(partner, i):
        drops = np.zeros(len(partner), bool)
        drops[partner[partner >= 0]] = True
        return i - drops[:i].sum()
    for i in same[:30]:
        sa = sigma(oracle.SCALE_ROT, a[1][slot(a[4], i)][None])[0]
        sb = sigma(oracle.CHOLESKY, b[1][slot(b[4], i)][None])[0]
        np.testing.assert_allclose(sa, sb, rtol=1e-4, atol=1e-4 * np.abs(sb).max())


def test_culled_pass_through_and_zero_merges():
    wl = synth.random_scene(48, 40, 200, seed=137, diag=(0.5, 3.0))
    wl.chol[:10, 0] = 0.0  # culled
    cfg = oracle.Config(48, 40)
    oxy, osh, orgb, m = oracle.merge(cfg, wl.xy, wl.chol, wl.rgb, 0)
    assert m == 0
    np.testing.assert_array_equal(oxy, wl.xy)
    np.testing.assert_array_equal(osh, wl.chol)
    oxy, osh, orgb, m, partner = oracle.merge(cfg, wl.xy, wl.chol, wl.rgb, 1000, with_partners=True)
    assert np.all(partner[:10] == -1) and not np.isin(np.arange(10), partner).any()
    assert m > 0
    np.testing.assert_array_equal(osh[:10], wl.chol[:10])
