"""The oracle's OpenMP timing driver (libgs2d_oracle_omp.so) computes what the
plain oracle computes: the same per-pixel functions with tile rows spread
over threads, so the image and counts are identical and the gradients agree
to the rounding of the double sums' order (CPU only)."""
import numpy as np
import pytest

import oracle
from raster_gaussian_02_b300 import synth


@pytest.mark.parametrize("mode", [oracle.SUM, oracle.COMPOSITE])
@pytest.mark.parametrize("threads", [1, 3, 8])
def test_omp_driver_matches_the_oracle(mode, threads):
    wl = synth.random_scene(120, 90, 800, seed=91 + mode, mode=mode, margin=4)
    cfg = oracle.Config(wl.width, wl.height, mode)
    assert oracle.omp_threads(threads) == threads
    s = oracle.Scene(cfg, wl.xy, wl.chol, wl.rgb, wl.depth, wl.opacity, wl.background)
    a, b = s.render(), s.render(omp=True)
    for k in ("image", "t_final", "last", "margin"):
        np.testing.assert_array_equal(a[k], b[k])
    assert a["masked"] == b["masked"] > 0
    dimg = synth.d_image(wl.height, wl.width, seed=3)
    ga, gb = s.render_bwd(dimg), s.render_bwd(dimg, omp=True)
    for k in ("xy", "chol", "rgb", "opacity", "background", "conic", "xy_abs"):
        scale = np.abs(ga[k]).max(initial=0.0)
        np.testing.assert_allclose(gb[k], ga[k], rtol=0, atol=1e-12 * max(scale, 1e-300))
    oracle.omp_threads(0)
