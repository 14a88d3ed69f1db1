"""absgrad (per-pixel absolute mean-gradient sums) on the GPU against the
CPU oracle, through the C ABI (needs a B300).  Asking for it leaves every
other output bit-identical."""
import numpy as np
import pytest

import oracle
from raster_gaussian_02_b300 import synth

from gpu_common import _gaussians_touching, check_grads, check_image, gpu_run, oracle_scene
from test_gpu_fused import fused_run

pytestmark = pytest.mark.gpu


def absgrad_parity(wl, fused=False):
    comp = wl.mode == synth.COMPOSITE
    plain = gpu_run(wl)
    g = fused_run(wl, absgrad=True) if fused else gpu_run(wl, absgrad=True)
    for k, v in plain["grads"].items():
        assert np.array_equal(g["grads"][k], v), k
    s = oracle_scene(wl)
    ok = check_image(plain, s.render(), comp)
    _, dimg = oracle.loss_l2(g["image"] if fused else plain["image"], wl.target)
    ref = s.render_bwd(plain["d_image"].astype(np.float64) if not fused else dimg)
    mask = None
    if comp:
        mask = np.ones(wl.n, bool)
        mask[_gaussians_touching(s, ~ok)] = False
    check_grads(g["grads"], ref, ["xy_abs"], mask=mask)
    assert np.all(g["grads"]["xy_abs"][s.proj.count == 0] == 0)
    assert np.all(g["grads"]["xy_abs"] >= np.abs(g["grads"]["xy"]) * (1 - 1e-5) - 1e-12)


@pytest.mark.parametrize("w,h,n,seed", [(1, 1, 3, 1), (17, 13, 40, 2), (250, 130, 3000, 5)])
@pytest.mark.parametrize("mode", [synth.SUM, synth.COMPOSITE])
def test_random_ragged(w, h, n, seed, mode):
    absgrad_parity(synth.random_scene(w, h, n, seed=seed, mode=mode, diag=(0.3, 6.0), margin=6))


def test_scale_rotation():
    absgrad_parity(synth.random_scene(150, 100, 3000, seed=83, diag=(0.5, 5.0), param=synth.SCALE_ROT))


@pytest.mark.parametrize("mode", [synth.SUM, synth.COMPOSITE])
def test_fused_call(mode):
    absgrad_parity(synth.random_scene(160, 120, 4000, seed=89, mode=mode, diag=(0.5, 5.0)), fused=True)


def test_image_768x512():
    absgrad_parity(synth.image_768x512())


def test_composite_768x512():
    absgrad_parity(synth.composite_768x512())


def test_heavy_2048x1360_sampled():
    wl = synth.heavy_2048x1360()
    g = gpu_run(wl, absgrad=True)
    s = oracle_scene(wl)
    rng = np.random.default_rng(8)
    valid = np.nonzero(s.proj.count > 0)[0]
    gids = np.sort(rng.choice(valid, size=1500, replace=False)).astype(np.int32)
    ref = s.render_bwd_gaussians(g["d_image"].astype(np.float64), gids)
    check_grads({"xy_abs": g["grads"]["xy_abs"][gids]}, ref, ["xy_abs"])
