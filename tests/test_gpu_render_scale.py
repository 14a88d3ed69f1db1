"""Rendering at any resolution (render scale) on the GPU against the CPU
oracle, through the C ABI (needs a B300): bit-exact projection and lists,
images and gradients (with respect to the unscaled parameters) within the
usual tolerances."""
import dataclasses

import numpy as np
import pytest

from raster_gaussian_02_b300 import synth

from gpu_common import check_lists, check_projection, full_parity, gpu_run, oracle_scene, _sampled_fwd_common
from test_gpu_fused import fused_parity

pytestmark = pytest.mark.gpu


def rescaled(wl, s):
    """The same Gaussians rendered at s output pixels per unit."""
    return dataclasses.replace(wl, width=int(round(wl.width * s)), height=int(round(wl.height * s)),
                               scale=float(s),
                               target=synth.random_scene(int(round(wl.width * s)),
                                                         int(round(wl.height * s)), 1, seed=3).target)


@pytest.mark.parametrize("s", [0.5, 1.5, 2.7])
@pytest.mark.parametrize("mode", [synth.SUM, synth.COMPOSITE])
def test_random_scene_at_scale(s, mode):
    wl = synth.random_scene(90, 60, 800, seed=109, mode=mode, diag=(0.5, 4.0), margin=4)
    full_parity(rescaled(wl, s))


def test_scale_rotation_at_scale():
    wl = synth.random_scene(80, 64, 800, seed=113, diag=(0.5, 4.0), param=synth.SCALE_ROT)
    full_parity(rescaled(wl, 1.75))


@pytest.mark.parametrize("mode", [synth.SUM, synth.COMPOSITE])
def test_fused_call_at_scale(mode):
    wl = synth.random_scene(100, 70, 1500, seed=127, mode=mode, diag=(0.5, 4.0))
    fused_parity(rescaled(wl, 2.0))


def test_headline_image_at_2048_wide():
    """The 768x512 fit rendered 2048x1365 wide (s = 8/3), forward sampled."""
    wl = synth.image_768x512()
    big = dataclasses.replace(wl, width=2048, height=1365, scale=2048 / 768, target=None)
    g = gpu_run(big, backward=False)
    s = oracle_scene(big)
    check_projection(g, s)
    check_lists(g, s)
    _sampled_fwd_common(g, s, np.random.default_rng(5))
