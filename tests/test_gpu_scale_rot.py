"""Scale-rotation shape parameters (s_x, s_y, theta) on the GPU against the
CPU oracle, through the C ABI (needs a B300).  The FP32 mask data (conic,
box) are bit-exact, which also pins the kernel's FP32 sin/cos to the
oracle's; images and gradients within the tolerances of the Cholesky path.
"""
import numpy as np
import pytest

import oracle
from raster_gaussian_02_b300 import synth

from gpu_common import (_sampled_bwd_common, check_lists, check_projection, full_parity, gpu_run,
                        oracle_scene)
from test_gpu_fused import fused_parity

pytestmark = pytest.mark.gpu

SR = synth.SCALE_ROT


@pytest.mark.parametrize("w,h,n,seed", [(1, 1, 3, 1), (17, 13, 40, 2), (100, 37, 300, 3),
                                        (250, 130, 3000, 5)])
@pytest.mark.parametrize("mode", [synth.SUM, synth.COMPOSITE])
def test_random_ragged(w, h, n, seed, mode):
    wl = synth.random_scene(w, h, n, seed=seed, mode=mode, diag=(0.3, 6.0), margin=6, param=SR)
    full_parity(wl)


def test_image_768x512_sr():
    full_parity(synth.image_768x512_sr())


def test_wide_angles_and_culling():
    """Angles over +-1000 rad exercise the range reduction; a zero scale,
    |theta| > 65536 and a non-finite angle are culled."""
    wl = synth.random_scene(120, 90, 2000, seed=61, diag=(0.5, 5.0), param=SR)
    rng = np.random.default_rng(0)
    wl.chol[:, 2] = rng.uniform(-1000, 1000, wl.n).astype(np.float32)
    wl.chol[0] = [0.0, 2.0, 0.3]
    wl.chol[1] = [2.0, 3.0, 70000.0]
    wl.chol[2] = [2.0, 3.0, np.inf]
    g, s, _ = full_parity(wl)
    assert list(s.proj.count[:3]) == [0, 0, 0]


@pytest.mark.parametrize("mode", [synth.SUM, synth.COMPOSITE])
def test_fused_call(mode):
    wl = synth.random_scene(150, 100, 3000, seed=67, mode=mode, diag=(0.5, 5.0), param=SR)
    fused_parity(wl)


def test_heavy_2048x1360_sr_full_size():
    wl = synth.heavy_2048x1360_sr()
    g = gpu_run(wl)
    s = oracle_scene(wl)
    check_projection(g, s)
    check_lists(g, s)
    _sampled_bwd_common(g, s, wl, np.random.default_rng(6))
