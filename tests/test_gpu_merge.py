"""The moment-matching merge on the GPU against the CPU oracle, through the
C ABI (needs a B300).  The pairs are integer decisions taken on the same
doubles, so the merged set must match exactly: positions, colours and (for
Cholesky factors) shapes bit for bit; scale-rotation shapes, which pass
through a double atan2/cos/sin, within 1e-6."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from raster_gaussian_02_b300 import gs2d, synth

from gpu_common import oracle_cfg, to_dev

pytestmark = pytest.mark.gpu


def gpu_merge(wl, k):
    R = gs2d.Rasterizer(wl.width, wl.height, wl.n, wl.mode, wl.cutoff_sigma, wl.t_min,
                        param=wl.param, scale=wl.scale)
    R.project(to_dev(wl.xy), to_dev(wl.chol), to_dev(wl.rgb))
    R.bin_and_sort(sync=True)
    xy, sh, rgb, m = R.merge(k)
    torch.cuda.synchronize()
    return xy.cpu().numpy(), sh.cpu().numpy(), rgb.cpu().numpy(), m


def check(wl, k):
    gx, gs, gr, gm = gpu_merge(wl, k)
    ox, osh, orgb, om = oracle.merge(oracle_cfg(wl), wl.xy, wl.chol, wl.rgb, k)
    assert gm == om
    assert np.array_equal(gx, ox)
    assert np.array_equal(gr, orgb)
    if wl.param == synth.SCALE_ROT:
        np.testing.assert_allclose(gs, osh, rtol=1e-6, atol=1e-6)
    else:
        assert np.array_equal(gs, osh)
    return gm


@pytest.mark.parametrize("param", [synth.CHOLESKY, synth.SCALE_ROT])
@pytest.mark.parametrize("w,h,n,seed", [(1, 1, 3, 1), (40, 30, 200, 2), (130, 90, 4000, 3)])
def test_random_scenes(param, w, h, n, seed):
    wl = synth.random_scene(w, h, n, seed=seed, diag=(0.3, 5.0), margin=4, param=param)
    wl.chol[:3, 1 if param == synth.SCALE_ROT else 0] = 0.0  # culled ones pass through
    for k in (0, 7, n // 8, n):
        check(wl, k)


def test_render_scale():
    wl = synth.random_scene(60, 45, 1500, seed=5, diag=(0.4, 3.0))
    check(dataclasses.replace(wl, width=150, height=113, scale=2.5), 300)


def test_image_768x512_to_40k():
    wl = synth.image_768x512()
    assert check(wl, 10_000) == 10_000


def test_heavy_2048x1360_sr():
    wl = synth.heavy_2048x1360_sr()
    assert check(wl, 50_000) > 0
