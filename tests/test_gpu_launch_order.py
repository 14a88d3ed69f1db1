"""gs2d_render_fwd with and without the binning's workspace.

With the workspace (and at most 2048 tiles) the forward's blocks take the
tiles in the counting sort's launch order, longest lists first, reading each
tile's range from its order slot; without it they take the tiles in index
order and read tile_ranges.  Every pixel is computed by the same thread
sequence either way, so the outputs must be bit-identical.  The parity tests
cover the workspace form against the oracle (the Rasterizer passes its
workspace); this file pins the other form to it."""
import pytest
import torch

from raster_gaussian_02_b300 import gs2d, synth
from gpu_common import to_dev

pytestmark = pytest.mark.gpu


def _scene(mode):
    if mode == "sum":
        return synth.image_768x512()
    return synth.composite_768x512()


@pytest.mark.parametrize("mode", ["sum", "composite"])
def test_same_outputs_without_the_workspace(mode):
    wl = _scene(mode)
    R = gs2d.Rasterizer(wl.width, wl.height, wl.n, wl.mode, wl.cutoff_sigma, wl.t_min)
    R.project(to_dev(wl.xy), to_dev(wl.chol), to_dev(wl.rgb), to_dev(wl.depth), to_dev(wl.opacity))
    assert R.bin_and_sort(sync=True) > 0
    bg = to_dev(wl.background)
    R.render_fwd(bg)
    torch.cuda.synchronize()
    with_ws = [R.image.clone()] + ([R.t_final.clone(), R.last.clone()] if R.t_final is not None else [])
    R.image.fill_(-1.0)
    if R.t_final is not None:
        R.t_final.fill_(-1.0)
        R.last.fill_(-1)
    gs2d.check(gs2d.gs2d_render_fwd(R.cfg, R.n, R.rec, R.tile_ranges, R.sorted_gid, bg, R.image,
                                    R.t_final, R.last, None), "gs2d_render_fwd")
    torch.cuda.synchronize()
    without = [R.image] + ([R.t_final, R.last] if R.t_final is not None else [])
    for a, b in zip(with_ws, without):
        assert torch.equal(a, b)


def test_misaligned_workspace_is_rejected():
    wl = synth.random_scene(64, 64, 100, seed=11)
    R = gs2d.Rasterizer(wl.width, wl.height, wl.n)
    R.project(to_dev(wl.xy), to_dev(wl.chol), to_dev(wl.rgb))
    R.bin_and_sort(sync=True)
    odd = R.workspace[4:]
    st = gs2d.gs2d_render_fwd(R.cfg, R.n, R.rec, R.tile_ranges, R.sorted_gid, None, R.image, None,
                              None, odd)
    assert st == gs2d.GS2D_ERR_INVALID_ARG
