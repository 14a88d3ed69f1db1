"""The fused forward + L2 loss + backward call (gs2d_render_fwd_bwd_l2)
against the CPU oracle, through the C ABI (needs a B300).

The fused pass must give what the three separate calls give: the same image
(the per-pixel code and summation order are shared, so bit-identical), the
oracle's loss of that image, and the oracle's gradients for the oracle's
dL/dC of that image, within the tolerances of the separate calls.
"""
import numpy as np
import pytest
import torch

import oracle
from raster_gaussian_02_b300 import gs2d, synth

from gpu_common import (GRAD_TOL, _gaussians_touching, check_grads, check_image, gpu_run,
                        oracle_scene, to_dev)

pytestmark = pytest.mark.gpu


def fused_run(wl, write_image=True, capacity=None, absgrad=False):
    R = gs2d.Rasterizer(wl.width, wl.height, wl.n, wl.mode, wl.cutoff_sigma, wl.t_min,
                        pair_capacity=capacity, param=wl.param, scale=wl.scale)
    R.project(to_dev(wl.xy), to_dev(wl.chol), to_dev(wl.rgb), to_dev(wl.depth),
              to_dev(wl.opacity))
    R.bin_and_sort(sync=True)
    if not write_image:
        R.image.fill_(-7.0)
    R.render_fwd_bwd_l2(to_dev(wl.target), to_dev(wl.background), write_image=write_image,
                        absgrad=absgrad)
    torch.cuda.synchronize()
    out = dict(image=R.image.cpu().numpy(), loss=float(R.loss.item()),
               grads=dict(xy=R.d_xy[: wl.n].cpu().numpy(), chol=R.d_shape[: wl.n].cpu().numpy(),
                          rgb=R.d_rgb[: wl.n].cpu().numpy()))
    if R.d_opacity is not None:
        out["grads"]["opacity"] = R.d_opacity[: wl.n].cpu().numpy()
        out["grads"]["background"] = R.d_background.cpu().numpy()
    if absgrad:
        out["grads"]["xy_abs"] = R.d_xy_abs[: wl.n].cpu().numpy()
    return out


def fused_parity(wl):
    comp = wl.mode == synth.COMPOSITE
    g = gpu_run(wl)     # separate calls: image, t_final, last, grads
    f = fused_run(wl)
    s = oracle_scene(wl)
    assert np.array_equal(f["image"], g["image"])
    ok = check_image(g, s.render(), comp)
    loss_ref, dimg_ref = oracle.loss_l2(f["image"], wl.target)
    assert abs(f["loss"] - loss_ref) <= 1e-5 * abs(loss_ref) + 1e-12, (f["loss"], loss_ref)
    gr = s.render_bwd(dimg_ref)
    keys = ["xy", "chol", "rgb"] + (["opacity", "background"] if comp else [])
    if comp:
        keep = np.ones(wl.n, bool)
        keep[_gaussians_touching(s, ~ok)] = False
        check_grads(f["grads"], gr, [k for k in keys if k != "background"], mask=keep)
        if ok.all():
            check_grads(f["grads"], gr, ["background"])
    else:
        check_grads(f["grads"], gr, keys)
    # and the separate calls agree with the fused one to FP32 rounding order
    check_grads({k: v.astype(np.float64) for k, v in f["grads"].items()},
                {k: v.astype(np.float64) for k, v in g["grads"].items()}, keys)
    return f, g, s


def test_small_64x64_sum():
    fused_parity(synth.small_64x64())


@pytest.mark.parametrize("w,h,n,seed", [(1, 1, 3, 1), (17, 13, 40, 2), (100, 37, 300, 3),
                                        (250, 130, 3000, 5)])
@pytest.mark.parametrize("mode", [synth.SUM, synth.COMPOSITE])
def test_random_ragged(w, h, n, seed, mode):
    wl = synth.random_scene(w, h, n, seed=seed, mode=mode, diag=(0.3, 6.0), margin=6)
    fused_parity(wl)


def test_image_768x512_sum():
    fused_parity(synth.image_768x512())


def test_composite_768x512():
    fused_parity(synth.composite_768x512())


def test_long_tile_lists():
    """Lists longer than one staging round (the sum backward restages)."""
    for mode in (synth.SUM, synth.COMPOSITE):
        wl = synth.random_scene(64, 48, 3000, seed=8, mode=mode, diag=(0.5, 2.0))
        wl.xy[:2500] = np.random.default_rng(0).uniform(20, 30, (2500, 2)).astype(np.float32)
        wl.chol[0] = [40.0, 3.0, 30.0]
        if mode == synth.COMPOSITE:
            wl.opacity[:] = np.minimum(wl.opacity, 0.3)
        fused_parity(wl)


def test_composite_early_termination_dense():
    wl = synth.random_scene(96, 80, 4000, seed=12, mode=synth.COMPOSITE, diag=(1.0, 4.0))
    wl.opacity[:] = 0.95
    fused_parity(wl)


@pytest.mark.parametrize("mode", [synth.SUM, synth.COMPOSITE])
def test_image_not_written_and_deterministic(mode):
    wl = synth.random_scene(200, 150, 5000, seed=7, mode=mode, diag=(0.5, 5.0))
    a = fused_run(wl)
    b = fused_run(wl, write_image=False)
    assert np.all(b["image"] == -7.0)
    assert a["loss"] == b["loss"]
    for k in a["grads"]:
        assert np.array_equal(a["grads"][k], b["grads"][k]), k


def test_no_gaussians():
    wl = synth.random_scene(40, 30, 0, seed=1)
    f = fused_run(wl)
    assert np.all(f["image"] == 0)
    loss_ref, _ = oracle.loss_l2(f["image"], wl.target)
    assert abs(f["loss"] - loss_ref) <= 1e-6 * loss_ref


def test_heavy_2048x1360_full_size():
    """Full size: sampled Gaussians against the oracle's per-Gaussian backward."""
    wl = synth.heavy_2048x1360()
    f = fused_run(wl)
    s = oracle_scene(wl)
    loss_ref, dimg_ref = oracle.loss_l2(f["image"], wl.target)
    assert abs(f["loss"] - loss_ref) <= 1e-5 * loss_ref
    rng = np.random.default_rng(4)
    valid = np.nonzero(s.proj.count > 0)[0]
    gids = np.sort(rng.choice(valid, size=1500, replace=False)).astype(np.int32)
    ref = s.render_bwd_gaussians(dimg_ref, gids)
    check_grads({k: f["grads"][k][gids] for k in ("xy", "chol", "rgb")}, ref, ("xy", "chol", "rgb"))


@pytest.mark.parametrize("k", [250, 262, 520])
@pytest.mark.parametrize("opacity", [0.08, 0.9])
def test_composite_long_lists_split_in_two(k, opacity):
    """Lists around and above the length at which the fused composite kernel
    splits a tile's backward between two blocks (256 entries): k small
    Gaussians on one tile, with low opacity (nothing terminates, both halves
    work) and high opacity (pixels terminate early, many in the front half)."""
    wl = synth.random_scene(64, 48, k + 200, seed=30 + k, mode=synth.COMPOSITE, diag=(0.5, 1.5))
    wl.xy[:k] = np.random.default_rng(k).uniform(17, 31, (k, 2)).astype(np.float32)
    wl.opacity[:k] = opacity
    f, g, s = fused_parity(wl)
    lens = s.ranges[:, 1] - s.ranges[:, 0]
    assert lens.max() >= k - 5  # the crowded tile's list
