"""GPU path against the CPU oracle, through the C ABI (needs a B300).

Full-image parity at sizes the oracle finishes in seconds (several tiles,
ragged edges, long lists), sampled parity at the full workload sizes, and
the edge cases: empty input, culled Gaussians, capacity misses, long tile
lists, early termination, other cutoffs, determinism.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle
from raster_gaussian_02_b300 import gs2d, synth

from gpu_common import (IMG_TOL, _gaussians_touching, check_grads, check_image, check_lists,
                        check_projection, full_parity, gpu_run, image_errors, oracle_scene, to_dev)

pytestmark = pytest.mark.gpu


# ------------------------------------------------------------- full parity --

def test_small_64x64_sum():
    full_parity(synth.small_64x64())


@pytest.mark.parametrize("w,h,n,seed", [(1, 1, 3, 1), (17, 13, 40, 2), (100, 37, 300, 3),
                                        (33, 65, 500, 4), (250, 130, 3000, 5)])
@pytest.mark.parametrize("mode", [synth.SUM, synth.COMPOSITE])
def test_random_ragged(w, h, n, seed, mode):
    wl = synth.random_scene(w, h, n, seed=seed, mode=mode, diag=(0.3, 6.0), margin=6)
    full_parity(wl)


def test_image_768x512_sum():
    full_parity(synth.image_768x512())


def test_composite_768x512():
    full_parity(synth.composite_768x512())


def test_long_tile_lists():
    """Thousands of Gaussians on one tile (lists longer than a staging chunk)
    plus one Gaussian covering the whole image."""
    for mode in (synth.SUM, synth.COMPOSITE):
        wl = synth.random_scene(64, 48, 3000, seed=8, mode=mode, diag=(0.5, 2.0))
        wl.xy[:2500] = np.random.default_rng(0).uniform(20, 30, (2500, 2)).astype(np.float32)
        wl.chol[0] = [40.0, 3.0, 30.0]
        if mode == synth.COMPOSITE:
            wl.opacity[:] = np.minimum(wl.opacity, 0.3)
        full_parity(wl)


@pytest.mark.parametrize("mode", [synth.SUM, synth.COMPOSITE])
def test_empty_tiles(mode):
    """Few Gaussians on a large image: most tiles have empty lists."""
    wl = synth.random_scene(300, 200, 25, seed=21, mode=mode, diag=(0.5, 6.0))
    g, s, _ = full_parity(wl)
    assert (s.ranges[:, 0] == s.ranges[:, 1]).sum() > 100


@pytest.mark.parametrize("w,h,n", [(1024, 512, 20000), (1040, 512, 20000), (720, 720, 3000)])
def test_sum_sort_paths_near_the_tile_limit(w, h, n):
    """2048, 2080 and 2025 tiles: the counting sort by tile (at most 2048
    tiles) and, above it, the radix passes give the oracle's lists."""
    wl = synth.random_scene(w, h, n, seed=w + n, diag=(0.5, 12.0))
    g = gpu_run(wl)
    s = oracle_scene(wl)
    check_projection(g, s)
    check_lists(g, s)


def test_composite_list_longer_than_shared_memory_sort():
    """One tile with more than 4096 Gaussians: its depth sort runs in the
    workspace instead of shared memory."""
    wl = synth.random_scene(48, 32, 7000, seed=19, mode=synth.COMPOSITE, diag=(0.5, 2.0))
    wl.xy[:6000] = np.random.default_rng(1).uniform(18, 30, (6000, 2)).astype(np.float32)
    wl.opacity[:] = np.minimum(wl.opacity, 0.001)  # no pixel reaches t_min: the test is about the sort
    wl.depth = (np.round(wl.depth * 50) / 50).astype(np.float32)  # many equal depths: ties by index
    g, s, _ = full_parity(wl)
    assert (s.ranges[:, 1] - s.ranges[:, 0]).max() > 4096


@pytest.mark.parametrize("w,h,n", [(1024, 512, 8000), (1040, 512, 8000)])
def test_composite_sort_paths_near_the_tile_limit(w, h, n):
    """2048 and 2080 tiles: counting sort + per-tile depth sort, and the radix
    passes, give the oracle's (depth, index) lists."""
    wl = synth.random_scene(w, h, n, seed=w + n + 1, mode=synth.COMPOSITE, diag=(0.5, 12.0))
    g = gpu_run(wl)
    s = oracle_scene(wl)
    check_projection(g, s)
    check_lists(g, s)


def test_composite_radix_many_partitions():
    """2752 tiles and about 630K pairs: the composite keys (tile, depth,
    index; 44 bits) go through six 8-bit radix passes over more than 128
    partitions of 2048 keys, where every digit's offsets come from the
    per-partition count tables and the scatter stages each partition in
    shared memory; the lists must be the oracle's."""
    wl = synth.random_scene(1024, 680, 100_000, seed=77, mode=synth.COMPOSITE, diag=(0.5, 8.0))
    g = gpu_run(wl, backward=False)
    s = oracle_scene(wl)
    assert g["P"] > 128 * 2048
    check_projection(g, s)
    check_lists(g, s)


def test_sum_radix_many_partitions_ragged():
    """Sum mode above 2048 tiles with more than 128 partitions and a last
    partition that is not full: lists bit-exact."""
    wl = synth.random_scene(1040, 688, 90_001, seed=78, diag=(0.5, 8.0))
    g = gpu_run(wl, backward=False)
    s = oracle_scene(wl)
    assert g["P"] > 128 * 2048 and g["P"] % 2048 != 0
    check_projection(g, s)
    check_lists(g, s)


def test_composite_early_termination_dense():
    wl = synth.random_scene(96, 80, 4000, seed=12, mode=synth.COMPOSITE, diag=(1.0, 4.0))
    wl.opacity[:] = 0.95
    g, s, ref = full_parity(wl)
    assert (ref["t_final"] < 1e-4).mean() > 0.3


def test_composite_no_termination():
    wl = synth.random_scene(80, 64, 2000, seed=13, mode=synth.COMPOSITE, diag=(1.0, 4.0))
    wl.t_min = 0.0
    full_parity(wl)


@pytest.mark.parametrize("k", [1.5, 2.0, 5.0])
def test_other_cutoffs(k):
    wl = synth.random_scene(120, 90, 1500, seed=14, diag=(0.5, 4.0))
    wl.cutoff_sigma = k
    full_parity(wl)


def test_heavy_tail_cropped():
    """Heavy-tailed sizes and rotations (the 2048x1360 distribution) on a
    crop the oracle renders in full."""
    rng = np.random.default_rng(15)
    n = 6000
    wl = synth.Workload("heavy_crop", 400, 272, synth.SUM, synth.positions_uniform(n, 272, 400, rng),
                        synth.cholesky_heavy_tail(n, rng), rng.uniform(0, 1, (n, 3)).astype(np.float32),
                        rng.uniform(0, 1, (3, 272, 400)).astype(np.float32))
    full_parity(wl)


# ------------------------------------------------------------ full sizes --

def _sampled_fwd(g, s, rng, m=20000, composite=False):
    H, W = s.cfg.height, s.cfg.width
    pix = rng.choice(H * W, size=min(m, H * W), replace=False)
    ref = s.render_pixels(pix)
    gimg = g["image"].reshape(3, -1)[:, pix].T
    ok = np.ones(len(pix), bool)
    if composite:
        ok = ref["margin"] >= 1e-4
        assert np.array_equal(g["last"].ravel()[pix][ok], ref["last"][ok])
    err = image_errors(gimg[ok], ref["rgb"][ok])
    assert err.max(initial=0) <= IMG_TOL, err.max()


def _sampled_bwd(g, s, rng, m=1500, keys=("xy", "chol", "rgb")):
    valid = np.nonzero(s.proj.count > 0)[0]
    gids = np.sort(rng.choice(valid, size=min(m, len(valid)), replace=False)).astype(np.int32)
    ref = s.render_bwd_gaussians(g["d_image"].astype(np.float64), gids)
    gpu = {k: g["grads"][k][gids] for k in keys}
    check_grads(gpu, ref, keys)


def test_heavy_2048x1360_full_size():
    wl = synth.heavy_2048x1360()
    g = gpu_run(wl)
    s = oracle_scene(wl)
    check_projection(g, s)
    check_lists(g, s)
    rng = np.random.default_rng(0)
    _sampled_fwd(g, s, rng)
    loss_ref, _ = oracle.loss_l2(g["image"], wl.target)
    assert abs(g["loss"] - loss_ref) <= 1e-5 * loss_ref
    _sampled_bwd(g, s, rng)


def test_render_4096x4096_2m_forward():
    wl = synth.render_4096x4096()
    g = gpu_run(wl, backward=False, capacity=8_000_000)
    s = oracle_scene(wl)
    check_projection(g, s)
    check_lists(g, s)
    _sampled_fwd(g, s, np.random.default_rng(1), m=20000)


@pytest.mark.parametrize("n", [10_000, 200_000, 1_000_000])
def test_sweep_768x512_forward(n):
    wl = synth.render_uniform(768, 512, n, seed=5000 + n)
    g = gpu_run(wl, backward=False)
    s = oracle_scene(wl)
    check_projection(g, s)
    check_lists(g, s)
    _sampled_fwd(g, s, np.random.default_rng(2), m=5000)


# ------------------------------------------------------------- edge cases --

def test_no_gaussians():
    for mode in (synth.SUM, synth.COMPOSITE):
        wl = synth.random_scene(40, 30, 0, seed=1, mode=mode)
        if mode == synth.COMPOSITE:
            wl.depth = np.zeros(0, np.float32)
            wl.opacity = np.zeros(0, np.float32)
            wl.background = np.array([0.2, 0.3, 0.4], np.float32)
        g = gpu_run(wl)
        assert g["P"] == 0
        assert np.all(g["ranges"] == 0)
        if mode == synth.SUM:
            assert np.all(g["image"] == 0)
        else:
            np.testing.assert_array_equal(g["image"], np.broadcast_to(wl.background[:, None, None], g["image"].shape))
            dimg = g["d_image"].astype(np.float64)
            np.testing.assert_allclose(g["grads"]["background"], dimg.sum(axis=(1, 2)), rtol=1e-5)


def test_all_culled():
    wl = synth.random_scene(48, 48, 64, seed=2)
    wl.xy[:20] = np.nan
    wl.chol[20:40, 0] = 0.0
    wl.chol[40:, 2] = np.inf
    g = gpu_run(wl)
    assert g["P"] == 0 and np.all(g["count"] == 0)
    assert np.all(g["image"] == 0)
    for k in ("xy", "chol", "rgb"):
        assert np.all(g["grads"][k] == 0)


def test_partially_culled_and_offscreen():
    wl = synth.random_scene(64, 64, 400, seed=3, margin=40)
    wl.xy[::7] = np.nan
    wl.chol[1::11, 2] = 0.0
    full_parity(wl)


def test_capacity_miss_sync_and_async():
    wl = synth.random_scene(96, 96, 800, seed=4, diag=(1.0, 6.0))
    s = oracle_scene(wl)
    P = s.num_pairs
    cap = P // 2
    R = gs2d.Rasterizer(wl.width, wl.height, wl.n, pair_capacity=cap)
    R.project(to_dev(wl.xy), to_dev(wl.chol), to_dev(wl.rgb))
    out = C.c_int64(0)
    st = gs2d.gs2d_bin_and_sort(R.cfg, R.n, R.rec, R.rect, R.count, R.capacity, out, R.tile_ranges,
                                R.sorted_gid, R.workspace)
    assert st == gs2d.GS2D_ERR_CAPACITY and out.value == P
    # asynchronous: the flags stay on the device and the lists are empty
    gs2d.check(gs2d.gs2d_bin_and_sort(R.cfg, R.n, R.rec, R.rect, R.count, R.capacity, None,
                                      R.tile_ranges, R.sorted_gid, R.workspace), "bin")
    st, pairs, flags = gs2d.gs2d_read_status(R.workspace)
    assert st == gs2d.GS2D_ERR_CAPACITY and pairs == P and flags & gs2d.GS2D_FLAG_CAPACITY
    assert torch.all(R.tile_ranges == 0)
    R.render_fwd()
    assert torch.all(R.image == 0)
    # growing the capacity fixes it
    assert R.bin_and_sort(sync=True, grow=True) == P
    R.render_fwd()
    ref = s.render()
    assert image_errors(R.image.cpu().numpy(), ref["image"]).max() <= IMG_TOL


def test_exact_capacity():
    wl = synth.random_scene(64, 64, 500, seed=6)
    P = oracle_scene(wl).num_pairs
    g = gpu_run(wl, capacity=P)
    assert g["P"] == P
    full = oracle_scene(wl).render()
    assert image_errors(g["image"], full["image"]).max() <= IMG_TOL


@pytest.mark.parametrize("mode", [synth.SUM, synth.COMPOSITE])
def test_deterministic(mode):
    """No atomics on floats anywhere: two runs are bit-identical."""
    wl = synth.random_scene(200, 150, 5000, seed=7, mode=mode, diag=(0.5, 5.0))
    a = gpu_run(wl)
    b = gpu_run(wl)
    assert np.array_equal(a["image"], b["image"])
    assert a["loss"] == b["loss"]
    for k in a["grads"]:
        assert np.array_equal(a["grads"][k], b["grads"][k]), k


@pytest.mark.parametrize("mode", [synth.SUM, synth.COMPOSITE])
@pytest.mark.parametrize("absgrad", [False, True])
def test_repeated_backward_over_one_binning(mode, absgrad):
    """Backward, fused pass and backward again over one binning: the two
    backward calls give the same gradients bit for bit (nothing carried over
    from an earlier call), the fused pass agrees with them, and all match
    the oracle."""
    wl = synth.random_scene(200, 150, 5000, seed=17, mode=mode, diag=(0.5, 5.0))
    R = gs2d.Rasterizer(wl.width, wl.height, wl.n, wl.mode, wl.cutoff_sigma, wl.t_min)
    R.project(to_dev(wl.xy), to_dev(wl.chol), to_dev(wl.rgb), to_dev(wl.depth), to_dev(wl.opacity))
    R.bin_and_sort(sync=True)
    bg = to_dev(wl.background)
    R.render_fwd(bg)
    R.loss_l2(to_dev(wl.target))
    runs = []
    for k in range(3):
        if k == 1:
            R.render_fwd_bwd_l2(to_dev(wl.target), bg, absgrad=absgrad)
        else:
            R.render_bwd(absgrad=absgrad)
        torch.cuda.synchronize()
        got = {"xy": R.d_xy[: wl.n].cpu().numpy(), "chol": R.d_shape[: wl.n].cpu().numpy(),
               "rgb": R.d_rgb[: wl.n].cpu().numpy()}
        if absgrad:
            got["xy_abs"] = R.d_xy_abs[: wl.n].cpu().numpy()
        runs.append(got)
    for k in runs[0]:
        assert np.array_equal(runs[0][k], runs[2][k]), k
    check_grads({k: v.astype(np.float64) for k, v in runs[1].items()},
                {k: v.astype(np.float64) for k, v in runs[0].items()}, list(runs[0].keys()))
    s = oracle_scene(wl)
    _, dimg = oracle.loss_l2(R.image.cpu().numpy(), wl.target)
    ref = s.render_bwd(dimg)
    keep = None
    if mode == synth.COMPOSITE:
        ok = check_image({"image": R.image.cpu().numpy(), "t_final": R.t_final.cpu().numpy(),
                          "last": R.last.cpu().numpy()}, s.render(), True)
        keep = np.ones(wl.n, bool)
        keep[_gaussians_touching(s, ~ok)] = False
    check_grads(runs[2], ref, list(runs[2].keys()), mask=keep)


def test_backward_with_external_gradient():
    """render_bwd given an arbitrary dL/dC (not from the L2 loss)."""
    for mode in (synth.SUM, synth.COMPOSITE):
        wl = synth.random_scene(120, 100, 1500, seed=9, mode=mode, diag=(0.5, 5.0))
        dimg = synth.d_image(100, 120, seed=3, scale=1e-3)
        g = gpu_run(wl, d_image=dimg)
        s = oracle_scene(wl)
        ref = s.render()
        ok = check_image(g, ref, mode == synth.COMPOSITE)
        gr = s.render_bwd(dimg.astype(np.float64))
        keys = ["xy", "chol", "rgb"] + (["opacity"] if mode == synth.COMPOSITE else [])
        if ok.all():
            check_grads(g["grads"], gr, keys + (["background"] if mode == synth.COMPOSITE else []))


def test_depth_ties_and_negative_zero():
    """Equal depths order by index; -0 and +0 are equal depths."""
    wl = synth.random_scene(64, 64, 600, seed=10, mode=synth.COMPOSITE, diag=(1.0, 5.0))
    wl.depth[:] = np.round(wl.depth * 4) / 4
    wl.depth[::5] = -0.0
    wl.depth[1::5] = 0.0
    wl.depth[2::9] = -0.5
    full_parity(wl)
