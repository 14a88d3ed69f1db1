"""Shared helpers of the GPU parity tests: run a workload through the C ABI
on the GPU and through the CPU oracle, and compare them.

Tolerances (derived from FP32 arithmetic, see the design notes):
  * projection (conic, box, rect, count), tile ranges and sorted lists:
    bit-exact (the touch rule and the lists are integer outcomes of the
    same FP32 operation sequence);
  * image: |gpu - ref| <= 1e-4 * max(1, |ref| / 10): absolute 1e-4 for every
    value up to 10 (every [0, 1] image, and most pixels of the sum images),
    relative 1e-5 above, where FP32's accumulation error grows with the sum
    (a pixel summing 2500 Gaussians on one tile misses a pure 1e-4 bound);
  * loss: relative 1e-5; d_image elementwise to FP32 rounding;
  * gradients, per tensor: ||gpu - ref|| / ||ref|| <= 1e-3 and
    max |gpu - ref| <= 1e-3 * max |ref|.
Composite pixels whose early-termination decision lies within 1e-4
(relative) of the threshold are "boundary-ambiguous": FP32 on the GPU and
double in the oracle may decide them differently; they are counted,
bounded, and excluded from the pixelwise checks.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from raster_gaussian_02_b300 import gs2d, synth

IMG_TOL = 1e-4
GRAD_TOL = 1e-3
AMBIG_MARGIN = 1e-4


def to_dev(a, dev="cuda"):
    if a is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def oracle_cfg(wl) -> oracle.Config:
    return oracle.Config(wl.width, wl.height, wl.mode, wl.cutoff_sigma, wl.t_min, param=wl.param,
                         scale=wl.scale)


def gpu_run(wl, d_image=None, capacity=None, sync=True, backward=True, absgrad=False):
    """Whole path on the GPU; returns numpy copies of every output."""
    R = gs2d.Rasterizer(wl.width, wl.height, wl.n, wl.mode, wl.cutoff_sigma, wl.t_min,
                        pair_capacity=capacity, param=wl.param, scale=wl.scale)
    xy, chol, rgb = to_dev(wl.xy), to_dev(wl.chol), to_dev(wl.rgb)
    depth, opac, bg = to_dev(wl.depth), to_dev(wl.opacity), to_dev(wl.background)
    R.project(xy, chol, rgb, depth, opac)
    P = R.bin_and_sort(sync=sync)
    if P is None:
        _, P, _ = gs2d.gs2d_read_status(R.workspace)
    R.render_fwd(bg)
    out = dict(R=R, P=int(P))
    if backward:
        if wl.target is not None:
            R.loss_l2(to_dev(wl.target))
        R.render_bwd(to_dev(d_image) if d_image is not None else None, absgrad=absgrad)
    torch.cuda.synchronize()
    rec = R.records()
    out.update(
        rect=R.rect[: wl.n].cpu().numpy(), count=R.count[: wl.n].cpu().numpy(),
        conic=rec["conic"].cpu().numpy(), box_x=rec["box_x"].cpu().numpy().astype(np.uint32),
        box_y=rec["box_y"].cpu().numpy().astype(np.uint32),
        ranges=R.tile_ranges.cpu().numpy(), sorted_gid=R.sorted_gid[: min(P, R.capacity)].cpu().numpy(),
        image=R.image.cpu().numpy())
    if R.t_final is not None:
        out["t_final"] = R.t_final.cpu().numpy()
        out["last"] = R.last.cpu().numpy()
    if backward:
        out["loss"] = float(R.loss.item()) if wl.target is not None else None
        out["d_image"] = R.d_image.cpu().numpy()
        out["grads"] = dict(xy=R.d_xy[: wl.n].cpu().numpy(), chol=R.d_shape[: wl.n].cpu().numpy(),
                            rgb=R.d_rgb[: wl.n].cpu().numpy())
        if R.d_opacity is not None:
            out["grads"]["opacity"] = R.d_opacity[: wl.n].cpu().numpy()
            out["grads"]["background"] = R.d_background.cpu().numpy()
        if absgrad:
            out["grads"]["xy_abs"] = R.d_xy_abs[: wl.n].cpu().numpy()
    return out


def oracle_scene(wl) -> oracle.Scene:
    return oracle.Scene(oracle_cfg(wl), wl.xy, wl.chol, wl.rgb, wl.depth, wl.opacity,
                        wl.background)


def check_projection(g, s: oracle.Scene):
    assert np.array_equal(g["count"], s.proj.count)
    assert np.array_equal(g["rect"], s.proj.rect)
    v = s.proj.count > 0
    assert np.array_equal(g["conic"][v].view(np.uint32), s.proj.conic[v].view(np.uint32))
    bb = s.proj.aabb[v]
    assert np.array_equal(g["box_x"][v] & 0xFFFF, bb[:, 0])
    assert np.array_equal(g["box_x"][v] >> 16, bb[:, 2])
    assert np.array_equal(g["box_y"][v] & 0xFFFF, bb[:, 1])
    assert np.array_equal(g["box_y"][v] >> 16, bb[:, 3])


def check_lists(g, s: oracle.Scene):
    """Lists bit-exact.  An empty tile's start is not unique (the oracle puts
    it where the list would begin, the library at 0): the library must give
    [0, 0) there."""
    assert g["P"] == s.num_pairs
    empty = s.ranges[:, 0] == s.ranges[:, 1]
    assert np.array_equal(g["ranges"][~empty], s.ranges[~empty])
    assert np.all(g["ranges"][empty] == 0)
    assert np.array_equal(g["sorted_gid"], s.sorted_gid)


IMG_REL_FROM = 10.0  # values above this get the relative bound IMG_TOL / IMG_REL_FROM


def image_errors(gpu, ref):
    """Error of each image value in units of its bound: the absolute error
    for values up to IMG_REL_FROM, the error relative to |ref| / IMG_REL_FROM
    above (so the check is `<= IMG_TOL` either way)."""
    return np.abs(gpu.astype(np.float64) - ref) / np.maximum(1.0, np.abs(ref) / IMG_REL_FROM)


def check_image(g, ref_fwd, composite: bool, max_ambiguous_frac=1e-3):
    ok = np.ones(ref_fwd["image"].shape[1:], bool)
    if composite:
        amb = ref_fwd["margin"] < AMBIG_MARGIN
        assert amb.mean() <= max_ambiguous_frac, amb.mean()
        ok = ~amb
        assert np.array_equal(g["last"][ok], ref_fwd["last"][ok])
        tref = ref_fwd["t_final"][ok]
        tf = np.abs(g["t_final"][ok].astype(np.float64) - tref)
        assert np.all(tf <= 1e-6 + 1e-4 * tref), tf.max(initial=0)
    err = image_errors(g["image"], ref_fwd["image"])[:, ok]
    if err.size and err.max() > IMG_TOL:
        k = np.unravel_index(np.argmax(err), err.shape)
        raise AssertionError(f"image error {err.max():.3g} at a pixel of value "
                             f"{ref_fwd['image'][:, ok][k]:.4g}")
    return ok


def check_grads(gpu: dict, ref: dict, keys, mask=None):
    for k in keys:
        a = gpu[k].astype(np.float64)
        b = ref[k]
        if mask is not None and a.ndim >= 1 and a.shape[0] == mask.shape[0]:
            a, b = a[mask], b[mask]
        nb = np.linalg.norm(b)
        if nb == 0:
            assert np.abs(a).max(initial=0) == 0, k
            continue
        rel = np.linalg.norm(a - b) / nb
        assert rel <= GRAD_TOL, (k, rel)
        assert np.abs(a - b).max() <= GRAD_TOL * np.abs(b).max(), (k, np.abs(a - b).max(), np.abs(b).max())


def full_parity(wl, composite=None, check_chain=True):
    """Every output of the path at a size the oracle renders in full."""
    composite = wl.mode == synth.COMPOSITE if composite is None else composite
    g = gpu_run(wl)
    s = oracle_scene(wl)
    check_projection(g, s)
    check_lists(g, s)
    ref = s.render()
    ok = check_image(g, ref, composite)
    # the loss kernel alone, on the GPU's own image
    loss_ref, dimg_ref = oracle.loss_l2(g["image"], wl.target)
    assert abs(g["loss"] - loss_ref) <= 1e-5 * abs(loss_ref) + 1e-12
    np.testing.assert_allclose(g["d_image"], dimg_ref, rtol=1e-5, atol=1e-7 * np.abs(dimg_ref).max())
    # the backward alone, on the GPU's own d_image
    gr = s.render_bwd(g["d_image"].astype(np.float64))
    keys = ["xy", "chol", "rgb"] + (["opacity", "background"] if composite else [])
    if composite:
        # Gaussians touching an ambiguous pixel see different stop decisions
        amb_pix = ~ok
        touched = _gaussians_touching(s, amb_pix)
        keep = np.ones(wl.n, bool)
        keep[touched] = False
        check_grads(g["grads"], gr, [k for k in keys if k != "background"], mask=keep)
        if not amb_pix.any():
            check_grads(g["grads"], gr, ["background"])
    else:
        check_grads(g["grads"], gr, keys)
    return g, s, ref


def _sampled_fwd_common(g, s: oracle.Scene, rng, m_pix=20000):
    """Sampled pixels against the oracle's per-pixel forward (sum mode)."""
    H, W = s.cfg.height, s.cfg.width
    pix = rng.choice(H * W, size=min(m_pix, H * W), replace=False)
    ref = s.render_pixels(pix)
    err = image_errors(g["image"].reshape(3, -1)[:, pix].T, ref["rgb"])
    assert err.max(initial=0) <= IMG_TOL, err.max()


def _sampled_bwd_common(g, s: oracle.Scene, wl, rng, m_pix=20000, m_gauss=1500):
    """Full-size check by sampling: pixels against the oracle's per-pixel
    forward, the loss, and Gaussians against its per-Gaussian backward."""
    H, W = s.cfg.height, s.cfg.width
    pix = rng.choice(H * W, size=min(m_pix, H * W), replace=False)
    ref = s.render_pixels(pix)
    err = image_errors(g["image"].reshape(3, -1)[:, pix].T, ref["rgb"])
    assert err.max(initial=0) <= IMG_TOL, err.max()
    loss_ref, _ = oracle.loss_l2(g["image"], wl.target)
    assert abs(g["loss"] - loss_ref) <= 1e-5 * loss_ref
    valid = np.nonzero(s.proj.count > 0)[0]
    gids = np.sort(rng.choice(valid, size=min(m_gauss, len(valid)), replace=False)).astype(np.int32)
    gr = s.render_bwd_gaussians(g["d_image"].astype(np.float64), gids)
    check_grads({k: g["grads"][k][gids] for k in ("xy", "chol", "rgb")}, gr, ("xy", "chol", "rgb"))


def _gaussians_touching(s: oracle.Scene, pix_mask):
    ii, jj = np.nonzero(pix_mask)
    out = set()
    tx = s.cfg.tiles_x
    for i, j in zip(ii, jj):
        t = (i // 16) * tx + j // 16
        a, b = s.ranges[t]
        out.update(int(x) for x in s.sorted_gid[a:b])
    return np.array(sorted(out), dtype=np.int64)
