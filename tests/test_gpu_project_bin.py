"""gs2d_project_bin_and_sort (projection and binning in one call) against the
two separate calls and against the oracle, through the C ABI (needs a B300).

With the counting sort (at most 2048 tiles and 2^20 Gaussians) the
projection runs inside the sort's histogram kernel; above that the call
projects first and then takes the radix path.  Either way every output must
equal what gs2d_project followed by gs2d_bin_and_sort writes, bit for bit,
and the lists must be the oracle's.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from raster_gaussian_02_b300 import gs2d, synth

from gpu_common import check_lists, check_projection, oracle_scene, to_dev

pytestmark = pytest.mark.gpu


def _run(wl, fused: bool, capacity=None):
    R = gs2d.Rasterizer(wl.width, wl.height, wl.n, wl.mode, wl.cutoff_sigma, wl.t_min,
                        pair_capacity=capacity, param=wl.param, scale=wl.scale)
    args = (to_dev(wl.xy), to_dev(wl.chol), to_dev(wl.rgb), to_dev(wl.depth), to_dev(wl.opacity))
    if fused:
        P = R.project_bin_and_sort(*args, sync=True)
    else:
        R.project(*args)
        P = R.bin_and_sort(sync=True)
    torch.cuda.synchronize()
    r = R.records()
    return dict(P=P, rec=R.rec[: wl.n * gs2d.RECORD_BYTES].cpu().numpy(),
                rect=R.rect[: wl.n].cpu().numpy(), count=R.count[: wl.n].cpu().numpy(),
                ranges=R.tile_ranges.cpu().numpy(), sorted_gid=R.sorted_gid[:P].cpu().numpy(),
                conic=r["conic"].cpu().numpy(), box_x=r["box_x"].cpu().numpy().astype(np.uint32),
                box_y=r["box_y"].cpu().numpy().astype(np.uint32))


def _same(a, b):
    assert a["P"] == b["P"]
    for k in ("rec", "rect", "count", "ranges", "sorted_gid"):
        assert np.array_equal(a[k], b[k]), k


@pytest.mark.parametrize("mode", [synth.SUM, synth.COMPOSITE])
@pytest.mark.parametrize("w,h,n,seed", [(1, 1, 3, 1), (100, 37, 300, 3), (250, 130, 3000, 5),
                                        (1040, 512, 20000, 7)])
def test_equals_separate_calls_and_oracle(mode, w, h, n, seed):
    """Ragged sizes, both modes; 1040x512 has 2112 tiles, past the counting
    sort's limit, so the radix path is covered too."""
    wl = synth.random_scene(w, h, n, seed=seed, mode=mode, diag=(0.3, 6.0), margin=6)
    f = _run(wl, True)
    _same(f, _run(wl, False))
    s = oracle_scene(wl)
    check_projection(f, s)
    check_lists(f, s)


@pytest.mark.parametrize("param", [synth.CHOLESKY, synth.SCALE_ROT])
def test_parameterizations_and_render_scale(param):
    wl = synth.random_scene(200, 150, 4000, seed=11, diag=(0.5, 5.0), param=param)
    wl.scale = 1.5
    wl.width, wl.height = 300, 225
    f = _run(wl, True)
    _same(f, _run(wl, False))
    check_lists(f, oracle_scene(wl))


def test_image_768x512_workload():
    wl = synth.image_768x512()
    f = _run(wl, True)
    _same(f, _run(wl, False))
    check_lists(f, oracle_scene(wl))


def test_no_gaussians_and_all_culled():
    wl = synth.random_scene(40, 30, 0, seed=1)
    f = _run(wl, True)
    assert f["P"] == 0 and np.all(f["ranges"] == 0)
    wl = synth.random_scene(40, 30, 50, seed=2)
    wl.xy[:] = -1000.0  # every box off screen
    f = _run(wl, True)
    assert f["P"] == 0 and np.all(f["count"] == 0) and np.all(f["ranges"] == 0)


def test_capacity_miss():
    """Too small a capacity: the synchronous call reports GS2D_ERR_CAPACITY
    and the true P, like gs2d_bin_and_sort; the retry with room succeeds."""
    wl = synth.random_scene(128, 96, 2000, seed=4, diag=(0.5, 4.0))
    P = oracle_scene(wl).num_pairs
    R = gs2d.Rasterizer(wl.width, wl.height, wl.n, wl.mode, wl.cutoff_sigma, wl.t_min,
                        pair_capacity=P // 2)
    args = (to_dev(wl.xy), to_dev(wl.chol), to_dev(wl.rgb), None, None)
    po = C.c_int64(0)
    st = gs2d.gs2d_project_bin_and_sort(R.cfg, wl.n, *args, R.rec, R.rect, R.count, R.capacity, po,
                                        R.tile_ranges, R.sorted_gid, R.workspace)
    assert st == gs2d.GS2D_ERR_CAPACITY and po.value == P
    assert R.project_bin_and_sort(*args, sync=True) == P  # grows and retries
    f = _run(wl, True, capacity=P)
    check_lists(f, oracle_scene(wl))
