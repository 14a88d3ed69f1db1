"""The kernel trace (gs2d_trace_begin / gs2d_trace_end) on the GPU: it names
every kernel a call launches, its events bracket each kernel (positive,
ordered durations that fit inside the step), it works eagerly and under
CUDA-graph capture, and it changes no result."""
import numpy as np
import pytest
import torch

from raster_gaussian_02_b300 import gs2d, synth

pytestmark = pytest.mark.gpu


def _setup(mode=synth.SUM):
    wl = synth.random_scene(200, 136, 3000, seed=77, mode=mode)
    dev = torch.device("cuda:0")
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    R = gs2d.Rasterizer(wl.width, wl.height, wl.n, wl.mode, device=dev)
    args = (t(wl.xy), t(wl.chol), t(wl.rgb), t(wl.depth), t(wl.opacity))
    R.project_bin_and_sort(*args, sync=True)
    target = t(wl.target)
    return R, args, target, t(wl.background)


def _outputs(R):
    return [x.clone() for x in (R.image, R.loss, R.d_xy, R.d_shape, R.d_rgb)]


@pytest.mark.parametrize("mode", [synth.SUM, synth.COMPOSITE])
def test_trace_names_every_kernel_and_changes_nothing(mode):
    R, args, target, bg = _setup(mode)

    def step():
        R.project_bin_and_sort(*args, sync=False)
        R.render_fwd_bwd_l2(target, bg)
    step()
    torch.cuda.synchronize()
    ref = _outputs(R)
    tr = gs2d.KernelTrace(32)
    with tr:
        step()
    torch.cuda.synchronize()
    for a, b in zip(ref, _outputs(R)):
        assert torch.equal(a, b)
    assert tr.launched == len(tr.names) >= 4
    assert all(n and n.startswith("k_") for n in tr.names), tr.names
    assert any(n.startswith("k_gather") for n in tr.names)
    want = "k_fused_comp" if mode == synth.COMPOSITE else "k_render_bwd_sum"
    assert any(n.startswith(want) for n in tr.names), tr.names
    d = tr.durations()
    assert all(ms > 0 for _, ms in d)
    # the events are recorded in stream order: each kernel starts after the last ended
    for i in range(1, len(d)):
        assert tr.events[2 * i - 1].elapsed_time(tr.events[2 * i]) >= 0
    assert gs2d.gs2d_trace_end() == 0  # no trace active any more


def test_trace_under_graph_capture():
    R, args, target, bg = _setup()
    s = torch.cuda.Stream()
    tr = gs2d.KernelTrace(32)

    def step():
        with tr:
            R.project_bin_and_sort(*args, sync=False)
            R.render_fwd_bwd_l2(target, bg)
    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    names = list(tr.names)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        for _ in range(3):
            a.record(s)
            g.replay()
            b.record(s)
    torch.cuda.synchronize()
    d = tr.durations()
    assert [n for n, _ in d] == names and len(names) >= 4
    assert all(ms > 0 for _, ms in d)
    total = sum(ms for _, ms in d)
    assert total <= a.elapsed_time(b) * 1.01 + 1e-3
