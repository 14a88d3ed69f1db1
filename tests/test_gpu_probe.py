"""The FP32 / SFU throughput probes (libgs2d_probe.so) on the GPU: they run,
write finite values, and measure rates of the order of the peaks derived
from the SM count, the lanes per SM and the maximum SM clock (a measured
rate far above the derived peak would mean the arithmetic was dropped)."""
import ctypes as C
import math

import pytest
import torch

from raster_gaussian_02_b300 import build as lib_build

pytestmark = pytest.mark.gpu


def test_probes_run_and_rates_are_plausible():
    import bench
    props = torch.cuda.get_device_properties(0)
    got = bench.probe_peaks(torch.device("cuda:0"), props.multi_processor_count)
    sm_mhz = 2032.0
    fp32 = props.multi_processor_count * 128 * 2 * sm_mhz * 1e6 / 1e12
    sfu = props.multi_processor_count * 32 * sm_mhz * 1e6  # 32 ex2 per SM per clock
    assert 0.3 * fp32 < got["fp32_tflops"] < 1.2 * fp32, (got, fp32)
    assert 0.3 * sfu < got["ex2_per_s"] < 1.2 * sfu, (got, sfu)


def test_probe_outputs_are_the_chains():
    """A few chains checked against the same recurrences on the host."""
    L = C.CDLL(lib_build.build_probe())
    L.gs2d_probe_fp32_fma.argtypes = [C.c_void_p, C.c_int32, C.c_int32, C.c_float, C.c_float, C.c_void_p]
    L.gs2d_probe_ex2.argtypes = [C.c_void_p, C.c_int32, C.c_int32, C.c_void_p]
    out = torch.empty(256, dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert L.gs2d_probe_fp32_fma(out.data_ptr(), 1, 10, 0.5, 1.0, s) == 0
    torch.cuda.synchronize()
    t = 5
    want = 0.0
    for j in range(8):
        a = (t + j) * 1e-3
        for _ in range(10):
            a = a * 0.5 + 1.0
        want += a
    assert math.isclose(out[t].item(), want, rel_tol=1e-5)
    assert L.gs2d_probe_ex2(out.data_ptr(), 1, 20, s) == 0
    torch.cuda.synchronize()
    want = 0.0
    for j in range(8):
        a = (t + j) * 1e-3
        for _ in range(20):
            a = 2.0 ** (-a)
        want += a
    assert math.isclose(out[t].item(), want, rel_tol=1e-4)
