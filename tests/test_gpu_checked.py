"""The parity scenarios again, against the bounds-checked build
(libgs2d_checked.so, compiled with GS2D_CHECKS), in a child process.

In that build every index the kernels take from data is tested before the
access it guards, and a failed test sets a bit in a device word instead of
touching memory.  The child runs the sum, composite, fused, absgrad, merge,
scale-rotation and combined projection + binning parity tests with
GS2D_CHECKED=1; the autouse fixture in conftest.py reads the word after each
test and fails the test unless it is zero.  The results must
also still match the oracle, so a check that fired would show up twice.
"""
import os
import subprocess
import sys

import pytest

from raster_gaussian_02_b300 import build, gs2d

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_checked_build_parity():
    build.build(checked=True)
    env = dict(os.environ, GS2D_CHECKED="1")
    files = ["tests/test_gpu_parity.py", "tests/test_gpu_fused.py", "tests/test_gpu_absgrad.py",
             "tests/test_gpu_merge.py", "tests/test_gpu_scale_rot.py",
             "tests/test_gpu_project_bin.py"]
    r = subprocess.run([sys.executable, "-m", "pytest", *files, "-x", "-q", "-m", "gpu",
                        "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]


def test_normal_build_has_no_checks():
    """The normal library reports that it carries no checks."""
    assert not gs2d.CHECKED
    st, word = gs2d.gs2d_debug_check_word()
    assert st == gs2d.GS2D_ERR_UNSUPPORTED and word == 0
