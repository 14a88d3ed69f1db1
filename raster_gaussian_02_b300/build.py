"""Builds the CUDA library raster_gaussian_02_b300/libgs2d.so for sm_103a.

nvcc compiles each csrc/*.cu to an object (in parallel) and links them into
one shared library with the CUDA runtime linked statically, so the library
needs only the driver at run time.  Objects live under _build/ (ignored).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJDIR = os.path.join(ROOT, "_build", "gs2d")
LIB = os.path.join(HERE, "libgs2d.so")
# The checked build (-DGS2D_CHECKS): every data-dependent index is tested
# before use and failures are recorded in device check words (for tests).
OBJDIR_CHECKED = os.path.join(ROOT, "_build", "gs2d_checked")
LIB_CHECKED = os.path.join(HERE, "libgs2d_checked.so")

# The FP32 / SFU throughput probes behind the roofline's peaks
# (include/gs2d_probe.h): a separate library, not part of the rasterizer.
PROBE_SRC = os.path.join(HERE, "probe", "peak_probe.cu")
LIB_PROBE = os.path.join(HERE, "libgs2d_probe.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "--expt-relaxed-constexpr", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + [os.path.join(INCLUDE, "gs2d.h")]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def _compile(src: str, verbose: bool, checked: bool = False) -> str:
    obj = os.path.join(OBJDIR_CHECKED if checked else OBJDIR, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *(["-DGS2D_CHECKS"] if checked else []), "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and r.stderr:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    lib = LIB_CHECKED if checked else LIB
    if not force and up_to_date(lib):
        return lib
    os.makedirs(OBJDIR_CHECKED if checked else OBJDIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, checked), _sources()))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def build_probe(force: bool = False) -> str:
    deps = [PROBE_SRC, os.path.join(INCLUDE, "gs2d_probe.h")]
    if (not force and os.path.exists(LIB_PROBE) and
            all(os.path.getmtime(p) <= os.path.getmtime(LIB_PROBE) for p in deps)):
        return LIB_PROBE
    tmp = LIB_PROBE + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-shared", "-cudart", "static", PROBE_SRC, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"probe build failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PROBE)
    return LIB_PROBE


if __name__ == "__main__":
    if "--probe" in sys.argv:
        print(build_probe(force="--force" in sys.argv))
    else:
        print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                    checked="--checked" in sys.argv))
