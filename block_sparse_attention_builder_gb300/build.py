"""Builds libmxsa.so in-tree for sm_103a with nvcc (one -gencode, the
translation units compiled in parallel, then linked against the shared CUDA
runtime so the library and PyTorch share one runtime instance)."""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libmxsa.so")
# A second library for the wait-limit test only: every on-device wait gives
# up after 50 ms, and a switch (mxsa_test_skip_barrier_arrival) keeps one CTA
# of the plan launch from arriving at a grid barrier.  Never loaded by the
# package itself.
TEST_LIB = os.path.join(OUT_DIR, "libmxsa_test.so")
TEST_FLAGS = ["-DMXSA_TEST_HOOKS", "-DMXSA_WAIT_LIMIT_NS=50000000ull"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    n = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(n):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libmxsa")
    return n


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + [
        os.path.join(ROOT, "include", "mxsa.h"), os.path.abspath(__file__)]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    """libmxsa.so, and the wait-limit test's library beside it."""
    _build_one(LIB, (), "", force, verbose)
    _build_one(TEST_LIB, TEST_FLAGS, "test_", force, verbose)
    return LIB


def _build_one(lib: str, extra_flags, obj_prefix: str, force: bool, verbose: bool) -> str:
    if not force and up_to_date(lib):
        return lib
    os.makedirs(OUT_DIR, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(OUT_DIR, obj_prefix + os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        objs = list(ex.map(compile_one, _sources()))
    tmp = lib + f".tmp{os.getpid()}"
    cudalib = os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")
    r = subprocess.run([nvcc, *ARCH, "-shared", "-cudart", "shared", "-Xlinker", "-rpath", "-Xlinker", cudalib,
                        "-o", tmp, *objs], capture_output=True,
                       text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))
