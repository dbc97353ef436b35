"""Build the CUDA library ``_build/libsdpa_gb300.so`` in-tree (nvcc, sm_103a)."""
from __future__ import annotations

import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libsdpa_gb300.so")
# the same sources built with -DSDPA_WAIT_TEST: a test-only library whose wait
# limit and one withheld K copy are set from the host (bounded-wait tests)
WAIT_TEST_LIB_PATH = os.path.join(BUILD_DIR, "libsdpa_gb300_waittest.so")
SOURCES = ["sdpa_api.cu"]
NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
              "-Xcompiler", "-fPIC", "-shared"]


def headers():
    """Every header the library's sources can include: all of csrc/*.cuh and
    the public headers under include/."""
    inc = os.path.join(ROOT, "include")
    return sorted([os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))] +
                  [os.path.join(inc, f) for f in os.listdir(inc) if f.endswith(".h")])


def _inputs():
    return [os.path.join(CSRC, f) for f in SOURCES] + headers()


def up_to_date(path: str = None) -> bool:
    path = path or LIB_PATH
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def _compile(path: str, extra, verbose: bool) -> str:
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    if not os.path.exists(nvcc):
        nvcc = "nvcc"
    tmp = path + f".tmp{os.getpid()}"
    cmd = [nvcc, *NVCC_FLAGS, *extra, *(["-Xptxas", "-v"] if verbose else []), "-o", tmp,
           *[os.path.join(CSRC, f) for f in SOURCES]]
    subprocess.run(cmd, check=True)
    os.replace(tmp, path)
    return path


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library unless it is newer than every source."""
    if not force and up_to_date():
        return LIB_PATH
    return _compile(LIB_PATH, [], verbose)


def build_wait_test(force: bool = False) -> str:
    """Compile the test-only library (SDPA_WAIT_TEST) unless it is current."""
    if not force and up_to_date(WAIT_TEST_LIB_PATH):
        return WAIT_TEST_LIB_PATH
    return _compile(WAIT_TEST_LIB_PATH, ["-DSDPA_WAIT_TEST"], False)


if __name__ == "__main__":
    print(build(force=True, verbose=True))
