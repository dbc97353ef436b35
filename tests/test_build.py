"""The build's dependency list (CPU only): every file a library source
includes is among the build's inputs, so an edit to any of them rebuilds the
library before tests or the benchmark load it."""
import os
import re

from scaled_dot_product_05_gb300 import build as cuda_build


def _local_includes(path):
    with open(path) as f:
        return re.findall(r'^\s*#\s*include\s+"([^"]+)"', f.read(), flags=re.M)


def test_every_local_include_is_a_build_input():
    inputs = {os.path.realpath(p) for p in cuda_build._inputs()}
    todo = [os.path.join(cuda_build.CSRC, f) for f in cuda_build.SOURCES]
    seen = set()
    while todo:
        src = todo.pop()
        for inc in _local_includes(src):
            dep = os.path.realpath(os.path.join(os.path.dirname(src), inc))
            assert os.path.exists(dep), f"{src} includes missing {inc}"
            assert dep in inputs, f"{inc} (included by {os.path.basename(src)}) is not a build input"
            if dep not in seen:
                seen.add(dep)
                todo.append(dep)
    # the kernels' headers are all reached
    names = {os.path.basename(p) for p in seen}
    assert {"sdpa_kernel.cuh", "sdpa_bwd.cuh", "sdpa_bwd_fp8.cuh", "ptx.cuh", "sdpa.h"} <= names


def test_a_newer_header_makes_the_build_stale(tmp_path, monkeypatch):
    lib = tmp_path / "lib.so"
    lib.write_bytes(b"")
    monkeypatch.setattr(cuda_build, "LIB_PATH", str(lib))
    newest = max(os.path.getmtime(p) for p in cuda_build._inputs())
    os.utime(lib, (newest + 10, newest + 10))
    assert cuda_build.up_to_date()
    # any header, the FP8 backward's included, newer than the library
    hdr = os.path.join(cuda_build.CSRC, "sdpa_bwd_fp8.cuh")
    os.utime(lib, (os.path.getmtime(hdr) - 10, os.path.getmtime(hdr) - 10))
    assert not cuda_build.up_to_date()
