"""Builds libpaged_gqa_decode.so in-tree (``_build/``) with nvcc for sm_103a.

Each .cu translation unit compiles in its own nvcc process, in parallel; the
objects are linked into one shared library whose only dependencies are the C
and C++ runtimes (cudart is linked statically and reaches the driver at run
time), so it loads on a machine without a GPU.
"""
from __future__ import annotations

import concurrent.futures
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB_NAME = "libpaged_gqa_decode.so"
LIB_PATH = os.path.join(BUILD, LIB_NAME)
# The checked build (-DPGD_CHECKED): every global index and TMA coordinate of
# the kernels is range-checked; a violation raises DECODE_ATTN_DEV_CHECK and
# skips the access.  A stand-in for a memory checker, for tests on small
# cases; selected at load time with DECODE_ATTN_CHECKED=1.
BUILD_CHECKED = os.path.join(HERE, "_build_checked")
LIB_CHECKED_NAME = "libpaged_gqa_decode_checked.so"
LIB_CHECKED_PATH = os.path.join(BUILD_CHECKED, LIB_CHECKED_NAME)


def checked_requested() -> bool:
    return os.environ.get("DECODE_ATTN_CHECKED") == "1"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "--expt-relaxed-constexpr", "-Xptxas", "-v"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found")
    return path


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (glob.glob(os.path.join(CSRC, "*")) +
            [os.path.join(os.path.dirname(HERE), "include", "decode_attn.h")])


def _up_to_date(lib: str) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _deps())


def _compile(src: str, out_dir: str, extra: tuple) -> tuple[str, str]:
    obj = os.path.join(out_dir, os.path.basename(src) + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    with open(obj + ".ptxas.txt", "w") as f:  # register / spill / smem report
        f.write(r.stderr)
    return obj, r.stderr


def build(force: bool = False, verbose: bool = False, checked=None) -> str:
    """Compile every .cu under csrc/ and link the shared library (the checked
    build when ``checked``, by default when DECODE_ATTN_CHECKED=1)."""
    if checked is None:
        checked = checked_requested()
    out_dir, lib = (BUILD_CHECKED, LIB_CHECKED_PATH) if checked else (BUILD, LIB_PATH)
    extra = ("-DPGD_CHECKED",) if checked else ()
    os.makedirs(out_dir, exist_ok=True)
    if not force and _up_to_date(lib):
        return lib
    srcs = _sources()
    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, len(srcs))) as ex:
        results = list(ex.map(lambda s: _compile(s, out_dir, extra), srcs))
    if verbose:
        for _, log in results:
            print(log)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))
