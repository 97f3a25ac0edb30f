"""Build libla.so in-tree with nvcc for sm_103a (no torch extension machinery).

Each .cu file under csrc/ compiles to an object in parallel; the objects link
into ``_lib/libla.so`` with the CUDA runtime linked statically, so the library
depends only on the driver at run time.  ``build_library()`` rebuilds only when
a source or header is newer than the library.

``build_library(debug=True)`` builds ``_lib/libla_debug.so`` beside it: the same
sources with ``-DLA_DEBUG`` and relocatable device code, which turns on the
kernels' device-side index checks (LA_DCHECK: a failed check records
LA_ERR_BOUNDS and its source line, and skips the access).  The binding loads it
instead of the regular library when the environment has LA_DEBUG=1.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
DEBUG_BUILD_DIR = os.path.join(PKG, "_build_debug")
LIB_DIR = os.path.join(PKG, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libla.so")
DEBUG_LIB_PATH = os.path.join(LIB_DIR, "libla_debug.so")
DEBUG_FLAGS = ["-DLA_DEBUG", "-rdc=true"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
                     "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h")) + [__file__]


def lib_path(debug: bool = False) -> str:
    return DEBUG_LIB_PATH if debug else LIB_PATH


def needs_build(debug: bool = False) -> bool:
    path = lib_path(debug)
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    return any(os.path.getmtime(p) > t for p in _deps())


def nvcc_command(src: str, obj: str, extra=(), debug: bool = False):
    """The nvcc command line that compiles one source (the debug flags added when asked)."""
    return [nvcc(), *NVCC_FLAGS, *(DEBUG_FLAGS if debug else []), *extra, "-c", src, "-o", obj]


def _compile(src: str, extra, debug: bool) -> str:
    obj = os.path.join(DEBUG_BUILD_DIR if debug else BUILD_DIR, os.path.splitext(os.path.basename(src))[0] + ".o")
    cmd = nvcc_command(src, obj, extra, debug)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, " ".join(cmd), r.stderr))
    return obj


def build_library(force: bool = False, verbose: bool = False, extra_flags=(), debug: bool = False) -> str:
    """Compile every csrc/*.cu and link _lib/libla.so (or _lib/libla_debug.so); return its path."""
    path = lib_path(debug)
    if not force and not needs_build(debug):
        return path
    os.makedirs(DEBUG_BUILD_DIR if debug else BUILD_DIR, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(lambda s: _compile(s, list(extra_flags), debug), srcs))
    tmp = path + ".tmp%d" % os.getpid()
    cmd = [nvcc(), *ARCH, *(["-rdc=true"] if debug else []), "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
    os.replace(tmp, path)
    if verbose:
        print("built", path)
    return path


if __name__ == "__main__":
    import sys
    build_library(force=True, verbose=True, debug="--debug" in sys.argv)
