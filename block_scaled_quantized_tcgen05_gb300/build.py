"""Build the C-ABI shared library ``libqgemm.so`` in-tree with nvcc for sm_103a.

Each translation unit under ``csrc/`` is compiled in parallel to an object file, then the objects
are linked into ``_build/libqgemm.so`` (CUDA runtime linked statically, so the library loads on a
machine without a GPU driver and every CUDA call then fails with a clean error).

``build(debug=True)`` builds the same sources with ``-DQGEMM_DEBUG`` into
``_build/debug/libqgemm_debug.so``: every kernel then checks its own index arithmetic (TMA
coordinates, scale-plane and workspace offsets, TMEM columns) and reports a failed check in the
device error word instead of making the access (``csrc/qgemm_debug.cuh``).  The binding loads it
when the environment variable ``QGEMM_DEBUG`` is ``1``.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libqgemm.so")
DEBUG_BUILD_DIR = os.path.join(BUILD_DIR, "debug")
DEBUG_LIB_PATH = os.path.join(DEBUG_BUILD_DIR, "libqgemm_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    return "nvcc"


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def up_to_date(debug: bool = False) -> bool:
    lib = DEBUG_LIB_PATH if debug else LIB_PATH
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          debug: bool = False) -> str:
    out_dir, lib_path = (DEBUG_BUILD_DIR, DEBUG_LIB_PATH) if debug else (BUILD_DIR, LIB_PATH)
    if not force and up_to_date(debug):
        return lib_path
    os.makedirs(out_dir, exist_ok=True)
    common = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "-I", INCLUDE, "-I", CSRC]
    if debug:
        common += ["-DQGEMM_DEBUG"]
    if ptxas_info:
        common += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
        cmd = common + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        results = list(ex.map(compile_one, _sources()))
    objs = []
    for src, obj, r in results:
        if verbose or ptxas_info or r.returncode:
            sys.stderr.write(r.stdout + r.stderr)
        if r.returncode:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}")
        objs.append(obj)
    tmp = lib_path + f".tmp{os.getpid()}"
    link = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("nvcc link failed")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                debug="--debug" in sys.argv))
