"""Build the CUDA library ``lib/libgdn_gb300.so`` for sm_103a with nvcc.

Every ``csrc/*.cu`` file is compiled in parallel to an object, then the
objects are linked into one shared library against the shared CUDA runtime.
``checked=True`` builds ``lib/libgdn_gb300_checked.so`` instead, with
``-DGDN_CHECKED``: every kernel then checks the index ranges it derives
against its tensors' extents (GDN_ERR_BOUNDS); the package loads it when the
environment sets ``GDN_CHECKED=1``.
Usage: ``python -m gated_delta_rule_kk_gb300.build_lib [--force] [--verbose] [--checked]``.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "lib")
BUILD_DIR = os.path.join(OUT_DIR, "obj")
LIB_NAME = "libgdn_gb300.so"
LIB_PATH = os.path.join(OUT_DIR, LIB_NAME)
CHECKED_LIB_PATH = os.path.join(OUT_DIR, "libgdn_gb300_checked.so")
CHECKED_BUILD_DIR = os.path.join(OUT_DIR, "obj_checked")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + [
    "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
    "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC,
]


def _nvcc():
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found (set NVCC or put it on PATH)")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h")) + \
        [os.path.abspath(__file__)]


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        print(r.stdout + r.stderr, flush=True)
    return r


def build(force: bool = False, verbose: bool = False, extra_flags=(), checked: bool = False) -> str:
    """Compile (if stale) and return the path of the shared library (the
    checked build with ``checked=True``)."""
    lib_path = CHECKED_LIB_PATH if checked else LIB_PATH
    build_dir = CHECKED_BUILD_DIR if checked else BUILD_DIR
    if checked:
        extra_flags = (*extra_flags, "-DGDN_CHECKED")
    os.makedirs(build_dir, exist_ok=True)
    deps = _deps()
    if not force and not _stale(lib_path, deps):
        return lib_path
    nvcc = _nvcc()
    headers = [d for d in deps if not d.endswith(".cu")]
    jobs = []
    objs = []
    for src in _sources():
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or _stale(obj, [src] + headers):
            jobs.append([nvcc, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj])
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        list(ex.map(lambda c: _run(c, verbose), jobs))
    tmp = lib_path + ".tmp"
    _run([nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs], verbose)
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    p = build(force="--force" in sys.argv, verbose="--verbose" in sys.argv,
              checked="--checked" in sys.argv)
    print(p)
