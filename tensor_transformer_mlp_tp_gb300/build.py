"""Build ``libtpmlp.so`` in-tree: every CUDA source for sm_103a, compiled in parallel.

``python -m tensor_transformer_mlp_tp_gb300.build`` (or ``build()``) compiles
``csrc/*.cu`` with ``nvcc -gencode arch=compute_103a,code=sm_103a -O3 -lineinfo``
into ``_build/`` and links the shared library next to this file.  The CUDA
runtime is linked statically and only the ``tpmlp_*`` symbols are exported,
so the library's runtime cannot be interposed by another copy loaded in the
same process (torch's).  Rebuilds only what changed.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libtpmlp.so")
# The debug build: the same sources with -DTPMLP_DEBUG_BOUNDS (bounds checks on hand-computed global indices)
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libtpmlp_debug.so")
INCLUDE = os.path.join(ROOT, "include")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "-I", INCLUDE, "-I", CSRC] + ARCH


def nvcc() -> str:
    cand = [os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"]
    for c in cand:
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtpmlp")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    return hs + [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]


def _mtime(p):
    return os.stat(p).st_mtime


def _compile(src: str, obj: str, verbose: bool, extra=()) -> str:
    cmd = [nvcc()] + NVCC_FLAGS + list(extra) + ["-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    return r.stderr


def build(force: bool = False, verbose: bool = False, debug_bounds: bool = False) -> str:
    """Compile and link libtpmlp.so (with `debug_bounds`, libtpmlp_debug.so: the bounds-checked debug build);
    returns its path."""
    bdir, lib = (BUILD_DEBUG, LIB_DEBUG) if debug_bounds else (BUILD, LIB)
    extra = ["-DTPMLP_DEBUG_BOUNDS"] if debug_bounds else []
    os.makedirs(bdir, exist_ok=True)
    srcs = _sources()
    newest_header = max(_mtime(h) for h in _headers())
    jobs = []
    objs = []
    for src in srcs:
        obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or not os.path.exists(obj) or _mtime(obj) < max(_mtime(src), newest_header):
            jobs.append((src, obj))
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
            for log in ex.map(lambda j: _compile(j[0], j[1], verbose, extra), jobs):
                if verbose and log:
                    sys.stderr.write(log)
    if force or jobs or not os.path.exists(lib) or _mtime(lib) < max(_mtime(o) for o in objs):
        exports = os.path.join(bdir, "exports.map")
        with open(exports, "w") as fh:
            fh.write("{ global: tpmlp_*; local: *; };\n")
        tmp = lib + ".tmp"
        cmd = [nvcc(), "-shared", "-cudart", "static"] + ARCH + objs + [
            "-Xlinker", f"--version-script={exports}", "-Xlinker", "--no-undefined", "-o", tmp]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug_bounds="--debug-bounds" in sys.argv))
