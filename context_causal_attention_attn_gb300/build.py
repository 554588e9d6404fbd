"""Build libcpattn.so in-tree with nvcc for sm_103a.

Each CUDA source is compiled in parallel to an object in ``_build/`` and the
objects are linked into ``context_causal_attention_attn_gb300/libcpattn.so``.
Rebuilds only when a source or header is newer than the library.  Builds
are serialised across processes by an exclusive lock on ``_build/.lock``, so
several processes (ranks of one job, test workers) may call build() at once:
the first compiles, the others wait and find the library up to date.

``build(debug=True)`` makes the bounds-checked library ``libcpattn_debug.so``
instead (sources compiled with ``-DCP_DEBUG_BOUNDS`` into ``_build/debug/``):
its kernels check every tile and row they touch against the tensors' extents
and report a failure through ``cp_check_device_error``.  The binding loads it
in place of the release library when the environment has ``CPATTN_DEBUG=1``.

    python -m context_causal_attention_attn_gb300.build [--force] [--debug]
"""

import concurrent.futures as cf
import contextlib
import fcntl
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libcpattn.so")
LIB_DEBUG = os.path.join(PKG, "libcpattn_debug.so")
DEBUG_FLAGS = ["-DCP_DEBUG_BOUNDS"]


def lib_path(debug=False):
    return LIB_DEBUG if debug else LIB


ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-I" + CSRC, "-I" + INCLUDE]


def nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(
        os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h")) + [__file__]


def up_to_date(debug=False):
    lib = lib_path(debug)
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def _compile(src, extra, debug=False):
    obj_dir = os.path.join(BUILD, "debug") if debug else BUILD
    os.makedirs(obj_dir, exist_ok=True)
    obj = os.path.join(obj_dir, os.path.basename(src) + ".o")
    cmd = [nvcc()] + ARCH + NVCC_FLAGS + (DEBUG_FLAGS if debug else []) + extra + [
        "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


@contextlib.contextmanager
def _locked():
    os.makedirs(BUILD, exist_ok=True)
    with open(os.path.join(BUILD, ".lock"), "w") as f:
        fcntl.flock(f, fcntl.LOCK_EX)
        try:
            yield
        finally:
            fcntl.flock(f, fcntl.LOCK_UN)


def build(force=False, verbose=False, extra=(), debug=False):
    """Compile and link; returns the path of the library (the bounds-checked
    one with debug=True)."""
    if not force and up_to_date(debug):
        return lib_path(debug)
    with _locked():
        if not force and up_to_date(debug):
            return lib_path(debug)
        return _build(verbose, extra, debug)


def _build(verbose, extra, debug=False):
    extra = list(extra)
    with cf.ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        results = list(ex.map(lambda s: _compile(s, extra, debug), sources()))
    objs = [o for o, _ in results]
    if verbose:
        for _, err in results:
            if err:
                sys.stderr.write(err)
    lib = lib_path(debug)
    tmp = lib + ".tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    force = "--force" in sys.argv
    verbose = "-v" in sys.argv
    extra = ["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else []
    print(build(force=force or bool(extra), verbose=verbose or bool(extra), extra=extra,
                debug="--debug" in sys.argv))
