"""Builds liblssar_attn_fwd.so in-tree with nvcc for sm_103a.

Every ``csrc/*.cu`` is compiled to an object under ``_build/`` (in parallel,
skipped when up to date) and linked into ``lssar_attn_fwd_gb300/_lib/``.
``debug=True`` builds liblssar_attn_fwd_debug.so instead (objects under
``_build_debug/``), compiled with -DLSSAR_DEBUG_CHECKS: the kernels check
their tensor-copy coordinates, TMEM lane and column ranges, work items and
global-store indices, and record a code (101-105) in the device error word
instead of making the access.
Usage: ``python -m lssar_attn_fwd_gb300.build [--force] [--verbose] [--debug]``.
"""

import concurrent.futures
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD_DIR = os.path.join(ROOT, "_build")
DEBUG_BUILD_DIR = os.path.join(ROOT, "_build_debug")
LIB_DIR = os.path.join(PKG, "_lib")
LIB_NAME = "liblssar_attn_fwd.so"
DEBUG_LIB_NAME = "liblssar_attn_fwd_debug.so"
DEBUG_FLAGS = ["-DLSSAR_DEBUG_CHECKS"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path():
    exe = shutil.which("nvcc")
    if exe:
        return exe
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found")


def lib_path(debug=False):
    return os.path.join(LIB_DIR, DEBUG_LIB_NAME if debug else LIB_NAME)


def _flags(extra=()):
    return ARCH + [
        # -fno-gnu-unique: function-local statics of template functions (the
        # per-device attribute flags of each kernel instance) stay private to
        # this library instead of being merged with another loaded build's
        "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2,-fno-gnu-unique",
        "-I", os.path.join(ROOT, "include"), "-I", CSRC,
    ] + list(extra)


def _newest_header():
    hs = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(ROOT, "include", "*.h"))
    return max((os.path.getmtime(h) for h in hs), default=0.0)


def build(force=False, verbose=False, ptxas_verbose=False, debug=False):
    """Compile and link the library (the debug-check variant with debug=True);
    returns its path."""
    nvcc = nvcc_path()
    build_dir = DEBUG_BUILD_DIR if debug else BUILD_DIR
    os.makedirs(build_dir, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    if not sources:
        raise RuntimeError("no CUDA sources found")
    hdr_time = _newest_header()
    extra = (["-Xptxas", "-v"] if ptxas_verbose else []) + (DEBUG_FLAGS if debug else [])
    jobs = []
    objects = []
    for src in sources:
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        objects.append(obj)
        if (force or not os.path.exists(obj) or os.path.getmtime(obj) < max(os.path.getmtime(src), hdr_time)):
            jobs.append([nvcc] + _flags(extra) + ["-c", src, "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    if jobs:
        with concurrent.futures.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for cmd, r in ex.map(run, jobs):
                if verbose or ptxas_verbose or r.returncode != 0:
                    sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
                if r.returncode != 0:
                    raise RuntimeError(f"nvcc failed for {cmd[-3]}")
    out = lib_path(debug)
    if jobs or not os.path.exists(out):
        tmp = out + ".tmp"
        # -Bsymbolic and --exclude-libs: the library binds its own functions and
        # its statically linked CUDA runtime to itself, so that two builds
        # (default and debug) can be loaded in one process side by side
        cmd = [nvcc] + ARCH + ["-shared", "-Xlinker", "-Bsymbolic", "-Xlinker", "--exclude-libs,ALL",
                               "-o", tmp] + objects
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
            raise RuntimeError("link failed")
        os.replace(tmp, out)
    return out


if __name__ == "__main__":
    p = build(force="--force" in sys.argv, verbose="--verbose" in sys.argv,
              ptxas_verbose="--ptxas" in sys.argv, debug="--debug" in sys.argv)
    print(p)
