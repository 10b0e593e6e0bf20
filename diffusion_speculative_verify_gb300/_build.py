"""Builds libsimsd.so in-tree with nvcc for sm_103a (one -gencode, parallel compiles).

`build(checked=True)` builds libsimsd_checked.so instead: the same sources compiled with
SIMSD_CHECKED, where every kernel checks each global index against its array's extent and
reports a violation in the device error word (SIMSD_DEVERR_BOUNDS); tests use it in place
of a memory checker."""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libsimsd.so")
BUILD_CHECKED = os.path.join(PKG, "_build_checked")
LIB_CHECKED = os.path.join(PKG, "libsimsd_checked.so")
SOURCES = ["layout.cu", "attn_simt.cu", "attn_tc.cu", "accept.cu", "route.cu", "api.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _newer(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, force: bool = False, extra_flags=None, checked: bool = False) -> str:
    nvcc = _nvcc()
    build_dir = BUILD_CHECKED if checked else BUILD
    lib = LIB_CHECKED if checked else LIB
    os.makedirs(build_dir, exist_ok=True)
    headers = [os.path.join(INCLUDE, "simsd.h")] + [
        os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")]
    flags = NVCC_FLAGS + (["-DSIMSD_CHECKED"] if checked else []) + list(extra_flags or [])
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(build_dir, src.replace(".cu", ".o"))
        if force or _newer(o, [s] + headers):
            jobs.append([nvcc] + ARCH + flags + ["-c", s, "-o", o])
    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return cmd
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        list(ex.map(run, jobs))
    objs = [os.path.join(build_dir, s.replace(".cu", ".o")) for s in SOURCES]
    if force or jobs or _newer(lib, objs):
        run([nvcc] + ARCH + ["-shared", "-o", lib] + objs + ["-cudart", "static", "-ldl"])
    return lib


if __name__ == "__main__":
    print(build(verbose=True, force="--force" in sys.argv, checked="--checked" in sys.argv))
