"""Builds libkvc.so in-tree with nvcc for sm_103a (no cmake, no torch extension).

Each .cu file under csrc/ compiles to an object in parallel, then one link
produces kv_cache_append_rope_gb300/libkvc.so (CUDA runtime linked statically,
driver entry points fetched at run time, so the library loads on a machine
without a GPU).  The same sources compiled with -DKVC_DEBUG give
libkvc_debug.so: every kernel then checks the lengths and slot indices it
derives against the capacity, recording a bit of the device error word and
skipping the access when one is out of range (the binding loads it when the
environment sets KVC_LIB=debug).
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libkvc.so")
DEBUG_LIB = os.path.join(PKG, "libkvc_debug.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc():
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkvc.so")
    return path


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(ROOT, "include", "kvc.h")]


def up_to_date(lib=LIB):
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps() + [os.path.abspath(__file__)])


def _compile(src, debug, verbose):
    out_dir = os.path.join(BUILD, "debug") if debug else BUILD
    obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-ffp-contract=off,-fno-fast-math",
           "-I" + os.path.join(ROOT, "include"), "-c", src, "-o", obj]
    if debug:
        cmd.insert(2, "-DKVC_DEBUG")
    if verbose:
        cmd.insert(2, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def _link(lib, objs):
    tmp = lib + ".tmp"
    cmd = [nvcc(), ARCH, "-shared", "-o", tmp] + objs + ["-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link of {os.path.basename(lib)} failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)


def build(force=False, verbose=False, debug=True):
    """Compile and link libkvc.so (and, with `debug`, libkvc_debug.so); returns libkvc.so's path."""
    variants = [False] + ([True] if debug else [])
    todo = [d for d in variants if force or not up_to_date(DEBUG_LIB if d else LIB)]
    if not todo:
        return LIB
    os.makedirs(os.path.join(BUILD, "debug"), exist_ok=True)
    jobs = [(s, d) for d in todo for s in sources()]
    with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 8, len(jobs))) as ex:
        results = list(ex.map(lambda j: (j[1], _compile(j[0], j[1], verbose)), jobs))
    if verbose:
        for _, (_, log) in results:
            sys.stderr.write(log)
    for d in todo:
        _link(DEBUG_LIB if d else LIB, [o for dd, (o, _) in results if dd == d])
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
