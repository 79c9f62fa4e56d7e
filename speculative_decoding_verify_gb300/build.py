"""Build libsdverify.so (CUDA, sm_103a) in-tree.

Each translation unit under csrc/ is compiled by its own nvcc process (in
parallel), then linked into one shared library next to this file.  Floating
point: no FMA contraction (``-fmad=false``) and no fast-math, so every fp32
operation the bit-exact contract names is one IEEE rounding; fused
multiply-adds appear only where the kernels call them explicitly.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libsdverify.so")
BUILD_DIR = os.path.join(ROOT, "_build")
# the bounds-checked variant (SD_DEBUG_BOUNDS), loaded by the package when SDV_DEBUG_BOUNDS=1
LIB_DBG = os.path.join(HERE, "libsdverify_dbg.so")
BUILD_DIR_DBG = os.path.join(ROOT, "_build_dbg")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_log: str | None = None,
          debug_bounds: bool | None = None) -> str:
    """Build the library (default: the variant the package loads, the bounds-checked one when
    SDV_DEBUG_BOUNDS=1) and return its path."""
    if debug_bounds is None:
        debug_bounds = os.environ.get("SDV_DEBUG_BOUNDS", "") == "1"
    build_dir, lib = (BUILD_DIR_DBG, LIB_DBG) if debug_bounds else (BUILD_DIR, LIB)
    os.makedirs(build_dir, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")]
    headers.append(os.path.join(ROOT, "include", "sdverify.h"))
    stamp = os.path.join(build_dir, "flags.txt")
    want = os.environ.get("SDV_NVCC_FLAGS", "")
    if not os.path.exists(stamp) or open(stamp).read() != want:
        force = True
        with open(stamp, "w") as f:
            f.write(want)
    srcs = sources()
    flags = ["-O3", "-std=c++17", "-lineinfo", "-fmad=false", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
             "-I", os.path.join(ROOT, "include")] + ARCH
    if ptxas_log:
        flags += ["-Xptxas", "-v"]
    extra = os.environ.get("SDV_NVCC_FLAGS", "").split()
    flags += extra
    if debug_bounds:
        flags += ["-DSD_DEBUG_BOUNDS"]
    objs = []
    jobs = []
    for s in srcs:
        o = os.path.join(build_dir, os.path.basename(s)[:-3] + ".o")
        objs.append(o)
        if force or _stale(o, [s] + headers):
            jobs.append((s, o))

    def compile_one(job):
        s, o = job
        cmd = [nvcc(), "-c", s, "-o", o + ".tmp"] + flags
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(s)}:\n{r.stdout}\n{r.stderr}")
        os.replace(o + ".tmp", o)
        return s, r.stderr

    logs = []
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
            for s, err in ex.map(compile_one, jobs):
                logs.append(f"== {os.path.basename(s)}\n{err}")
                if verbose:
                    print(f"compiled {os.path.basename(s)}", file=sys.stderr)
    if ptxas_log and logs:
        with open(ptxas_log, "w") as f:
            f.write("\n".join(logs))
    if force or jobs or _stale(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [nvcc(), "-shared", "-o", tmp] + objs + ARCH + ["-lcudart"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import argparse

    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--ptxas-log", default=None)
    ap.add_argument("--debug-bounds", action="store_true", help="the bounds-checked variant")
    a = ap.parse_args()
    print(build(force=a.force, verbose=True, ptxas_log=a.ptxas_log, debug_bounds=a.debug_bounds or None))
