"""Build the CUDA library in-tree: one nvcc compile per translation unit (in
parallel), then a shared-library link with the static CUDA runtime.

Output: ``paged_kv_cache_231_gb300/libpagedkv.so``. Objects and the ptxas report
(registers / spills / shared memory per kernel) go to ``paged_kv_cache_231_gb300/_build``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
INCLUDE = os.path.join(ROOT, "include")
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libpagedkv.so")
SOURCES = ["runtime.cpp", "attention.cu", "scatter.cu", "combine.cu", "sparse.cu",
           "sparse16.cu", "static_workspace.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpagedkv")


def _deps():
    files = [os.path.join(INCLUDE, "pagedkv.h")]
    files += [os.path.join(CSRC, f) for f in os.listdir(CSRC)
              if f.endswith((".h", ".cuh"))]
    return files


def _stale(target, inputs):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(f) > t for f in inputs)


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    common = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O3", "-I", INCLUDE,
              "-I", CSRC] + ARCH
    if debug:
        common += ["-DPKV_DEBUG=1"]
    # extra definitions for tuning builds, e.g. "-DPKV_DEC_STAGES=6 -DPKV_CTAS_PER_SM=1"
    common += os.environ.get("PKV_NVCC_DEFINES", "").split()
    deps = _deps()
    jobs = []
    objs = []
    for src in SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(BUILD, src + ".o")
        objs.append(obj)
        if force or _stale(obj, [path] + deps):
            cmd = [cc, "-c", path, "-o", obj] + common
            if src.endswith(".cu"):
                cmd += ["-Xptxas", "-v"]
            jobs.append((src, cmd))

    def run(job):
        src, cmd = job
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, cmd, r

    if jobs:
        with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            results = list(ex.map(run, jobs))
        report = []
        for src, cmd, r in results:
            report.append(f"== {src}\n{r.stdout}{r.stderr}")
            if r.returncode != 0:
                sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
                raise RuntimeError(f"nvcc failed for {src}")
            if verbose:
                sys.stderr.write(r.stderr)
        with open(os.path.join(BUILD, "ptxas.log"), "a") as f:
            f.write("\n".join(report))
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + ".tmp"
        cmd = [cc, "-shared", "-o", tmp] + objs + ARCH + ["-cudart", "static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
            raise RuntimeError("link of libpagedkv.so failed")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
