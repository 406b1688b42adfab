"""Build libpagedkv.so in-tree (sm_103a), compiling translation units in parallel.

Usage: ``python -m paged_kv_cache_259_gb300.build`` or ``build_library()``.
The library lands next to this file; objects go to ``_build/`` (both ignored by git).
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libpagedkv.so")

CUDA_SOURCES = [
    "pkv_status.cu",
    "pkv_cache_ops.cu",
    "pkv_decode.cu",
    "pkv_decode_f32.cu",
    "pkv_decode_bf16.cu",
    "pkv_decode_e4m3.cu",
    "pkv_decode_noalloc.cu",
    "pkv_prefill.cu",
    "pkv_pipeline.cu",
]
CXX_SOURCES = ["block_manager.cpp"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
                     "--expt-relaxed-constexpr", "-Xptxas", "-v"]
CXX_FLAGS = ["-O2", "-fPIC", "-fvisibility=hidden", "-std=c++17", "-Wall"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _run(cmd, log):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    with open(log, "w") as f:
        f.write(" ".join(cmd) + "\n" + r.stdout)
    if r.returncode != 0:
        raise RuntimeError(f"build step failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout[-4000:]}")
    return r.stdout


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build_library(force=False, verbose=False):
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(os.path.dirname(HERE), "include", "pagedkv.h"))
    jobs = []
    objs = []
    for src in CUDA_SOURCES + CXX_SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(BUILD, src + ".o")
        objs.append(obj)
        if force or _stale(obj, [path] + headers):
            if src.endswith(".cu"):
                cmd = [nvcc] + NVCC_FLAGS + ["-c", path, "-o", obj]
            else:
                cmd = ["g++"] + CXX_FLAGS + ["-c", path, "-o", obj]
            jobs.append((cmd, obj + ".log"))
    with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        outs = list(ex.map(lambda j: _run(*j), jobs))
    if verbose:
        for o in outs:
            print(o)
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + ".tmp"
        _run([nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs,
             os.path.join(BUILD, "link.log"))
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose="-v" in sys.argv))
