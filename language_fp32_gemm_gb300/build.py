"""Build ``libphobos_gemm.so`` in-tree with nvcc for sm_103a only.

Each CUDA translation unit is compiled in parallel, then linked into one
shared library next to this file (static CUDA runtime; the driver API is
reached through the runtime's entry-point query, so the library loads on a
host without a GPU).
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIBRARY = os.path.join(HERE, "libphobos_gemm.so")
SOURCES = ["phobos_gemm.cu", "sgemm_tc.cu", "sgemm_ffma.cu", "split.cu", "noalloc.cu",
           "cluster_plan.cc", "cluster_pod.cu"]
HEADERS = ["ptx.cuh", "internal.h", "host_rules.h", "cluster_internal.h",
           os.path.join("..", "..", "include", "phobos_gemm.h"),
           os.path.join("..", "..", "include", "phobos_cluster.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "--expt-relaxed-constexpr"]


def nvcc():
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found")
    return path


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force=False, verbose=False, extra_flags=()):
    """Compile and link the library if any source changed; return its path."""
    os.makedirs(BUILD, exist_ok=True)
    headers = [os.path.normpath(os.path.join(CSRC, h)) for h in HEADERS]
    objects, jobs = [], []
    for src in SOURCES:
        src_path = os.path.join(CSRC, src)
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        objects.append(obj)
        if force or _stale(obj, [src_path] + headers):
            cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra_flags, "-c", src_path, "-o", obj]
            jobs.append(cmd)

    def run(cmd):
        if verbose:
            print(" ".join(cmd), flush=True)
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("nvcc failed:\n%s\n%s%s" % (" ".join(cmd), res.stdout, res.stderr))
        if verbose and (res.stdout or res.stderr):
            print(res.stdout + res.stderr, flush=True)

    if jobs:
        with ThreadPoolExecutor(len(jobs)) as pool:
            list(pool.map(run, jobs))
    if force or jobs or _stale(LIBRARY, objects):
        tmp = LIBRARY + ".tmp%d" % os.getpid()
        run([nvcc(), *ARCH, "-shared", "-o", tmp, *objects, "-cudart", "static"])
        os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
