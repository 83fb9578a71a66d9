"""Test-only pieces of the cluster runtime's host-logic tests.

The pods of these tests keep their arena in host memory. Their step leaf is
the function below: C = alpha*A*B + beta*C on raw row-major pointers, in fp64,
rounded to fp32 once per leaf. It exists so that planning, placement, the
FREE pass, the two-phase STORE and the re-plan after a lost node can be
checked without a GPU. The GPU tests run the same runtime with its leaves on
phobos_sgemm_ex.
"""
import ctypes
import os

import numpy as np

from language_fp32_gemm_gb300 import cluster


def _view(addr, rows, ld, cols):
    buf = (ctypes.c_float * (rows * ld)).from_address(addr)
    return np.ctypeslib.as_array(buf).reshape(rows, ld)[:, :cols]


def host_gemm(m, n, k, alpha, a, lda, b, ldb, beta, c, ldc):
    A = _view(a, m, lda, k).astype(np.float64)
    B = _view(b, k, ldb, n).astype(np.float64)
    C = _view(c, m, ldc, n)
    C[...] = (float(alpha) * (A @ B) + float(beta) * C.astype(np.float64)).astype(np.float32)


def slow_host_gemm(m, n, k, alpha, a, lda, b, ldb, beta, c, ldc):
    """host_gemm that takes 0.15 s per leaf, so a pod is still busy when the
    scheduler gives up on its heartbeat."""
    import time
    time.sleep(0.15)
    host_gemm(m, n, k, alpha, a, lda, b, ldb, beta, c, ldc)


def write_job(tmp, M, N, K, alpha, beta, seed, lo, hi=None):
    """Seeded A, B, C_old as raw fp32 files under `tmp`; returns (Job, A, B, C_old)."""
    import seeded_inputs as si
    A = si.uniform_pm1(seed, 0, (M, K))
    B = si.uniform_pm1(seed, 1, (K, N))
    C0 = si.uniform_pm1(seed, 2, (M, N))
    paths = {n: os.path.join(str(tmp), "%s.f32" % n) for n in "ABC"}
    A.tofile(paths["A"])
    B.tofile(paths["B"])
    C0.tofile(paths["C"])
    text = "\n".join([
        "source = sgemm",
        "dim M = %d" % M, "dim N = %d" % N, "dim K = %d" % K,
        "tensor A = read f32 %dx%d file://%s" % (M, K, paths["A"]),
        "tensor B = read f32 %dx%d file://%s" % (K, N, paths["B"]),
        "tensor C = readwrite f32 %dx%d file://%s" % (M, N, paths["C"]),
        "scalar alpha = f32 %r" % alpha,
        "scalar beta = f32 %r" % beta,
    ] + ["cluster TILE_%s in [%d, %d]" % (ax, l, h) for ax, l, h in zip("MNK", lo, hi or lo)])
    return cluster.parse_job(text), A, B, C0


def result(job):
    return np.fromfile(job.C.path, dtype=np.float32).reshape(job.M, job.N)
