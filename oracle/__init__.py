"""CPU oracle for the fp32 GEMM ``C = alpha*A*B + beta*C_old`` (row-major).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The product library never
imports this package, and this package imports nothing from the product.

The arithmetic lives in ``sgemm_oracle.c`` (plain C, fp64 accumulation over k
ascending); this module only marshals numpy arrays into it and states the
acceptance rule.  Definition followed: the ``matmul`` listing of the
"@cluster" attribute page ("What the cluster compiler accepts") and the
"Matrix Multiplication" section of "Show HN: Phobos - A tiny scale-free kernel
language with tile-DAG support".

Acceptance rule (the error scale is the oracle's ``den``):
    err = max_ij |C[i,j] - ref64[i,j]| / den[i,j]
with entries where den == 0 required to equal ``float32(ref64)`` exactly and
any NaN failing.  Bounds: 2**-20 for the split-TF32 (3xTF32), FFMA and
K-chunked modes, 2**-10 for single-pass TF32.  The fp16/bf16-input mode is
checked against the oracle of its rounded inputs (``round_inputs``) with
2**-13, and against the fp32 inputs with 2**-9 (fp16) or 2**-6 (bf16).
"""
import ctypes
import os

import numpy as np

from . import build as _build

TOL_FP32 = 2.0 ** -20   # 3xTF32, FFMA, K-chunked
TOL_TF32 = 2.0 ** -10   # single-pass TF32
# fp16 / bf16 inputs (the reduced-precision tensor-core mode).  Against the
# oracle of the rounded inputs, only the fp32 accumulation differs: partial sums
# of K = 512 added by truncating fp32 adds (<= 512 * 2^-23 = 2^-14 of sum|ab|),
# then added with round-to-nearest (< 2^-18 for K up to 2^16) and scaled once.
TOL_HALF_ACC = 2.0 ** -13
# Against the oracle of the fp32 inputs, each product r(a) r(b) differs from a b
# by at most (2u + u^2)|ab|, u = 2^-11 (fp16) or 2^-8 (bf16), plus the above.
TOL_FP16 = 2.0 ** -9
TOL_BF16 = 2.0 ** -6

_lib = None


def load_library(path):
    """Open an oracle shared library at ``path`` and declare its signatures."""
    lib = ctypes.CDLL(path)
    i64, f32, i32 = ctypes.c_int64, ctypes.c_float, ctypes.c_int
    vp = ctypes.c_void_p
    lib.oracle_sgemm.argtypes = [i64, i64, i64, f32, vp, i64, vp, i64, f32,
                                 vp, i64, vp, vp, i32]
    lib.oracle_sgemm.restype = i32
    lib.oracle_sgemm_entries.argtypes = [i64, i64, i64, f32, vp, i64, vp, i64,
                                         f32, vp, i64, vp, vp, i64, vp, vp, i32]
    lib.oracle_sgemm_entries.restype = i32
    return lib


def load():
    """Return the ctypes handle of ``liboracle.so``, compiling it if needed."""
    global _lib
    if _lib is None:
        _lib = load_library(_build.build())
    return _lib


def default_threads():
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover - non-Linux hosts
        return max(1, os.cpu_count() or 1)


def _ld(x, name):
    """Leading dimension (in elements) of a row-major float32 2-D array."""
    if x.dtype != np.float32 or x.ndim != 2:
        raise TypeError("%s must be a 2-D float32 array" % name)
    if x.size == 0:
        return max(x.shape[1], 1)
    if x.shape[0] == 1:
        return max(x.shape[1], 1) if x.strides[1] == 4 else _bad(name)
    if x.strides[1] != 4 or x.strides[0] % 4 != 0 or x.strides[0] < 0:
        raise ValueError("%s must be row-major with unit inner stride" % name)
    return max(x.strides[0] // 4, x.shape[1], 1)


def _bad(name):
    raise ValueError("%s must be row-major with unit inner stride" % name)


def _ptr(x):
    return None if x is None else x.ctypes.data


def _shapes(A, B, C_old, beta):
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError("inner dimensions differ: A is %dx%d, B is %dx%d" % (M, K, K2, N))
    lda, ldb = _ld(A, "A"), _ld(B, "B")
    if C_old is None:
        if beta != 0:
            raise ValueError("C_old is required when beta != 0")
        ldc = max(N, 1)
    else:
        if C_old.shape != (M, N):
            raise ValueError("C_old must be %dx%d" % (M, N))
        ldc = _ld(C_old, "C_old")
    return M, N, K, lda, ldb, ldc


def sgemm(A, B, C_old, alpha, beta, nthreads=None, want_den=True, lib=None):
    """Full oracle: return ``(ref64, den)`` as M x N float64 arrays.

    ``A`` (M x K), ``B`` (K x N) and ``C_old`` (M x N, may be None when beta is 0)
    are float32 arrays, row-major, possibly with padded rows.  ``alpha`` and
    ``beta`` are rounded to float32 first, as the library takes them.  ``lib``
    selects another build of the oracle (the mutation tests use it).
    """
    M, N, K, lda, ldb, ldc = _shapes(A, B, C_old, beta)
    ref = np.zeros((M, N), dtype=np.float64)
    den = np.zeros((M, N), dtype=np.float64) if want_den else None
    st = (lib or load()).oracle_sgemm(M, N, K, float(np.float32(alpha)), _ptr(A), lda,
                             _ptr(B), ldb, float(np.float32(beta)), _ptr(C_old),
                             ldc, _ptr(ref), _ptr(den),
                             nthreads or default_threads())
    if st != 0:
        raise RuntimeError("oracle_sgemm failed with status %d" % st)
    return ref, den


def sgemm_entries(A, B, C_old, alpha, beta, rows, cols, nthreads=None, lib=None):
    """Sampled oracle: ``(ref64, den)`` for the entries ``(rows[e], cols[e])``."""
    M, N, K, lda, ldb, ldc = _shapes(A, B, C_old, beta)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if rows.shape != cols.shape or rows.ndim != 1:
        raise ValueError("rows and cols must be 1-D and of equal length")
    n = rows.shape[0]
    ref = np.zeros(n, dtype=np.float64)
    den = np.zeros(n, dtype=np.float64)
    st = (lib or load()).oracle_sgemm_entries(M, N, K, float(np.float32(alpha)), _ptr(A),
                                     lda, _ptr(B), ldb, float(np.float32(beta)),
                                     _ptr(C_old), ldc, _ptr(rows), _ptr(cols), n,
                                     _ptr(ref), _ptr(den),
                                     nthreads or default_threads())
    if st != 0:
        raise RuntimeError("oracle_sgemm_entries failed with status %d" % st)
    return ref, den


def max_rel_error(C, ref64, den):
    """The acceptance metric: max |C - ref64| / den over all entries.

    Entries with ``den == 0`` contribute 0 when ``C`` equals ``float32(ref64)``
    exactly and ``inf`` otherwise; a NaN in ``C`` gives ``inf``.
    """
    C = np.asarray(C, dtype=np.float64)
    ref64 = np.asarray(ref64, dtype=np.float64)
    den = np.asarray(den, dtype=np.float64)
    if C.shape != ref64.shape or den.shape != ref64.shape:
        raise ValueError("shape mismatch")
    if C.size == 0:
        return 0.0
    if np.isnan(C).any():
        return float("inf")
    diff = np.abs(C - ref64)
    zero = den == 0
    err = np.zeros_like(diff)
    nz = ~zero
    err[nz] = diff[nz] / den[nz]
    exact = C[zero] == ref64.astype(np.float32).astype(np.float64)[zero]
    err[zero] = np.where(exact, 0.0, np.inf)
    return float(err.max())


def ref32(ref64):
    """Round the fp64 oracle result to fp32 (round to nearest even)."""
    return np.asarray(ref64, dtype=np.float64).astype(np.float32)


def round_inputs(x, fmt):
    """Each fp32 value rounded to the nearest fp16 or bf16 value, ties to even,
    returned as fp32 (both types embed exactly in fp32).

    This is the input cast of the reduced-precision tensor-core mode: "Show HN:
    Phobos", section "Side-quest: Cheating", casts the fp32 data to a 16-bit
    type before the tensor cores and keeps an fp32 accumulator.  The mode's
    result is the plain definition applied to the rounded inputs:
    sgemm(round_inputs(A), round_inputs(B), C_old, alpha, beta).

    fp16 uses numpy's IEEE binary16 conversion (a library step).  bf16 is the
    upper half of the fp32 bit pattern, rounded to nearest with ties to even on
    the discarded 16 bits.  Finite inputs only.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    if fmt == "fp16":
        return x.astype(np.float16).astype(np.float32)
    if fmt == "bf16":
        bits = x.view(np.uint32).astype(np.uint64)
        keep_odd = (bits >> 16) & 1          # ties go to the even upper half
        r = ((bits + 0x7FFF + keep_odd) >> 16) << 16
        return r.astype(np.uint32).view(np.float32)
    raise ValueError("fmt must be 'fp16' or 'bf16'")

