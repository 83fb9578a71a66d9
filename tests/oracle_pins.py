"""Checks that tie the CPU oracle to facts that do not depend on the oracle.

Each ``pin_*`` function takes the oracle's two entry points (so that the
mutation test can hand it a deliberately broken build) and raises
``AssertionError`` when the oracle disagrees with:

* exact rational arithmetic on tiny inputs (brute force, ``fractions``),
* integer inputs whose exact product numpy's int64 matmul gives,
* the closed forms A = I  (C = alpha*B + beta*C_old) and B = 0 (C = beta*C_old),
* the transpose identity (A B)^T = B^T A^T and linearity in alpha,
* a library fp64 matmul within the fp64 rounding bound.

The definition they pin: C = alpha * A B + beta * C_old with A (M x K) and
B (K x N) row-major, from the ``matmul`` listing on the "@cluster" attribute
page and the "Matrix Multiplication" section of "Show HN: Phobos".
"""
from fractions import Fraction

import numpy as np

import oracle
import seeded_inputs as si

TINY_SHAPES = [(1, 1, 1), (2, 3, 5), (3, 5, 7), (5, 7, 2), (7, 16, 17),
               (16, 17, 3), (17, 2, 16), (4, 4, 1)]


def _rand(seed, stream, shape):
    return si.uniform_pm1(seed, stream, shape)


def pin_bruteforce(lib=None):
    """ref64 equals the exact rational result within the fp64 summation bound."""
    for t, (M, N, K) in enumerate(TINY_SHAPES):
        A = _rand(100 + t, 0, (M, K))
        B = _rand(100 + t, 1, (K, N))
        C = _rand(100 + t, 2, (M, N))
        alpha, beta = np.float32(1.25), np.float32(-0.375)
        ref, den = oracle.sgemm(A, B, C, alpha, beta, nthreads=2, lib=lib)
        for i in range(M):
            for j in range(N):
                exact = Fraction(0)
                scale = Fraction(0)
                for k in range(K):
                    p = Fraction(float(A[i, k])) * Fraction(float(B[k, j]))
                    exact += p
                    scale += abs(p)
                exact = Fraction(float(alpha)) * exact + Fraction(float(beta)) * Fraction(float(C[i, j]))
                scale = abs(Fraction(float(alpha))) * scale + abs(Fraction(float(beta))) * abs(Fraction(float(C[i, j])))
                # K additions in fp64 plus the two scalar products and one add.
                bound = Fraction(K + 3) * Fraction(2) ** -52 * scale
                assert abs(Fraction(float(ref[i, j])) - exact) <= bound, (M, N, K, i, j)
                assert abs(Fraction(float(den[i, j])) - scale) <= bound, ("den", M, N, K, i, j)


def pin_integer_exact(lib=None, M=37, N=29, K=41):
    """Integer entries: ref64 equals exact int64 arithmetic, for odd shapes.

    The three matrices are views into wider buffers (lda, ldb, ldc larger than
    the row length), so a mistake in a leading dimension shows up here.
    """
    A = si.integers(7, 0, (M, K + 3))[:, :K]
    B = si.integers(7, 1, (K, N + 5))[:, :N]
    C = si.integers(7, 2, (M, N + 2))[:, :N]
    ref, den = oracle.sgemm(A, B, C, 1.5, 0.5, nthreads=3, lib=lib)
    P = A.astype(np.int64) @ B.astype(np.int64)
    # alpha*P + beta*C = (3P + C) / 2 exactly
    exact = (3 * P + C.astype(np.int64)).astype(np.float64) / 2.0
    assert np.array_equal(ref, exact)
    absP = np.abs(A.astype(np.int64)) @ np.abs(B.astype(np.int64))
    assert np.array_equal(den, (3 * absP + np.abs(C.astype(np.int64))).astype(np.float64) / 2.0)
    assert np.array_equal(oracle.ref32(ref), exact.astype(np.float32))


def pin_identity(lib=None, M=23, N=19):
    """A = I (M = K): C = alpha*B + beta*C_old, bit for bit in fp64."""
    A = np.eye(M, dtype=np.float32)
    B = _rand(11, 1, (M, N))
    C = _rand(11, 2, (M, N))
    alpha, beta = np.float32(0.75), np.float32(0.25)
    ref, den = oracle.sgemm(A, B, C, alpha, beta, lib=lib)
    expect = float(alpha) * B.astype(np.float64) + float(beta) * C.astype(np.float64)
    assert np.array_equal(ref, expect)
    assert np.array_equal(den, abs(float(alpha)) * np.abs(B.astype(np.float64))
                          + abs(float(beta)) * np.abs(C.astype(np.float64)))


def pin_zero_b(lib=None, M=13, N=9, K=31):
    """B = 0: C = beta*C_old exactly (and alpha*A*0 contributes nothing)."""
    A = _rand(12, 0, (M, K))
    B = np.zeros((K, N), dtype=np.float32)
    C = _rand(12, 2, (M, N))
    ref, den = oracle.sgemm(A, B, C, 1.5, -0.5, lib=lib)
    assert np.array_equal(ref, -0.5 * C.astype(np.float64))
    assert np.array_equal(den, 0.5 * np.abs(C.astype(np.float64)))


def pin_transpose(lib=None, M=11, N=7, K=13):
    """(A B)^T = B^T A^T: the transposed problem gives the transposed result."""
    A = _rand(13, 0, (M, K))
    B = _rand(13, 1, (K, N))
    C = _rand(13, 2, (M, N))
    ref, den = oracle.sgemm(A, B, C, 0.5, 2.0, lib=lib)
    refT, denT = oracle.sgemm(np.ascontiguousarray(B.T), np.ascontiguousarray(A.T),
                              np.ascontiguousarray(C.T), 0.5, 2.0, lib=lib)
    assert np.array_equal(ref, refT.T)
    assert np.array_equal(den, denT.T)


def pin_linearity(lib=None, M=9, N=12, K=10):
    """beta = 0: doubling alpha doubles the result exactly (power-of-two scaling)."""
    A = _rand(14, 0, (M, K))
    B = _rand(14, 1, (K, N))
    r1, _ = oracle.sgemm(A, B, None, 0.75, 0.0, lib=lib)
    r2, _ = oracle.sgemm(A, B, None, 1.5, 0.0, lib=lib)
    assert np.array_equal(r2, 2.0 * r1)
    assert np.any(r1 != 0)


def pin_library_matmul(lib=None, M=33, N=47, K=65):
    """Agreement with numpy's fp64 matmul within the fp64 rounding bound."""
    A = si.normal(15, 0, (M, K))
    B = si.normal(15, 1, (K, N))
    C = si.normal(15, 2, (M, N))
    ref, den = oracle.sgemm(A, B, C, -0.5, 1.25, lib=lib)
    A64, B64, C64 = A.astype(np.float64), B.astype(np.float64), C.astype(np.float64)
    expect = -0.5 * (A64 @ B64) + 1.25 * C64
    scale = 0.5 * (np.abs(A64) @ np.abs(B64)) + 1.25 * np.abs(C64)
    assert np.all(np.abs(ref - expect) <= 4 * (K + 3) * 2.0 ** -52 * scale)
    assert np.allclose(den, scale, rtol=4 * (K + 3) * 2.0 ** -52, atol=0)


def pin_entries(lib=None, M=40, N=33, K=21):
    """The sampled mode gives the full mode's values at the sampled positions."""
    A = _rand(16, 0, (M, K))
    B = _rand(16, 1, (K, N))
    C = _rand(16, 2, (M, N))
    ref, den = oracle.sgemm(A, B, C, 1.0, 0.5, lib=lib)
    rows, cols = si.sample_indices(16, 3, M, N, 50)
    r, d = oracle.sgemm_entries(A, B, C, 1.0, 0.5, rows, cols, nthreads=4, lib=lib)
    assert np.array_equal(r, ref[rows, cols])
    assert np.array_equal(d, den[rows, cols])
    # and the sampled mode on its own against exact integers
    Ai, Bi, Ci = si.integers(17, 0, (M, K)), si.integers(17, 1, (K, N)), si.integers(17, 2, (M, N))
    r, _ = oracle.sgemm_entries(Ai, Bi, Ci, 1.5, 0.5, rows, cols, lib=lib)
    P = Ai.astype(np.int64) @ Bi.astype(np.int64)
    assert np.array_equal(r, ((3 * P + Ci.astype(np.int64)) / 2.0)[rows, cols])


ALL_PINS = [pin_bruteforce, pin_integer_exact, pin_identity, pin_zero_b, pin_transpose,
            pin_linearity, pin_library_matmul, pin_entries]
