"""The stored integer example against exact arithmetic and the oracle."""
import numpy as np

import oracle
from golden_io import read_fixture


def test_integer_fixture():
    M, N, K, alpha, beta, m = read_fixture("sgemm_int_4x3x5.txt")
    A, B, C, expect = m["A"], m["B"], m["C_old"], m["C"]
    assert A.shape == (M, K) and B.shape == (K, N)
    exact = alpha * (A.astype(np.int64) @ B.astype(np.int64)) + beta * C.astype(np.int64)
    assert np.array_equal(expect, exact)
    ref, _ = oracle.sgemm(A, B, C, alpha, beta)
    assert np.array_equal(ref, expect)
