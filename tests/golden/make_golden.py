"""Write the small integer GEMM fixture in this folder from the CPU oracle.

The fixture is an input-output example of the definition
C = alpha * A B + beta * C_old (the ``matmul`` listing of the "@cluster"
attribute page; "Matrix Multiplication" in "Show HN: Phobos"), with integer
entries so that every value is exact and can be checked by hand.  Only the
oracle and the seeded input generator are called.
Run:  python tests/golden/make_golden.py
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import seeded_inputs as si  # noqa: E402

M, N, K, ALPHA, BETA, SEED = 4, 3, 5, 1.5, 0.5, 42


def main():
    A = si.integers(SEED, 0, (M, K))
    B = si.integers(SEED, 1, (K, N))
    C = si.integers(SEED, 2, (M, N))
    ref, _ = oracle.sgemm(A, B, C, ALPHA, BETA)
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "sgemm_int_4x3x5.txt")
    with open(path, "w") as fh:
        fh.write("# C = alpha*A*B + beta*C_old, row-major; definition: '@cluster' page matmul\n")
        fh.write("# listing and 'Show HN: Phobos', section 'Matrix Multiplication'.\n")
        fh.write("# Written by tests/golden/make_golden.py from the CPU oracle; integers -4..4.\n")
        fh.write("M %d N %d K %d alpha %r beta %r\n" % (M, N, K, ALPHA, BETA))
        for name, mat in (("A", A), ("B", B), ("C_old", C), ("C", ref)):
            fh.write(name + "\n")
            for row in mat:
                fh.write(" ".join(repr(float(v)) for v in row) + "\n")
    print(path)


if __name__ == "__main__":
    main()
