"""Reader for the text fixtures under tests/golden/."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_fixture(name):
    lines = [l.strip() for l in open(os.path.join(GOLDEN, name)) if l.strip() and not l.startswith("#")]
    head = lines[0].split()
    meta = {head[i]: head[i + 1] for i in range(0, len(head), 2)}
    M, N, K = int(meta["M"]), int(meta["N"]), int(meta["K"])
    alpha, beta = float(meta["alpha"]), float(meta["beta"])
    mats, at = {}, 1
    for name, rows in (("A", M), ("B", K), ("C_old", M), ("C", M)):
        assert lines[at] == name
        mats[name] = np.array([[float(v) for v in lines[at + 1 + r].split()] for r in range(rows)],
                              dtype=np.float32 if name != "C" else np.float64)
        at += rows + 1
    return M, N, K, alpha, beta, mats
