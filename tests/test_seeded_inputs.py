"""The seeded input generator against SplitMix64's sequential definition."""
import numpy as np

import seeded_inputs as si

MASK = (1 << 64) - 1


def _mix_py(z):
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK
    return z ^ (z >> 31)


def _sequential(state, count):
    out = []
    for _ in range(count):
        state = (state + 0x9E3779B97F4A7C15) & MASK
        out.append(_mix_py(state))
    return out


def test_counter_form_equals_sequential_generator():
    for state in (0, 1, 1234567, (1 << 64) - 1):
        got = [int(v) for v in si.splitmix64_sequence(state, 9)]
        assert got == _sequential(state, 9)


def test_streams_use_their_own_base_and_offsets():
    base = int(si.stream_base(5, 3))
    assert base == _mix_py((5 * (1 << 20) + 3) & MASK)
    whole = si.stream_bits(5, 3, 40)
    assert [int(v) for v in whole] == _sequential(base, 40)
    assert np.array_equal(si.stream_bits(5, 3, 10, offset=30), whole[30:])


def test_value_maps():
    u = si.uniform_pm1(1, 0, (1000,))
    assert u.dtype == np.float32 and u.min() >= -1.0 and u.max() < 1.0
    # every value is a multiple of 2**-23 (24-bit grid on [-1, 1))
    assert np.all(np.round(u.astype(np.float64) * 2 ** 23) == u.astype(np.float64) * 2 ** 23)
    z = si.integers(1, 1, (5000,))
    assert set(np.unique(z).tolist()) == set(range(-4, 5))
    n = si.normal(1, 2, (200000,), sd=0.5)
    assert abs(float(n.mean())) < 0.01 and abs(float(n.std()) - 0.5) < 0.01


def test_chunked_generation_matches_unchunked(monkeypatch):
    a = si.uniform_pm1(9, 1, (3, 1000))
    monkeypatch.setattr(si, "_CHUNK", 257)
    b = si.uniform_pm1(9, 1, (3, 1000))
    assert np.array_equal(a, b)
    c = si.normal(9, 1, (3, 1000))
    monkeypatch.setattr(si, "_CHUNK", 1 << 22)
    assert np.array_equal(c, si.normal(9, 1, (3, 1000)))


def test_row_blocks_equal_slices_of_the_whole_matrix(monkeypatch):
    # the large-matrix GPU tests draw and upload a matrix block by block
    whole = si.integers(21, 3, (37, 53), -2, 2)
    blocks = [si.integer_rows(21, 3, (37, 53), r0, min(37, r0 + 8), -2, 2) for r0 in range(0, 37, 8)]
    assert np.array_equal(np.concatenate(blocks), whole)
    monkeypatch.setattr(si, "_CHUNK", 100)
    assert np.array_equal(si.integer_rows(21, 3, (37, 53), 30, 37, -2, 2), whole[30:])
    assert si.integer_rows(21, 3, (37, 53), 5, 5).shape == (0, 53)
    # element n of the matrix is draw n of the stream
    x = si.stream_bits(21, 3, 1, 11 * 53 + 7)[0]
    assert whole[11, 7] == float(int(x >> np.uint64(32)) % 5 - 2)


def test_workload_table():
    w = si.workload("sgemm_8192")
    assert (w.M, w.N, w.K, w.alpha, w.beta, w.seed) == (8192, 8192, 8192, 0.75, 0.25, 2)
    w = si.workload("sgemm_3001x5003x1999")
    assert (w.M, w.N, w.K) == (3001, 5003, 1999)
    r, c = si.workload("sgemm_16384").samples()
    assert r.min() >= 0 and r.max() < 16384 and c.max() == 16383 and len(r) >= 4096


def test_every_workload_matches_its_stated_recipe():
    # (M, N, K, alpha, beta, seed, A, B, C_old) as the five benchmark workloads state them
    want = {
        "sgemm_256": (256, 256, 256, 1.5, 0.5, 0, "uniform", "uniform", "uniform"),
        "sgemm_256_int": (256, 256, 256, 1.5, 0.5, 0, "int", "int", "int"),
        "sgemm_4096_beta0": (4096, 4096, 4096, 1.0, 0.0, 1, "normal", "normal", "uniform"),
        "sgemm_4096_beta1": (4096, 4096, 4096, 1.0, 1.0, 1, "normal", "normal", "uniform"),
        "sgemm_8192": (8192, 8192, 8192, 0.75, 0.25, 2, "uniform", "uniform", "normal"),
        "sgemm_3001x5003x1999": (3001, 5003, 1999, 1.0, 0.5, 3, "normal", "normal", "uniform"),
        "sgemm_65536x256x4096": (65536, 256, 4096, 1.0, 0.5, 3, "normal", "normal", "uniform"),
        "sgemm_16384": (16384, 16384, 16384, 1.0, 0.0, 4, "uniform", "uniform", "zeros"),
    }
    assert set(si.WORKLOADS) == set(want)
    for name, (M, N, K, alpha, beta, seed, a, b, c) in want.items():
        w = si.workload(name)
        assert (w.M, w.N, w.K, w.alpha, w.beta, w.seed) == (M, N, K, alpha, beta, seed), name
        assert (w.a[0], w.b[0], w.c[0]) == (a, b, c), name
    # N(0, 1/sqrt(K)): the standard deviation is 1/sqrt(K)
    for name in ("sgemm_3001x5003x1999", "sgemm_65536x256x4096"):
        w = si.workload(name)
        assert w.a[1] == w.b[1] == 1.0 / np.sqrt(w.K)
    # the two shapes that share seed 3 draw from different streams
    assert set(si.workload("sgemm_3001x5003x1999").streams).isdisjoint(
        si.workload("sgemm_65536x256x4096").streams)
