"""The CPU oracle against facts fixed by the definition and by mathematics.

CPU only.  See ``oracle_pins.py`` for what each pin checks and why it is
independent of the oracle's own code.
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


def test_beta_zero_does_not_read_c_old():
    A = si.uniform_pm1(20, 0, (6, 5))
    B = si.uniform_pm1(20, 1, (5, 4))
    C = np.full((6, 4), np.nan, dtype=np.float32)
    ref, den = oracle.sgemm(A, B, C, 1.0, 0.0)
    assert np.isfinite(ref).all() and np.isfinite(den).all()
    ref2, _ = oracle.sgemm(A, B, None, 1.0, 0.0)
    assert np.array_equal(ref, ref2)


def test_alpha_zero_and_empty_k_give_beta_c():
    C = si.uniform_pm1(21, 2, (5, 7))
    A = si.uniform_pm1(21, 0, (5, 3))
    B = si.uniform_pm1(21, 1, (3, 7))
    ref, den = oracle.sgemm(A, B, C, 0.0, 0.5)
    assert np.array_equal(ref, 0.5 * C.astype(np.float64))
    ref, den = oracle.sgemm(np.zeros((5, 0), np.float32), np.zeros((0, 7), np.float32), C, 2.0, 0.5)
    assert np.array_equal(ref, 0.5 * C.astype(np.float64))
    assert np.array_equal(den, 0.5 * np.abs(C.astype(np.float64)))


def test_empty_outputs():
    ref, den = oracle.sgemm(np.zeros((0, 3), np.float32), np.zeros((3, 4), np.float32), None, 1.0, 0.0)
    assert ref.shape == (0, 4)
    ref, den = oracle.sgemm(np.zeros((3, 2), np.float32), np.zeros((2, 0), np.float32), None, 1.0, 0.0)
    assert ref.shape == (3, 0)


def test_padded_leading_dimensions():
    M, N, K = 9, 11, 7
    big_a = si.uniform_pm1(22, 0, (M, K + 5))
    big_b = si.uniform_pm1(22, 1, (K, N + 3))
    big_c = si.uniform_pm1(22, 2, (M, N + 1))
    A, B, C = big_a[:, :K], big_b[:, :N], big_c[:, :N]
    r1, d1 = oracle.sgemm(A, B, C, 1.5, 0.5)
    r2, d2 = oracle.sgemm(np.ascontiguousarray(A), np.ascontiguousarray(B),
                          np.ascontiguousarray(C), 1.5, 0.5)
    assert np.array_equal(r1, r2) and np.array_equal(d1, d2)


def test_thread_count_does_not_change_the_result():
    A = si.normal(23, 0, (50, 40))
    B = si.normal(23, 1, (40, 30))
    C = si.normal(23, 2, (50, 30))
    r1, d1 = oracle.sgemm(A, B, C, 0.3, 0.7, nthreads=1)
    r7, d7 = oracle.sgemm(A, B, C, 0.3, 0.7, nthreads=7)
    assert np.array_equal(r1, r7) and np.array_equal(d1, d7)


def test_bad_arguments_are_rejected():
    lib = oracle.load()
    # lda < K
    assert lib.oracle_sgemm(2, 2, 3, 1.0, None, 2, None, 2, 0.0, None, 2, None, None, 1) == 1
    # negative size
    assert lib.oracle_sgemm(-1, 2, 3, 1.0, None, 3, None, 2, 0.0, None, 2, None, None, 1) == 1
    with pytest.raises(ValueError):
        oracle.sgemm(np.zeros((2, 3), np.float32), np.zeros((4, 2), np.float32), None, 1.0, 0.0)
    with pytest.raises(ValueError):
        oracle.sgemm(np.zeros((2, 3), np.float32), np.zeros((3, 2), np.float32), None, 1.0, 1.0)
    A = np.zeros((2, 3), np.float32)
    with pytest.raises(RuntimeError):
        oracle.sgemm_entries(A, np.zeros((3, 2), np.float32), None, 1.0, 0.0, [2], [0])


def test_error_metric():
    ref = np.array([1.0, 0.0, -2.0])
    den = np.array([1.0, 0.0, 4.0])
    assert oracle.max_rel_error(np.array([1.0, 0.0, -2.0]), ref, den) == 0.0
    assert oracle.max_rel_error(np.array([1.5, 0.0, -2.0]), ref, den) == 0.5
    assert oracle.max_rel_error(np.array([1.0, 1e-30, -2.0]), ref, den) == float("inf")
    assert oracle.max_rel_error(np.array([np.nan, 0.0, -2.0]), ref, den) == float("inf")
    assert oracle.max_rel_error(np.array([1.0, 0.0, -1.0]), ref, den) == 0.25
    assert oracle.TOL_FP32 == 2.0 ** -20 and oracle.TOL_TF32 == 2.0 ** -10


def _nearest_even(x, table_bits, to_float):
    """Brute force: the value of the 16-bit table nearest to each x, ties to the
    even bit pattern, found by searching every finite value of the type."""
    with np.errstate(invalid="ignore"):
        vals = to_float(table_bits).astype(np.float64)
    ok = np.isfinite(vals)
    vals, bits = vals[ok], table_bits[ok]
    order = np.argsort(vals, kind="stable")
    vals, bits = vals[order], bits[order]
    keep = np.concatenate(([True], np.diff(vals) != 0))  # +0 and -0 are one value
    vals, bits = vals[keep], bits[keep]
    out = np.empty(x.shape, dtype=np.float64)
    for n, v in enumerate(x.astype(np.float64)):
        j = int(np.searchsorted(vals, v))
        cands = [c for c in (j - 1, j) if 0 <= c < len(vals)]
        best = min(cands, key=lambda c: (abs(vals[c] - v), int(bits[c]) & 1))
        out[n] = vals[best]
    return out


def _probe_values():
    rng = np.random.default_rng(3)
    x = np.concatenate([
        rng.standard_normal(3000),
        rng.uniform(-1, 1, 3000) * 2.0 ** rng.integers(-20, 15, 3000),
        # exact ties of both types: 1 + (2j+1) * 2^-11 and 1 + (2j+1) * 2^-8
        1 + (2 * np.arange(40) + 1) * 2.0 ** -11, -(1 + (2 * np.arange(40) + 1) * 2.0 ** -8),
        [0.0, 1.0, -1.0, 0.5, 65504.0, 2.0 ** -14, 3.0 * 2 ** -9],
    ])
    return x.astype(np.float32)


def test_round_inputs_fp16_is_nearest_even():
    """fp16 rounding of the oracle equals an exhaustive nearest-value search."""
    x = _probe_values()
    x = x[np.abs(x) <= 65504]
    table = np.arange(1 << 16, dtype=np.uint16)
    want = _nearest_even(x, table, lambda b: b.view(np.float16))
    got = oracle.round_inputs(x, "fp16").astype(np.float64)
    assert np.array_equal(got, want)


def test_round_inputs_bf16_is_nearest_even():
    """bf16 rounding of the oracle equals an exhaustive nearest-value search."""
    x = _probe_values()
    table = np.arange(1 << 16, dtype=np.uint32)
    want = _nearest_even(x, table, lambda b: (b << 16).astype(np.uint32).view(np.float32))
    got = oracle.round_inputs(x, "bf16").astype(np.float64)
    assert np.array_equal(got, want)
    # values a bf16 holds exactly are unchanged, and the rounding is monotone
    exact = np.arange(-255, 256, dtype=np.float32) * 0.25  # 8 significant bits at most
    assert np.array_equal(oracle.round_inputs(exact, "bf16"), exact)
    s = np.sort(x)
    assert np.all(np.diff(oracle.round_inputs(s, "bf16").astype(np.float64)) >= 0)


@pytest.mark.parametrize("mutant", ["truncate", "ties_away", "fp16_truncate"])
def test_rounding_pins_catch_mutants(mutant):
    """Plausible mistakes in the 16-bit input rounding fail the exhaustive pins."""
    x = _probe_values()
    if mutant == "fp16_truncate":
        x = x[np.abs(x) <= 65504]
        table = np.arange(1 << 16, dtype=np.uint16)
        want = _nearest_even(x, table, lambda b: b.view(np.float16))
        # round toward zero: drop the 13 low mantissa bits (normal range only)
        bits = x.view(np.uint32)
        bad = ((bits >> 13) << 13).view(np.float32).astype(np.float16).astype(np.float64)
    else:
        table = np.arange(1 << 16, dtype=np.uint32)
        want = _nearest_even(x, table, lambda b: (b << 16).astype(np.uint32).view(np.float32))
        bits = x.view(np.uint32).astype(np.uint64)
        if mutant == "truncate":
            r = (bits >> 16) << 16
        else:  # ties away from zero instead of to even
            r = ((bits + 0x8000) >> 16) << 16
        bad = r.astype(np.uint32).view(np.float32).astype(np.float64)
    assert not np.array_equal(bad, want), mutant
