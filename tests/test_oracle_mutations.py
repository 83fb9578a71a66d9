"""Plant plausible mistakes in copies of the oracle and check the pins catch them.

Each mutant is the oracle's C source with one textual change (a dropped term,
a flipped sign, a transposed operand, a shortened loop ...), compiled with the
oracle's own build step into a temporary directory.  A mutant that passes
every pin would mean the pins cannot tell that mistake from the definition.
CPU only; the real oracle is not modified.
"""
import os

import pytest

import oracle
from oracle import build as oracle_build
from oracle_pins import ALL_PINS

MUTANTS = {
    "drop_beta_term": [("value += job->beta * c;", "(void)c;")],
    "sign_flip": [("s[j] += aik * bkj;", "s[j] -= aik * bkj;")],
    "transposed_b": [("const float *brow = job->B + k * job->ldb;", "const float *brow = job->B + k;"),
                     ("const double bkj = (double)brow[j];", "const double bkj = (double)brow[j * job->ldb];")],
    "short_k_loop": [("for (int64_t k = 0; k < K; ++k) {\n      const double aik = (double)job->A[i * job->lda + k];\n      const double abs_aik",
                      "for (int64_t k = 0; k < K - 1; ++k) {\n      const double aik = (double)job->A[i * job->lda + k];\n      const double abs_aik")],
    "alpha_ignored": [("double value = job->alpha * s[j];", "double value = s[j];")],
    "den_without_abs": [("a[j] += abs_aik * fabs(bkj);", "a[j] += abs_aik * bkj;")],
    "wrong_a_stride": [("const double aik = (double)job->A[i * job->lda + k];\n      const double abs_aik",
                        "const double aik = (double)job->A[i * job->K + k];\n      const double abs_aik")],
    "c_old_transposed": [("const double c = (double)job->C_old[i * job->ldc + j];",
                          "const double c = (double)job->C_old[j * job->ldc + i];")],
    "entries_drop_last_k": [("for (int64_t k = 0; k < job->K; ++k) {", "for (int64_t k = 1; k < job->K; ++k) {")],
    "fp32_accumulation": [("double *s = (double *)malloc", "float *s = (float *)malloc")],
}


def _apply(src, edits):
    for old, new in edits:
        assert src.count(old) >= 1, "mutation anchor not found: %r" % old[:60]
        src = src.replace(old, new, 1)
    return src


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    src = open(oracle_build.SOURCE).read()
    mutated = _apply(src, MUTANTS[name])
    c_path = os.path.join(tmp_path, "mutant_%s.c" % name)
    with open(c_path, "w") as fh:
        fh.write(mutated)
    so_path = os.path.join(tmp_path, "libmutant_%s.so" % name)
    lib = oracle.load_library(oracle_build.build(source=c_path, output=so_path, force=True))
    caught = []
    for pin in ALL_PINS:
        try:
            pin(lib=lib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, "no pin detects mutant %s" % name
