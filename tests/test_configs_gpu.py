"""The full-size workloads on the GPU, checked against the CPU oracle.

Each workload runs once per math mode through the C ABI with the launch
configuration the benchmark uses (the automatic plan).  The 4096^3 (beta 0
and beta 1), 8192^3, 3001 x 5003 x 1999 and 65536 x 256 x 4096 workloads are
compared with the full oracle on every output element, as "Show HN: Phobos",
"Are we cuBLAS yet?" checks every element of its 4096^3 run; the oracle runs
once per workload and serves both modes.  The 16384^3 workload (and its
K-chunked cluster-split mode with 4096-deep K chunks) is checked on 4096
seeded entries plus the corners and last row/column stripes (the ragged edge
tiles), recomputed by the oracle one by one.  The largest error of every
workload is printed in pytest's terminal summary.
"""
import numpy as np
import pytest

import language_fp32_gemm_gb300 as phobos
import oracle
import seeded_inputs as si
from gpu_util import tolerance

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

MAX_ERRORS = {}  # "workload mode" -> max error, for the terminal summary


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from language_fp32_gemm_gb300 import build as lib_build
    lib_build.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


_inputs = {}
_full = {}


def inputs(name):
    if name not in _inputs:
        _inputs.clear()
        w = si.workload(name)
        _inputs[name] = (w, w.A(), w.B(), w.C_old())
    return _inputs[name]


def full_oracle(name):
    """(ref64, den) of the whole workload, computed once for both modes."""
    if name not in _full:
        _full.clear()
        w, A, B, C0 = inputs(name)
        _full[name] = oracle.sgemm(A, B, None if w.beta == 0 else C0, w.alpha, w.beta)
    return _full[name]


def run_on_gpu(dev, name, math, plan=None):
    w, A, B, C0 = inputs(name)
    dA = torch.from_numpy(A).to(dev)
    dB = torch.from_numpy(B).to(dev)
    dC = torch.from_numpy(C0).to(dev)
    phobos.sgemm(dA, dB, dC, w.alpha, w.beta, math=math, plan=plan)
    torch.cuda.synchronize()
    st = phobos.phobos_check_device(0)
    assert st == phobos.PHOBOS_OK, phobos.status_string(st)
    del dA, dB
    return w, dC


def run_full(dev, name, math):
    w, dC = run_on_gpu(dev, name, math)
    got = dC.cpu().numpy()
    del dC
    torch.cuda.empty_cache()
    ref, den = full_oracle(name)
    err = oracle.max_rel_error(got, ref, den)
    MAX_ERRORS["%s %s (all %d entries)" % (name, math, got.size)] = err
    assert err <= tolerance(math), "%s %s: max rel error %.3g" % (name, math, err)
    return err


def run_sampled(dev, name, math, plan=None, label=None):
    w, A, B, C0 = inputs(name)
    w, dC = run_on_gpu(dev, name, math, plan)
    rows, cols = w.samples()
    idx_r = torch.from_numpy(rows).to(dev)
    idx_c = torch.from_numpy(cols).to(dev)
    got = dC[idx_r, idx_c].cpu().numpy()
    assert torch.isfinite(dC).all().item()
    del dC
    torch.cuda.empty_cache()
    ref, den = oracle.sgemm_entries(A, B, C0, w.alpha, w.beta, rows, cols)
    err = oracle.max_rel_error(got, ref, den)
    MAX_ERRORS["%s %s (%d sampled entries)" % (name, label or math, got.size)] = err
    assert err <= tolerance(math), "%s %s: max rel error %.3g" % (name, math, err)
    return err


@pytest.mark.parametrize("math", ["default", "tf32"])
@pytest.mark.parametrize("name", ["sgemm_4096_beta0", "sgemm_4096_beta1"])
def test_square_4096(dev, name, math):
    run_full(dev, name, math)


@pytest.mark.parametrize("math", ["default", "tf32"])
def test_square_8192_headline(dev, math):
    run_full(dev, "sgemm_8192", math)


@pytest.mark.parametrize("math", ["default", "tf32"])
def test_unaligned_3001x5003x1999(dev, math):
    run_full(dev, "sgemm_3001x5003x1999", math)


@pytest.mark.parametrize("math", ["default", "tf32"])
def test_tall_skinny_65536x256x4096(dev, math):
    run_full(dev, "sgemm_65536x256x4096", math)


@pytest.mark.parametrize("super_k", [None, 4096])
def test_square_16384(dev, super_k):
    plan = None
    if super_k is not None:
        plan = phobos.phobos_gemm_plan(16384, 16384, 16384, 16384, 16384, 16384, "3xtf32")
        plan.super_k = super_k
    run_sampled(dev, "sgemm_16384", "default" if plan is None else "3xtf32", plan=plan,
                label=None if plan is None else "3xtf32 super_k=4096")
