"""The full-size workloads on the GPU, checked on seeded sampled entries.

Each workload runs once through the C ABI with the launch configuration the
benchmark uses (the automatic plan), and 4096 seeded entries plus the corners
and last row/column stripes (the ragged edge tiles) are recomputed by the CPU
oracle one by one.  The K-chunked (cluster split) mode of the 16384^3 shape
runs with 4096-deep K chunks.
"""
import numpy as np
import pytest

import language_fp32_gemm_gb300 as phobos
import oracle
import seeded_inputs as si
from gpu_util import tolerance

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from language_fp32_gemm_gb300 import build as lib_build
    lib_build.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


_cache = {}


def inputs(name):
    if name not in _cache:
        _cache.clear()
        w = si.workload(name)
        _cache[name] = (w, w.A(), w.B(), w.C_old())
    return _cache[name]


def run_sampled(dev, name, math, plan=None, beta=None):
    w, A, B, C0 = inputs(name)
    beta = w.beta if beta is None else beta
    dA = torch.from_numpy(A).to(dev)
    dB = torch.from_numpy(B).to(dev)
    dC = torch.from_numpy(C0).to(dev)
    phobos.sgemm(dA, dB, dC, w.alpha, beta, math=math, plan=plan)
    torch.cuda.synchronize()
    st = phobos.phobos_check_device(0)
    assert st == phobos.PHOBOS_OK, phobos.status_string(st)
    rows, cols = w.samples()
    idx_r = torch.from_numpy(rows).to(dev)
    idx_c = torch.from_numpy(cols).to(dev)
    got = dC[idx_r, idx_c].cpu().numpy()
    assert torch.isfinite(dC).all().item()
    del dA, dB, dC
    torch.cuda.empty_cache()
    ref, den = oracle.sgemm_entries(A, B, C0, w.alpha, beta, rows, cols)
    err = oracle.max_rel_error(got, ref, den)
    assert err <= tolerance(math), "%s %s: max rel error %.3g" % (name, math, err)
    return err


@pytest.mark.parametrize("math", ["default", "tf32"])
@pytest.mark.parametrize("name", ["sgemm_4096_beta0", "sgemm_4096_beta1"])
def test_square_4096(dev, name, math):
    run_sampled(dev, name, math)


@pytest.mark.parametrize("math", ["default", "tf32"])
def test_square_8192_headline(dev, math):
    run_sampled(dev, "sgemm_8192", math)


@pytest.mark.parametrize("math", ["default", "tf32"])
def test_unaligned_3001x5003x1999(dev, math):
    run_sampled(dev, "sgemm_3001x5003x1999", math)


@pytest.mark.parametrize("math", ["default", "tf32"])
def test_tall_skinny_65536x256x4096(dev, math):
    run_sampled(dev, "sgemm_65536x256x4096", math)


@pytest.mark.parametrize("super_k", [None, 4096])
def test_square_16384(dev, super_k):
    plan = None
    if super_k is not None:
        plan = phobos.phobos_gemm_plan(16384, 16384, 16384, 16384, 16384, 16384, "3xtf32")
        plan.super_k = super_k
    run_sampled(dev, "sgemm_16384", "default" if plan is None else "3xtf32", plan=plan)
