"""The fp16 / bf16-input tensor-core mode against the CPU oracle.

The mode casts the fp32 inputs to a 16-bit type before the tensor cores and
accumulates in fp32 ("Show HN: Phobos", "Side-quest: Cheating").  Its result
is therefore the definition applied to the rounded inputs, and the tight check
is against ``oracle.sgemm(round_inputs(A), round_inputs(B), ...)`` with
oracle.TOL_HALF_ACC (2^-13), which leaves room only for the fp32
accumulation.  The loose check against the fp32 inputs (2^-9 fp16, 2^-6 bf16)
bounds what the input rounding costs.  Integer inputs and B = 0 are
bit-exact: small integers are exact in both types, and so are their
products and sums below 2^24.
"""
import numpy as np
import pytest

import language_fp32_gemm_gb300 as phobos
import oracle
import seeded_inputs as si
from gpu_util import padded, run_gemm

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

FMTS = ["fp16", "bf16"]
LOOSE = {"fp16": oracle.TOL_FP16, "bf16": oracle.TOL_BF16}


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from language_fp32_gemm_gb300 import build as lib_build
    lib_build.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def check(dev, A, B, C0, alpha, beta, fmt, plan=None, offsets=(0, 0, 0)):
    C = run_gemm(torch, dev, A, B, C0, alpha, beta, fmt, plan=plan, offsets=offsets)
    ref, den = oracle.sgemm(oracle.round_inputs(A, fmt), oracle.round_inputs(B, fmt), C0, alpha, beta)
    err = oracle.max_rel_error(C, ref, den)
    assert err <= oracle.TOL_HALF_ACC, "%s vs rounded inputs: %.3g" % (fmt, err)
    ref2, den2 = oracle.sgemm(A, B, C0, alpha, beta)
    err2 = oracle.max_rel_error(C, ref2, den2)
    assert err2 <= LOOSE[fmt], "%s vs fp32 inputs: %.3g" % (fmt, err2)
    return err, err2


SHAPES = [(1, 1, 1), (7, 13, 5), (128, 256, 64), (129, 257, 65), (300, 260, 200),
          (513, 384, 1000), (16, 520, 64), (130, 17, 260), (1000, 700, 1333)]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "%dx%dx%d" % s)
def test_shapes(dev, shape, fmt):
    M, N, K = shape
    seed = 2000 + M * 7 + N * 3 + K
    A = si.normal(seed, 0, (M, K))
    B = si.normal(seed, 1, (K, N))
    C0 = si.uniform_pm1(seed, 2, (M, N))
    check(dev, A, B, C0, 1.25, -0.5, fmt)


@pytest.mark.parametrize("fmt", FMTS)
def test_padded_and_unaligned(dev, fmt):
    M, N, K = 200, 150, 90
    A = padded(si.normal(41, 0, (M, K)), 3)
    B = padded(si.normal(41, 1, (K, N)), 5)
    C0 = padded(si.uniform_pm1(41, 2, (M, N)), 1)
    check(dev, A, B, C0, 0.75, 0.25, fmt, offsets=(1, 3, 2))


@pytest.mark.parametrize("fmt", FMTS)
def test_integer_inputs_bit_exact(dev, fmt):
    w = si.workload("sgemm_256_int")
    A, B, C0 = w.A(), w.B(), w.C_old()
    C = run_gemm(torch, dev, A, B, C0, w.alpha, w.beta, fmt)
    ref, _ = oracle.sgemm(A, B, C0, w.alpha, w.beta)
    assert np.array_equal(C, oracle.ref32(ref))


@pytest.mark.parametrize("fmt", FMTS)
def test_zero_b_bit_exact_and_beta_zero_ignores_nan(dev, fmt):
    M, N, K = 150, 300, 70
    A = si.normal(42, 0, (M, K))
    C0 = si.uniform_pm1(42, 2, (M, N))
    C = run_gemm(torch, dev, A, np.zeros((K, N), np.float32), C0, 1.5, -0.5, fmt)
    assert np.array_equal(C, (-0.5 * C0.astype(np.float64)).astype(np.float32))
    B = si.normal(42, 1, (K, N))
    nan = np.full((M, N), np.nan, np.float32)
    C = run_gemm(torch, dev, A, B, nan, 1.0, 0.0, fmt)
    assert np.isfinite(C).all()


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape,split,super_k", [((512, 512, 2048), 0, None), ((2304, 2304, 700), 0, None),
                                                  ((520, 390, 2100), 0, 512)])
def test_tail_split_and_k_chunks(dev, fmt, shape, split, super_k):
    M, N, K = shape
    A = si.normal(43, 0, (M, K))
    B = si.normal(43, 1, (K, N))
    C0 = si.uniform_pm1(43, 2, (M, N))
    plan = phobos.phobos_gemm_plan(M, N, K, K, N, N, fmt)
    plan.tail_split = split
    if super_k is not None:
        plan.super_k = super_k
    check(dev, A, B, C0, 1.0, 0.5, fmt, plan=plan)


@pytest.mark.parametrize("fmt", FMTS)
def test_plan_rules(dev, fmt):
    plan = phobos.phobos_gemm_plan(512, 512, 512, 512, 512, 512, fmt)
    assert plan.path == (phobos.PHOBOS_PATH_FP16 if fmt == "fp16" else phobos.PHOBOS_PATH_BF16)
    assert plan.tile_k == 64 and plan.cluster_m == 2
    A = torch.zeros(512, 512, device=dev)
    C = torch.zeros(512, 512, device=dev)
    for field, value in (("a_split", 2), ("stages", plan.stages - 1), ("tile_k", 32), ("super_k", 96)):
        bad = phobos.phobos_gemm_plan(512, 512, 512, 512, 512, 512, fmt)
        setattr(bad, field, value)
        with pytest.raises(phobos.PhobosError):
            phobos.sgemm(A, A, C, 1.0, 0.0, math=fmt, plan=bad)
    # a 16-bit plan under another math mode is refused
    with pytest.raises(phobos.PhobosError):
        phobos.sgemm(A, A, C, 1.0, 0.0, math="3xtf32", plan=plan)


@pytest.mark.parametrize("fmt", FMTS)
def test_square_8192_sampled(dev, fmt):
    """The benchmark's workload and launch configuration, on sampled entries."""
    w = si.workload("sgemm_8192")
    A, B, C0 = w.A(), w.B(), w.C_old()
    dA, dB, dC = (torch.from_numpy(x).to(dev) for x in (A, B, C0))
    phobos.sgemm(dA, dB, dC, w.alpha, w.beta, math=fmt)
    torch.cuda.synchronize()
    rows, cols = w.samples()
    got = dC[torch.from_numpy(rows).to(dev), torch.from_numpy(cols).to(dev)].cpu().numpy()
    assert torch.isfinite(dC).all().item()
    del dA, dB, dC
    torch.cuda.empty_cache()
    ref, den = oracle.sgemm_entries(oracle.round_inputs(A, fmt), oracle.round_inputs(B, fmt), C0,
                                    w.alpha, w.beta, rows, cols)
    assert oracle.max_rel_error(got, ref, den) <= oracle.TOL_HALF_ACC
