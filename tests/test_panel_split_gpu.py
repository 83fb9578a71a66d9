"""The in-kernel panel split (plan a_split = 3) on the GPU, through the C ABI.

Two extra warps of every CTA split the caller's A and B into tf32 big/small
panels in the workspace while the GEMM runs, and each CTA's producer waits
only for the panels of its current tile.  The split values are the same
function of x as the pre-pass's and the tiles accumulate in the same order,
so the result must equal the pre-pass plan's bit for bit; it is also checked
against the CPU oracle.  Shapes cover ragged M, N and K (partial panels, K not
a multiple of 32 or of the 256-deep split item), padded leading dimensions,
pointers that are not 16-byte aligned (scalar loads), the K-chunked mode, the
tail split, and the host-buffer path whose later row bands reuse B.
"""
import numpy as np
import pytest

import language_fp32_gemm_gb300 as phobos
import oracle
import seeded_inputs as si
from gpu_util import padded, run_gemm, tolerance

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


def plan_for(M, N, K, lda, ldb, ldc, math, a_split, **fields):
    p = phobos.phobos_gemm_plan(M, N, K, lda, ldb, ldc, math)
    assert p.cluster_m == 2  # CTA pairs
    p.a_split = a_split
    for name, value in fields.items():
        setattr(p, name, value)
    return p


def bits(x):
    return np.ascontiguousarray(x).view(np.uint32)


SHAPES = [(512, 512, 256), (777, 1300, 1000), (300, 2000, 61), (2048, 1792, 1025),
          (1024, 768, 4096)]


@pytest.mark.parametrize("math", ["3xtf32", "tf32"])
@pytest.mark.parametrize("shape", SHAPES, ids=["x".join(map(str, s)) for s in SHAPES])
def test_panel_split_matches_the_oracle_and_the_prepass_bitwise(dev, shape, math):
    M, N, K = shape
    A = si.normal(111, 0, (M, K))
    B = si.normal(111, 1, (K, N))
    C0 = si.uniform_pm1(111, 2, (M, N))
    C3 = run_gemm(torch, dev, A, B, C0, 1.25, 0.5, math, plan=plan_for(M, N, K, K, N, N, math, 3))
    C1 = run_gemm(torch, dev, A, B, C0, 1.25, 0.5, math, plan=plan_for(M, N, K, K, N, N, math, 1))
    ref, den = oracle.sgemm(A, B, C0, 1.25, 0.5)
    assert oracle.max_rel_error(C3, ref, den) <= tolerance(math)
    assert np.array_equal(bits(C3), bits(C1))


@pytest.mark.parametrize("offsets", [(0, 0, 0), (1, 3, 2)], ids=["aligned", "unaligned"])
def test_panel_split_any_leading_dimension_and_alignment(dev, offsets):
    M, N, K = 640, 900, 517
    A = padded(si.normal(112, 0, (M, K)), 3)
    B = padded(si.normal(112, 1, (K, N)), 5)
    C0 = padded(si.uniform_pm1(112, 2, (M, N)), 2)
    lda, ldb, ldc = A.strides[0] // 4, B.strides[0] // 4, C0.strides[0] // 4
    plan = plan_for(M, N, K, lda, ldb, ldc, "3xtf32", 3)
    C = run_gemm(torch, dev, A, B, C0, 0.75, 0.25, "3xtf32", plan=plan, offsets=offsets)
    ref, den = oracle.sgemm(A, B, C0, 0.75, 0.25)
    assert oracle.max_rel_error(C, ref, den) <= oracle.TOL_FP32


def test_panel_split_integer_inputs_are_exact(dev):
    M, N, K = 700, 600, 333
    A = si.integers(113, 0, (M, K))
    B = si.integers(113, 1, (K, N))
    C0 = si.integers(113, 2, (M, N))
    C = run_gemm(torch, dev, A, B, C0, 1.5, 0.5, "3xtf32",
                 plan=plan_for(M, N, K, K, N, N, "3xtf32", 3))
    ref, _ = oracle.sgemm(A, B, C0, 1.5, 0.5)
    assert np.array_equal(C, ref.astype(np.float32))


@pytest.mark.parametrize("super_k", [512, 1024])
def test_panel_split_in_the_k_chunked_mode(dev, super_k):
    # one launch per K chunk, each splitting its own K range of A and B
    M, N, K = 1024, 1280, 3000
    A = si.normal(114, 0, (M, K))
    B = si.normal(114, 1, (K, N))
    C0 = si.uniform_pm1(114, 2, (M, N))
    plan = plan_for(M, N, K, K, N, N, "3xtf32", 3, super_k=super_k)
    C = run_gemm(torch, dev, A, B, C0, 1.0, 0.5, "3xtf32", plan=plan)
    ref, den = oracle.sgemm(A, B, C0, 1.0, 0.5)
    assert oracle.max_rel_error(C, ref, den) <= oracle.TOL_FP32


@pytest.mark.parametrize("tail_split", [1, 0, 3, 8])
def test_panel_split_with_the_tail_split(dev, tail_split):
    # 10 x 8 = 80 pair tiles: one wave over 76 pairs and a tail of 4 tiles,
    # whose pieces start inside K chunks
    M, N, K = 2560, 2048, 2048
    A = si.normal(115, 0, (M, K))
    B = si.normal(115, 1, (K, N))
    C0 = si.uniform_pm1(115, 2, (M, N))
    plan = plan_for(M, N, K, K, N, N, "3xtf32", 3, tail_split=tail_split)
    C = run_gemm(torch, dev, A, B, C0, 1.0, 1.0, "3xtf32", plan=plan)
    C1 = run_gemm(torch, dev, A, B, C0, 1.0, 1.0, "3xtf32",
                  plan=plan_for(M, N, K, K, N, N, "3xtf32", 1, tail_split=tail_split))
    ref, den = oracle.sgemm(A, B, C0, 1.0, 1.0)
    assert oracle.max_rel_error(C, ref, den) <= oracle.TOL_FP32
    assert np.array_equal(bits(C), bits(C1))


def test_panel_split_host_bands_reuse_the_split_of_b(dev):
    # phobos_sgemm_host runs M >= 2048 as row bands; N > 1536 takes the panel
    # split, and bands after the first reuse the first band's split of B.
    M, N, K = 4100, 1700, 300
    A = si.normal(116, 0, (M, K))
    B = si.normal(116, 1, (K, N))
    C0 = si.uniform_pm1(116, 2, (M, N))
    C = C0.copy()
    st = phobos.phobos_sgemm_host(M, N, K, 1.5, A.ctypes.data, K, B.ctypes.data, N, 0.5,
                                  C.ctypes.data, N, 0, phobos.PHOBOS_MATH_DEFAULT)
    assert st == phobos.PHOBOS_OK
    ref, den = oracle.sgemm(A, B, C0, 1.5, 0.5)
    assert oracle.max_rel_error(C, ref, den) <= oracle.TOL_FP32


@pytest.mark.parametrize("beta", [0.0, 0.5])
def test_host_bands_stream_b_in_k_chunks(dev, beta):
    # With K >= 2048 the first band runs as K-chunked step leaves, each waiting
    # for its own rows of B on the copy stream: 2048 rows in two bands, K =
    # 2500 in chunks of 512 (the last one 452 deep), N > 1536.
    M, N, K = 2048, 1700, 2500
    A = padded(si.normal(118, 0, (M, K)), 3)
    B = padded(si.normal(118, 1, (K, N)), 2)
    C0 = si.uniform_pm1(118, 2, (M, N))
    C = C0.copy()
    lda, ldb = A.strides[0] // 4, B.strides[0] // 4
    st = phobos.phobos_sgemm_host(M, N, K, 1.25, A.ctypes.data, lda, B.ctypes.data, ldb, beta,
                                  C.ctypes.data, N, 0, phobos.PHOBOS_MATH_DEFAULT)
    assert st == phobos.PHOBOS_OK
    ref, den = oracle.sgemm(A, B, C0, 1.25, beta)
    assert oracle.max_rel_error(C, ref, den) <= oracle.TOL_FP32


def test_panel_split_is_the_default_for_wide_split_tf32(dev):
    # The automatic choice (a_split = 0) takes the panel split for N > 1536;
    # the result equals the forced plan's bit for bit.
    M, N, K = 1536, 2048, 700
    A = si.normal(117, 0, (M, K))
    B = si.normal(117, 1, (K, N))
    C0 = si.uniform_pm1(117, 2, (M, N))
    auto = run_gemm(torch, dev, A, B, C0, 1.0, 0.5, "default")
    forced = run_gemm(torch, dev, A, B, C0, 1.0, 0.5, "3xtf32",
                      plan=plan_for(M, N, K, K, N, N, "3xtf32", 3))
    assert np.array_equal(bits(auto), bits(forced))
