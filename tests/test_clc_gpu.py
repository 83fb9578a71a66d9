"""Cluster Launch Control (plan clc = 1) on the GPU, through the C ABI.

The grid holds one CTA pair per output tile; the pairs that fit on the GPU
start on their own tiles and take the others from the hardware by
cancelling the launch of pairs that have not started ("Clusters et DSMEM",
3.7, Cluster Launch Control).  Each tile is computed whole, in the same order
of operations as the static persistent walk without the tail split, so with
tail_split = 1 the result must equal that walk's bit for bit, whichever way
A and B are split, and the oracle's within the split-TF32 bound.  By default
the last partial wave's tiles are cut into K pieces, added by whichever piece
finishes last in a fixed order: checked against the oracle and against a
repeat run, bit for bit.  Shapes run
from one tile (every request cancels nothing) to far more tiles than pairs
fit at once (most tiles come from cancelled launches), with ragged edges,
padded leading dimensions and K-chunked launches.
"""
import numpy as np
import pytest

import language_fp32_gemm_gb300 as phobos
import oracle
import seeded_inputs as si
from gpu_util import padded, run_gemm

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


def plan_for(M, N, K, lda, ldb, ldc, **fields):
    p = phobos.phobos_gemm_plan(M, N, K, lda, ldb, ldc, "3xtf32")
    assert p.cluster_m == 2  # CTA pairs
    for name, value in fields.items():
        setattr(p, name, value)
    return p


def bits(x):
    return np.ascontiguousarray(x).view(np.uint32)


# tiles of 256 x 256: 1, 4, 16 (ragged), 80 and 256 (more than the 76 pairs
# that fit at once), 120 (ragged)
SHAPES = [(256, 256, 96), (512, 512, 256), (777, 1300, 1000), (2560, 2048, 2048),
          (4096, 4096, 512), (3001, 2500, 333)]


@pytest.mark.parametrize("a_split", [0, 1, 3], ids=["auto", "prepass", "panel_split"])
@pytest.mark.parametrize("shape", SHAPES, ids=["x".join(map(str, s)) for s in SHAPES])
def test_clc_equals_the_static_walk_bitwise(dev, shape, a_split):
    M, N, K = shape
    A = si.normal(121, 0, (M, K))
    B = si.normal(121, 1, (K, N))
    C0 = si.uniform_pm1(121, 2, (M, N))
    C = run_gemm(torch, dev, A, B, C0, 1.25, 0.5, "3xtf32",
                 plan=plan_for(M, N, K, K, N, N, clc=1, tail_split=1, a_split=a_split))
    S = run_gemm(torch, dev, A, B, C0, 1.25, 0.5, "3xtf32",
                 plan=plan_for(M, N, K, K, N, N, tail_split=1, a_split=a_split))
    ref, den = oracle.sgemm(A, B, C0, 1.25, 0.5)
    assert oracle.max_rel_error(C, ref, den) <= oracle.TOL_FP32
    assert np.array_equal(bits(C), bits(S))


@pytest.mark.parametrize("offsets", [(0, 0, 0), (1, 3, 2)], ids=["aligned", "unaligned"])
def test_clc_any_leading_dimension_and_alignment(dev, offsets):
    M, N, K = 1600, 2300, 517
    A = padded(si.normal(122, 0, (M, K)), 3)
    B = padded(si.normal(122, 1, (K, N)), 5)
    C0 = padded(si.uniform_pm1(122, 2, (M, N)), 2)
    lda, ldb, ldc = A.strides[0] // 4, B.strides[0] // 4, C0.strides[0] // 4
    C = run_gemm(torch, dev, A, B, C0, 0.75, 0.25, "3xtf32",
                 plan=plan_for(M, N, K, lda, ldb, ldc, clc=1), offsets=offsets)
    ref, den = oracle.sgemm(A, B, C0, 0.75, 0.25)
    assert oracle.max_rel_error(C, ref, den) <= oracle.TOL_FP32


@pytest.mark.parametrize("super_k", [512, 1024])
def test_clc_in_the_k_chunked_mode(dev, super_k):
    # one launch per K chunk, each dealing its tiles through its own queue
    M, N, K = 2304, 2560, 3000
    A = si.normal(123, 0, (M, K))
    B = si.normal(123, 1, (K, N))
    C0 = si.uniform_pm1(123, 2, (M, N))
    C = run_gemm(torch, dev, A, B, C0, 1.0, 0.5, "3xtf32",
                 plan=plan_for(M, N, K, K, N, N, clc=1, tail_split=1, super_k=super_k))
    S = run_gemm(torch, dev, A, B, C0, 1.0, 0.5, "3xtf32",
                 plan=plan_for(M, N, K, K, N, N, tail_split=1, super_k=super_k))
    P = run_gemm(torch, dev, A, B, C0, 1.0, 0.5, "3xtf32",
                 plan=plan_for(M, N, K, K, N, N, clc=1, super_k=super_k))  # tail pieces
    ref, den = oracle.sgemm(A, B, C0, 1.0, 0.5)
    assert oracle.max_rel_error(C, ref, den) <= oracle.TOL_FP32
    assert oracle.max_rel_error(P, ref, den) <= oracle.TOL_FP32
    assert np.array_equal(bits(C), bits(S))


# tail tiles: 4 of 80 (cut into 8 pieces), 28 of 256 (2 pieces), 12 of 240 (6)
TAIL_SHAPES = [(2560, 2048, 2048), (4096, 4096, 1024), (3001, 5003, 1999)]


@pytest.mark.parametrize("tail_split", [0, 3, 8], ids=["auto", "3_pieces", "8_pieces"])
@pytest.mark.parametrize("shape", TAIL_SHAPES, ids=["x".join(map(str, s)) for s in TAIL_SHAPES])
def test_clc_tail_pieces_match_the_oracle_and_repeat_bitwise(dev, shape, tail_split):
    # The last partial wave's tiles are cut into K pieces; every piece leaves
    # its partial sum behind and the last one to finish adds them in K order,
    # so the result does not depend on which piece finishes last.
    M, N, K = shape
    A = si.normal(126, 0, (M, K))
    B = si.normal(126, 1, (K, N))
    C0 = si.uniform_pm1(126, 2, (M, N))
    plan = plan_for(M, N, K, K, N, N, clc=1, tail_split=tail_split)
    C1 = run_gemm(torch, dev, A, B, C0, 1.25, 0.5, "3xtf32", plan=plan)
    C2 = run_gemm(torch, dev, A, B, C0, 1.25, 0.5, "3xtf32", plan=plan)
    ref, den = oracle.sgemm(A, B, C0, 1.25, 0.5)
    assert oracle.max_rel_error(C1, ref, den) <= oracle.TOL_FP32
    assert np.array_equal(bits(C1), bits(C2))


def test_clc_tail_pieces_integer_inputs_are_exact(dev):
    M, N, K = 4096, 4096, 1024  # 28 tail tiles in 2 pieces each
    A = si.integers(127, 0, (M, K))
    B = si.integers(127, 1, (K, N))
    C0 = si.integers(127, 2, (M, N))
    C = run_gemm(torch, dev, A, B, C0, 1.5, 0.5, "3xtf32", plan=plan_for(M, N, K, K, N, N, clc=1))
    ref, _ = oracle.sgemm(A, B, C0, 1.5, 0.5, want_den=False)
    assert np.array_equal(C, ref.astype(np.float32))  # integer sums below 2^24: exact


def test_clc_integer_inputs_are_exact_over_many_tiles(dev):
    # 1024 tiles, 13 times the pairs that fit at once
    M = N = 8192
    K = 160
    A = si.integers(124, 0, (M, K))
    B = si.integers(124, 1, (K, N))
    C0 = si.integers(124, 2, (M, N))
    C = run_gemm(torch, dev, A, B, C0, 1.5, 0.5, "3xtf32", plan=plan_for(M, N, K, K, N, N, clc=1))
    ref, _ = oracle.sgemm(A, B, C0, 1.5, 0.5, want_den=False)
    assert np.array_equal(C, ref.astype(np.float32))  # integer sums below 2^24: exact


@pytest.mark.parametrize("shape", [(2560, 2048, 256), (8192, 8192, 160)], ids=["80_tiles", "1024_tiles"])
def test_clc_tiles_come_from_cancelled_launches(dev, shape):
    # While timing events are set the leaders count the tiles they took from
    # cancelled launches.  At most 76 pairs fit on the GPU at once and none
    # exits while launches are pending, so all but those first pairs' tiles
    # must come from cancellations.
    M, N, K = shape
    tiles = (M // 256) * (N // 256)
    dA = torch.from_numpy(si.normal(125, 0, (M, K))).to(dev)
    dB = torch.from_numpy(si.normal(125, 1, (K, N))).to(dev)
    dC = torch.zeros((M, N), dtype=torch.float32, device=dev)
    plan = plan_for(M, N, K, K, N, N, clc=1, tail_split=1)  # whole tiles only
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()  # torch creates the CUDA events on their first record
    stop.record()
    torch.cuda.synchronize()
    phobos.phobos_kernel_clc_tiles()  # clear
    phobos.phobos_set_timing_events(start.cuda_event, stop.cuda_event)
    try:
        phobos.sgemm(dA, dB, dC, 1.0, 0.0, math="3xtf32", plan=plan)
    finally:
        phobos.phobos_set_timing_events(None, None)
    n = phobos.phobos_kernel_clc_tiles()
    assert phobos.phobos_check_device(0) == phobos.PHOBOS_OK
    assert tiles - 76 <= n <= tiles - 1, (n, tiles)
    phobos.sgemm(dA, dB, dC, 1.0, 0.0, math="3xtf32", plan=plan)
    assert phobos.phobos_kernel_clc_tiles() == 0  # not timed: not counted


def test_clc_beside_work_on_another_stream(dev):
    # Matrix products queued on another stream may hold SMs when the GEMM
    # starts: pairs that do not fit start later, and the hardware deals the
    # remaining tiles to the pairs that run.  Each tile is computed the same
    # way whoever takes it, so the result equals the static walk's.
    M, N, K = 4096, 4096, 1024
    A = si.normal(128, 0, (M, K))
    B = si.normal(128, 1, (K, N))
    C0 = si.uniform_pm1(128, 2, (M, N))
    dA, dB = torch.from_numpy(A).to(dev), torch.from_numpy(B).to(dev)
    dC = torch.from_numpy(C0).to(dev)
    X = torch.randn(8192, 8192, device=dev, dtype=torch.bfloat16)
    other = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(other):
        for _ in range(4):
            X @ X
    phobos.sgemm(dA, dB, dC, 1.0, 0.5, math="3xtf32",
                 plan=plan_for(M, N, K, K, N, N, clc=1, tail_split=1))
    torch.cuda.synchronize()
    assert phobos.phobos_check_device(0) == phobos.PHOBOS_OK
    S = run_gemm(torch, dev, A, B, C0, 1.0, 0.5, "3xtf32",
                 plan=plan_for(M, N, K, K, N, N, tail_split=1))
    assert np.array_equal(bits(dC.cpu().numpy()), bits(S))
