"""GPU parity of the multicast cluster mode of the tensor-core path.

With plan.multicast = 1 (cluster 2 x 2) a thread-block cluster holds two CTA
pairs that compute horizontally adjacent 256 x 256 tiles.  Both need the same
rows of A, so each pair TMA-loads half of them and multicasts it into the
shared-memory rings of both pairs (the "Clusters et DSMEM" chapter, section
3.5; the super-tile of the "@cluster" page maps onto such a cluster).  B stays
per pair.

Every case is checked against the CPU oracle with the bars of the other
tensor-core tests.  Tiles computed whole (no tail split) see the same MMA
sequence as in the pair kernel, so there the two kernels must agree bit for
bit.
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


def plan_for(M, N, K, math, multicast, lda=None, ldb=None, ldc=None, **fields):
    plan = phobos.phobos_gemm_plan(M, N, K, lda or K, ldb or N, ldc or N, math)
    assert plan.cluster_m == 2 and plan.tile_n == 256
    if multicast:
        plan.multicast = 1
        plan.cluster_n = 2
    for name, value in fields.items():
        setattr(plan, name, value)
    return plan


def check(dev, A, B, C0, alpha, beta, math, plan, offsets=(0, 0, 0)):
    C = run_gemm(torch, dev, A, B, C0, alpha, beta, math, plan=plan, offsets=offsets)
    ref, den = oracle.sgemm(A, B, C0, alpha, beta)
    err = oracle.max_rel_error(C, ref, den)
    assert err <= tolerance(math), "%s: max rel error %.3g" % (math, err)
    return C


@pytest.mark.parametrize("math", ["3xtf32", "tf32"])
@pytest.mark.parametrize("shape", [
    (512, 512, 256),     # one cluster tile
    (300, 260, 200),     # ragged edges inside one cluster tile
    (1000, 700, 332),    # 3 tile columns: the last cluster's second pair is past N
    (777, 1290, 333),    # ragged edges, short K
    (1536, 2048, 1024),  # 24 cluster tiles: more than one wave on some clusters
], ids=lambda s: "%dx%dx%d" % s)
def test_multicast_matches_oracle_and_pair_kernel(dev, math, shape):
    M, N, K = shape
    A = si.normal(111, 0, (M, K))
    B = si.normal(111, 1, (K, N))
    C0 = si.uniform_pm1(111, 2, (M, N))
    C_mc = check(dev, A, B, C0, 1.25, 0.75, math, plan_for(M, N, K, math, True, tail_split=1))
    C_pair = check(dev, A, B, C0, 1.25, 0.75, math, plan_for(M, N, K, math, False, tail_split=1))
    # the same tiles with the same MMA sequence: the same bits
    assert np.array_equal(C_mc, C_pair)


@pytest.mark.parametrize("math", ["3xtf32", "tf32"])
@pytest.mark.parametrize("shape,split,super_k", [
    ((512, 512, 2048), 0, None),     # one cluster tile: automatic split over idle clusters
    ((512, 512, 2048), 3, None),     # forced, uneven K pieces
    ((2560, 2560, 2048), 8, None),   # 50 cluster tiles: tail shares across tiles
    ((2500, 2510, 1100), 8, 512),    # the same inside K chunks, ragged edges
    ((520, 390, 2100), 0, 512),      # split inside every K chunk of the cluster split
    # 3 tile columns: the second pair of each last cluster is past N, yet it
    # still computes (zeros) and hands over its tail pieces
    ((1000, 700, 2048), 0, None),
    ((1000, 700, 2048), 3, None),
], ids=lambda v: str(v))
def test_multicast_tail_split_and_k_chunks(dev, math, shape, split, super_k):
    M, N, K = shape
    fields = {"tail_split": split}
    if super_k is not None:
        fields["super_k"] = super_k
    plan = plan_for(M, N, K, math, True, **fields)
    A = si.normal(112, 0, (M, K))
    B = si.normal(112, 1, (K, N))
    C0 = si.uniform_pm1(112, 2, (M, N))
    C1 = check(dev, A, B, C0, 0.5, 1.5, math, plan)
    C2 = run_gemm(torch, dev, A, B, C0, 0.5, 1.5, math, plan=plan)
    assert np.array_equal(C1, C2)  # deterministic


@pytest.mark.parametrize("math", ["3xtf32", "tf32"])
def test_multicast_integer_inputs_bit_exact(dev, math):
    M, N, K = 640, 768, 256
    A = si.integers(113, 0, (M, K))
    B = si.integers(113, 1, (K, N))
    C0 = si.integers(113, 2, (M, N))
    C = run_gemm(torch, dev, A, B, C0, 1.5, 0.5, math, plan=plan_for(M, N, K, math, True))
    ref, _ = oracle.sgemm(A, B, C0, 1.5, 0.5)
    assert np.array_equal(C, ref.astype(np.float32))


def test_multicast_padded_and_unaligned_operands(dev):
    M, N, K = 700, 900, 300
    A = padded(si.normal(114, 0, (M, K)), 3)
    B = padded(si.normal(114, 1, (K, N)), 1)
    C0 = padded(si.uniform_pm1(114, 2, (M, N)), 5)
    lda, ldb, ldc = A.strides[0] // 4, B.strides[0] // 4, C0.strides[0] // 4
    plan = plan_for(M, N, K, "3xtf32", True, lda, ldb, ldc)
    check(dev, A, B, C0, -0.75, 0.25, "3xtf32", plan, offsets=(1, 3, 1))


def test_multicast_headline_shape_sampled(dev):
    # 8192^3 with the benchmark's inputs, checked on seeded sampled entries
    w = si.workload("sgemm_8192")
    A, B, C0 = w.A(), w.B(), w.C_old()
    dA, dB, dC = (torch.from_numpy(x).to(dev) for x in (A, B, C0))
    plan = plan_for(w.M, w.N, w.K, "3xtf32", True)
    phobos.sgemm(dA, dB, dC, w.alpha, w.beta, math="3xtf32", plan=plan)
    torch.cuda.synchronize()
    assert phobos.phobos_check_device(0) == phobos.PHOBOS_OK
    rows, cols = w.samples()
    got = dC[torch.from_numpy(rows).to(dev), torch.from_numpy(cols).to(dev)].cpu().numpy()
    del dA, dB, dC
    torch.cuda.empty_cache()
    ref, den = oracle.sgemm_entries(A, B, C0, w.alpha, w.beta, rows, cols)
    assert oracle.max_rel_error(got, ref, den) <= oracle.TOL_FP32


def test_multicast_plan_needs_pairs_and_tf32(dev):
    M, N, K = 512, 512, 256
    A = torch.zeros(M, K, device=dev)
    B = torch.zeros(K, N, device=dev)
    C = torch.zeros(M, N, device=dev)
    bad = plan_for(M, N, K, "3xtf32", True, a_split=2)  # A split inside the kernel
    with pytest.raises(phobos.PhobosError) as e:
        phobos.sgemm(A, B, C, 1.0, 0.0, math="3xtf32", plan=bad)
    assert e.value.status == phobos.PHOBOS_ERR_UNSUPPORTED
    bad = phobos.phobos_gemm_plan(M, N, K, K, N, N, "bf16")
    bad.multicast, bad.cluster_n = 1, 2
    with pytest.raises(phobos.PhobosError) as e:
        phobos.sgemm(A, B, C, 1.0, 0.0, math="bf16", plan=bad)
    assert e.value.status == phobos.PHOBOS_ERR_UNSUPPORTED
