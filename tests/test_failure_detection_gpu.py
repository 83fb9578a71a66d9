"""Failure detection on the GPU without a GPU fault.

Every mbarrier wait in the tensor-core kernel is bounded (about two seconds);
when one expires the kernel records where in a device status word, stops all
of its roles (in every CTA of a pair or multicast cluster), releases its
tensor memory and returns.  PHOBOS_TEST_WITHHOLD_LOAD=1 makes the producer
skip the first operand load, so the MMA issuer's wait for it runs out;
PHOBOS_TEST_WITHHOLD_SPLIT=1 makes the in-kernel panel split never publish its
first item, so the producer's wait for that panel runs out.  The
test checks that the host reads PHOBOS_ERR_TIMEOUT and that the context stays
usable: the next call is correct.  Nothing here faults, traps or hangs the
GPU.
"""
import numpy as np
import pytest

import language_fp32_gemm_gb300 as phobos
import oracle
import seeded_inputs as si

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


@pytest.mark.parametrize("shape,multicast,a_split,withhold,clc", [
    ((128, 256, 96), 0, 0, "LOAD", 0), ((256, 256, 96), 0, 0, "LOAD", 0),
    ((256, 512, 96), 1, 0, "LOAD", 0), ((256, 256, 96), 0, 3, "LOAD", 0),
    ((256, 256, 96), 0, 3, "SPLIT", 0), ((2560, 2048, 96), 0, 1, "LOAD", 1),
    ((2560, 2048, 96), 0, 3, "LOAD", 1)],
    ids=["single_cta", "cta_pair", "multicast_cluster", "panel_split", "panel_split_flag",
         "cluster_launch_control", "cluster_launch_control_panel_split"])
def test_expired_wait_is_reported_and_context_survives(dev, shape, multicast, a_split, withhold,
                                                       clc, monkeypatch):
    # withhold = LOAD: the producer skips its first operand load and the MMA
    # issuer's wait expires; SPLIT (in-kernel panel split): the splitter never
    # publishes its first item's flag and the producer's wait for it expires.
    # With Cluster Launch Control (clc = 1) the 80 tiles outnumber the pairs
    # that fit at once: every pair times out on its first tile, after its
    # leader has asked for (and may have cancelled) a pair not yet launched.
    M, N, K = shape
    plan = phobos.phobos_gemm_plan(M, N, K, K, N, N, "3xtf32")
    assert plan.cluster_m == (2 if M > 128 else 1)
    if multicast:  # two CTA pairs sharing A through TMA multicast
        plan.multicast, plan.cluster_n = 1, 2
    plan.a_split = a_split  # 3: A and B split by the GEMM kernel's splitter warps
    plan.clc = clc
    A = si.normal(71, 0, (M, K))
    B = si.normal(71, 1, (K, N))
    dA, dB = torch.from_numpy(A).to(dev), torch.from_numpy(B).to(dev)
    dC = torch.full((M, N), 5.0, device=dev)
    assert phobos.phobos_check_device(0) == phobos.PHOBOS_OK  # nothing pending
    monkeypatch.setenv("PHOBOS_TEST_WITHHOLD_" + withhold, "1")
    phobos.sgemm(dA, dB, dC, 1.0, 0.0, math="3xtf32", plan=plan)
    st = phobos.phobos_check_device(0)
    monkeypatch.delenv("PHOBOS_TEST_WITHHOLD_" + withhold)
    assert st == phobos.PHOBOS_ERR_TIMEOUT, phobos.status_string(st)
    assert bool((dC == 5.0).all())  # the aborted kernel wrote nothing
    assert phobos.phobos_check_device(0) == phobos.PHOBOS_OK  # the word was cleared
    # the context is intact: a normal call gives the right answer
    phobos.sgemm(dA, dB, dC, 1.0, 0.0, math="3xtf32", plan=plan)
    assert phobos.phobos_check_device(0) == phobos.PHOBOS_OK
    ref, den = oracle.sgemm(A, B, None, 1.0, 0.0)
    assert oracle.max_rel_error(dC.cpu().numpy(), ref, den) <= oracle.TOL_FP32


def test_workspace_allocation_failure_is_reported(dev):
    # A workspace of about a terabyte cannot be allocated; the call must say so
    # before launching anything (no operand is read).
    M = N = 1 << 20
    K = 1 << 16
    x = torch.zeros(16, device=dev)
    st = phobos.phobos_sgemm_ex(M, N, K, 1.0, x.data_ptr(), K, x.data_ptr(), N, 0.0,
                                x.data_ptr(), N, 0, phobos.PHOBOS_MATH_3XTF32)
    assert st == phobos.PHOBOS_ERR_OUT_OF_MEMORY
    torch.cuda.synchronize()
    assert phobos.phobos_check_device(0) == phobos.PHOBOS_OK
