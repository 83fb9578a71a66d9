"""The no-allocation split-TF32 entry point, through the C ABI.

phobos_sgemm_noalloc is for callers that may not allocate device memory
themselves: a serving process whose device memory its own allocator reserved
up front (a new cudaMalloc could fail or fragment that pool), or a
latency-critical loop that cannot take cudaMalloc/cudaFree's implicit
synchronisation.  Its scratch is a fixed array inside the library, shared by
every call.  These tests check that calls in a row each agree with the CPU
oracle and with the allocating entry point, within the 3xTF32 tolerance, and
that a problem too large for the fixed scratch is refused without touching C.

This file is named to be collected last; it passes alone or after the others.
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


def _noalloc(dA, dB, dC, alpha, beta, stream):
    M, K = dA.shape
    N = dB.shape[1]
    return phobos.phobos_sgemm_noalloc(M, N, K, alpha, dA.data_ptr(), K, dB.data_ptr(), N, beta,
                                       dC.data_ptr(), N, stream)


def test_calls_in_a_row_match_the_oracle_and_the_allocating_entry_point(dev):
    stream = torch.cuda.current_stream(dev).cuda_stream
    # Three calls in a row.  Each later problem is smaller than the first, so
    # stale operands of earlier calls sit in the shared scratch around its
    # buffers.  K = 2000 takes the 8-block TMEM partials of K above 1024.
    for seed, (M, N, K) in ((61, (1000, 900, 700)), (63, (256, 256, 2000)),
                            (62, (300, 260, 200))):
        A = si.normal(seed, 0, (M, K))
        B = si.normal(seed, 1, (K, N))
        C0 = si.uniform_pm1(seed, 2, (M, N))
        alpha, beta = 1.25, 0.5
        dA, dB = torch.from_numpy(A).to(dev), torch.from_numpy(B).to(dev)
        c_noalloc = torch.from_numpy(C0).to(dev)
        c_alloc = torch.from_numpy(C0).to(dev)
        st = _noalloc(dA, dB, c_noalloc, alpha, beta, stream)
        assert st == phobos.PHOBOS_OK, phobos.status_string(st)
        st = phobos.phobos_sgemm_ex(M, N, K, alpha, dA.data_ptr(), K, dB.data_ptr(), N, beta,
                                    c_alloc.data_ptr(), N, stream, phobos.PHOBOS_MATH_3XTF32)
        assert st == phobos.PHOBOS_OK, phobos.status_string(st)
        torch.cuda.synchronize()
        # no expired wait in either entry point's status word
        assert phobos.phobos_check_device(stream) == phobos.PHOBOS_OK
        got = c_noalloc.cpu().numpy()
        want = c_alloc.cpu().numpy().astype(np.float64)
        ref, den = oracle.sgemm(A, B, C0, alpha, beta)
        assert np.isfinite(got).all()
        assert oracle.max_rel_error(got, ref, den) <= oracle.TOL_FP32, (M, N, K)
        assert np.max(np.abs(got.astype(np.float64) - want) / den) <= oracle.TOL_FP32, (M, N, K)


def test_too_large_for_the_scratch_is_refused(dev):
    M = N = K = 4096  # split operands of 256 MiB > the fixed 64 MiB
    A = torch.zeros(M, K, device=dev)
    B = torch.zeros(K, N, device=dev)
    C = torch.full((M, N), 3.0, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    st = _noalloc(A, B, C, 1.0, 0.0, stream)
    assert st == phobos.PHOBOS_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert bool((C == 3.0).all())
