"""The cluster runtime with its pods on the GPU: every leaf is phobos_sgemm_ex.

Three pod processes share the one GPU, each with its own device arena, as the
pages' prototype ran its nodes on one machine with a slice of VRAM each
("Show HN: Phobos", "The Cluster Prototype"). Results are checked against the
CPU oracle with the K-chunked bound (2^-20).

The failure case makes one pod exit on the host right after its first STORE,
with no device work in flight. The scheduler must notice the missing
heartbeat and re-plan that node's other outputs onto the two pods left.
"""
import numpy as np
import pytest

import language_fp32_gemm_gb300 as phobos
import oracle
from language_fp32_gemm_gb300 import cluster

import cluster_host

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from language_fp32_gemm_gb300 import build as lib_build
    lib_build.build()
    return torch.device("cuda:0")


def check(job, A, B, C0):
    got = cluster_host.result(job)
    ref, den = oracle.sgemm(A, B, C0, job.alpha, job.beta)
    assert np.isfinite(got).all()
    err = oracle.max_rel_error(got, ref, den)
    assert err <= oracle.TOL_FP32, err


@pytest.mark.parametrize("beta", [0.0, 0.5])
def test_segments_in_process_on_the_gpu(tmp_path, beta):
    job, A, B, C0 = cluster_host.write_job(tmp_path, 777, 901, 655, 1.5, beta, seed=51, lo=(256, 384, 200))
    p = cluster.plan(job, 2, budget=32 << 20)
    for n in range(2):
        cluster.run_segment(p.segments[n], job, 32 << 20, cluster.DEVICE_CUDA, staging_bytes=1 << 20)
    torch.cuda.synchronize()
    assert phobos.phobos_check_device(0) == phobos.PHOBOS_OK
    check(job, A, B, C0)


def test_three_gpu_pods(tmp_path):
    job, A, B, C0 = cluster_host.write_job(tmp_path, 1536, 1280, 1000, 0.75, 0.5, seed=52, lo=(512, 512, 384))
    sc = cluster.run_local(job, 3, budget=64 << 20, heartbeat_timeout=20.0, deadline=600)
    assert sc.replans == 0 and sc.exitcodes == [0, 0, 0]
    check(job, A, B, C0)


def test_lost_gpu_pod_is_replanned(tmp_path):
    job, A, B, C0 = cluster_host.write_job(tmp_path, 1536, 1280, 1000, 1.25, -0.5, seed=53, lo=(512, 512, 384))
    sc = cluster.run_local(job, 3, budget=64 << 20, heartbeat_timeout=3.0, fail={1: ("stored", 1)},
                           deadline=600)
    assert sc.exitcodes[1] == 3 and sc.replans == 1
    check(job, A, B, C0)
