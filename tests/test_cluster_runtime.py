"""The cluster runtime end to end on host-memory pods (no GPU).

The pods keep their arena in host memory, and the test's fp64 leaf
(tests/cluster_host.py) computes their step leaves. The rest is the
product's own code path:
  - the native planner and pod executor (arena, dependency-driven issue,
    storage I/O, two-phase STORE);
  - the scheduler and pod processes with their TCPStore control plane,
    heartbeats and re-plan.
The result is checked against the CPU oracle with the bound of the K-chunked
mode (2^-20 of sum |alpha a b| + |beta c|): the init leaf seeds beta*C_old,
and every chunk adds alpha*A_c*B_c ("Show HN: Phobos", "Matrix
Multiplication" and "The DAG Compiler").

The failures are made on the host, as the pages' failure model has it ("a
node misses its heartbeat"): a pod process exits between two instructions.
  - After a STORE, the scheduler re-plans that node's unstored outputs onto
    the nodes left.
  - After phase 1 of a STORE, the scheduler also finishes the staged tile
    from its side file.
"""
import os

import numpy as np
import pytest

import language_fp32_gemm_gb300 as phobos
import oracle
from language_fp32_gemm_gb300 import build as lib_build
from language_fp32_gemm_gb300 import cluster

import cluster_host


@pytest.fixture(scope="module", autouse=True)
def lib():
    lib_build.build()
    return phobos.library()


def check(job, A, B, C0):
    got = cluster_host.result(job)
    ref, den = oracle.sgemm(A, B, C0, job.alpha, job.beta)
    assert np.isfinite(got).all()
    err = oracle.max_rel_error(got, ref, den)
    assert err <= oracle.TOL_FP32, err


@pytest.mark.parametrize("beta", [0.0, -0.75])
def test_segments_in_process(tmp_path, beta):
    job, A, B, C0 = cluster_host.write_job(tmp_path, 203, 171, 150, 1.5, beta, seed=41, lo=(64, 48, 40))
    p = cluster.plan(job, 3, budget=1 << 20)
    stored = []
    for n in range(3):
        cluster.run_segment(p.segments[n], job, 1 << 20, cluster.DEVICE_HOST,
                            on_stored=stored.append, host_gemm=cluster_host.host_gemm)
    gm, gn = job.grid(64, 48)
    assert sorted(stored) == sorted(cluster.output_tile_ids(job, p.super).values())
    assert len(stored) == gm * gn
    assert not [f for f in os.listdir(tmp_path) if ".tile-" in f]  # side files removed
    check(job, A, B, C0)


def test_arena_smaller_than_peak_is_refused(tmp_path):
    job, A, B, C0 = cluster_host.write_job(tmp_path, 64, 64, 64, 1.0, 0.0, seed=42, lo=(32, 32, 32))
    p = cluster.plan(job, 1, budget=1 << 20)
    peak = cluster.segment_info(p.segments[0])["peak_bytes"]
    with pytest.raises(phobos.PhobosError) as e:
        cluster.run_segment(p.segments[0], job, peak - 256, cluster.DEVICE_HOST,
                            host_gemm=cluster_host.host_gemm)
    assert e.value.status == phobos.PHOBOS_ERR_OUT_OF_MEMORY
    before = np.fromfile(job.C.path, dtype=np.float32)
    assert np.array_equal(before, C0.ravel())  # nothing was stored


def test_hook_can_stop_a_pod(tmp_path):
    job, A, B, C0 = cluster_host.write_job(tmp_path, 64, 64, 64, 1.0, 0.5, seed=43, lo=(32, 32, 32))
    p = cluster.plan(job, 1, budget=1 << 20)
    with pytest.raises(phobos.PhobosError) as e:
        cluster.run_segment(p.segments[0], job, 1 << 20, cluster.DEVICE_HOST,
                            on_staged=lambda t: False, host_gemm=cluster_host.host_gemm)
    assert e.value.status == phobos.PHOBOS_ERR_INVALID_VALUE
    # phase 1 happened (a side file), phase 2 did not (C untouched)
    assert [f for f in os.listdir(tmp_path) if ".tile-" in f]
    assert np.array_equal(np.fromfile(job.C.path, dtype=np.float32), C0.ravel())


def test_three_pods(tmp_path):
    job, A, B, C0 = cluster_host.write_job(tmp_path, 260, 230, 190, 0.75, 0.25, seed=44, lo=(64, 64, 64))
    sc = cluster.run_local(job, 3, budget=1 << 20, device=cluster.DEVICE_HOST,
                           host_gemm=cluster_host.host_gemm, heartbeat_timeout=20.0, deadline=300)
    assert sc.replans == 0 and sc.exitcodes == [0, 0, 0]
    check(job, A, B, C0)


@pytest.mark.parametrize("phase", ["stored", "staged"])
def test_lost_node_is_replanned(tmp_path, phase):
    job, A, B, C0 = cluster_host.write_job(tmp_path, 300, 260, 130, 1.25, 0.5, seed=45, lo=(64, 64, 64))
    sc = cluster.run_local(job, 3, budget=1 << 20, device=cluster.DEVICE_HOST,
                           host_gemm=cluster_host.host_gemm, heartbeat_timeout=1.5,
                           fail={1: (phase, 1)}, deadline=300)
    assert sc.exitcodes[1] == 3 and sc.exitcodes[0] == 0 and sc.exitcodes[2] == 0
    assert sc.replans == 1
    kind, lost, redo = sc.log[-1]
    assert kind == "replan" and lost == [1]
    first = sc.first_plan.outputs[1]
    if phase == "stored":
        assert redo == first[1:]  # the first output was stored before the exit
    else:
        assert redo == first[1:]  # the staged one was finished from its side file
    check(job, A, B, C0)


def test_slow_node_declared_dead_stops_cleanly(tmp_path):
    """A pod that still runs but stops heart-beating is declared dead.

    Its unstored outputs are re-planned. The pod refuses to write into C from
    then on, since its staged hook sees the dead mark, and it leaves without
    reporting a failure. The result is complete and correct (beta != 0, so C
    is read in place)."""
    job, A, B, C0 = cluster_host.write_job(tmp_path, 256, 256, 96, 1.0, 0.5, seed=46, lo=(64, 64, 32))
    sc = cluster.run_local(job, 3, budget=1 << 20, device=cluster.DEVICE_HOST,
                           host_gemm=cluster_host.slow_host_gemm, heartbeat_timeout=1.0,
                           heartbeat_overrides={1: 30.0}, deadline=300)
    assert sc.replans >= 1
    assert any(kind == "replan" and lost == [1] for kind, lost, *_ in sc.log)
    assert sc.exitcodes == [0, 0, 0]
    check(job, A, B, C0)
