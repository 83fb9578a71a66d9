"""bench.py's multi-rank path on CPU: two gloo ranks, each an independent
replica, aggregate to the slowest rank's time and the whole job's rate."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [120.0, 150.0][rank]   # rank 1 is the slower replica
    max_ms, gflops = bench.aggregate_rate(local_ms, 2.0e9, 10, world)
    out[rank] = (max_ms, gflops)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_with_gloo():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    # both ranks see the slowest rank's time; the rate counts both replicas
    for r in range(2):
        max_ms, gflops = out[r]
        assert max_ms == 150.0
        assert gflops == pytest.approx(2 * 2.0e9 * 10 / 0.150 / 1e9)


def test_single_rank_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    max_ms, gflops = bench.aggregate_rate(50.0, 1.0e9, 4, 1)
    assert max_ms == 50.0 and gflops == pytest.approx(4 * 1.0e9 / 0.05 / 1e9)


def test_reference_arm_prints_one_contract_line():
    # The reference arm (the CPU oracle on a row sample) runs without a GPU:
    # its JSON line carries the keys the benchmark contract asks for.
    import json
    import subprocess
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload",
                          "sgemm_256", "--steps", "2", "--warmup", "1",
                          "--reference-budget", "3"],
                         cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GFLOP/s" and d["value"] > 0
    assert d["steps"] == 2 and d["warmup"] == 1 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "GFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == "sgemm_256"


def test_multicast_refused_under_a_two_rank_launch():
    # TMA multicast is a one-GPU option: bench.py launched as two ranks (the
    # way a multi-GPU run is launched) must refuse --multicast before it
    # touches a device or starts a process group.
    import subprocess
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--gpus", "2",
           "--steps", "1", "--warmup", "1", "--multicast"]
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert out.returncode != 0
    assert "--multicast runs on one GPU only" in out.stderr
    assert not [l for l in out.stdout.splitlines() if l.startswith("{")]
