"""The cluster runtime's planner (host logic, no GPU).

Pinned to what the pages print for their cluster prototype ("Show HN: Phobos",
"The Cluster Prototype"): SGEMM at M = N = K = 20480 with 10240 super-tiles
on 4 nodes plans 72 instructions, 18 per node (5 ALLOC, 4 LOAD, 3 COMPUTE,
1 STORE, 5 FREE), with a peak of 1.2 GiB resident per node. Placement follows
the "@cluster" attribute page ("What runs today": super-tiles dealt round
robin by row-major index). FREE placement follows "The DAG Compiler": each
FREE comes after the last use of its tile.
"""
import pytest

import language_fp32_gemm_gb300 as phobos
from language_fp32_gemm_gb300 import build as lib_build
from language_fp32_gemm_gb300 import cluster

GiB = 1 << 30


@pytest.fixture(scope="module", autouse=True)
def lib():
    lib_build.build()
    return phobos.library()


def job_of(M, N, K, beta=0.0, lo=(4096, 4096, 4096), hi=None, alpha=1.0):
    t = lambda n, s: cluster.Tensor(n, "read" if n != "C" else "readwrite", s, "/nonexistent/" + n)
    return cluster.Job(M, N, K, alpha, beta, t("A", (M, K)), t("B", (K, N)), t("C", (M, N)),
                       tuple(lo), tuple(hi or lo))


def test_pages_prototype_instruction_counts():
    job = job_of(20480, 20480, 20480, beta=0.0, lo=(10240, 10240, 10240))
    p = cluster.plan(job, 4, budget=int(1.4 * GiB))
    assert p.super == (10240, 10240, 10240)
    total = 0
    for n in range(4):
        info = cluster.segment_info(p.segments[n])
        ops = info["ops"]
        assert info["instrs"] == 18
        assert (ops["ALLOC"], ops["LOAD"], ops["INIT"] + ops["STEP"], ops["STORE"], ops["FREE"]) == (5, 4, 3, 1, 5)
        # C, one A and one B tile of 10240^2 fp32 (400 MiB each) at once
        assert info["peak_bytes"] == 3 * 10240 * 10240 * 4
        assert round(info["peak_bytes"] / GiB, 1) == 1.2
        total += info["instrs"]
    assert total == 72
    assert p.outputs == {0: [0], 1: [1], 2: [2], 3: [3]}


def test_beta_loads_c_first():
    job = job_of(20480, 20480, 20480, beta=0.5, lo=(10240, 10240, 10240))
    p = cluster.plan(job, 4, budget=2 * GiB)
    ins = cluster.segment_instrs(p.segments[0])
    assert [i["op"] for i in ins[:3]] == ["ALLOC", "LOAD", "INIT"]
    assert ins[1]["tensor"] == "C"
    assert cluster.segment_info(p.segments[0])["ops"]["LOAD"] == 5


def test_round_robin_placement_and_ragged_edges():
    job = job_of(1000, 1100, 300, lo=(384, 384, 128))
    p = cluster.plan(job, 4, budget=64 << 20)
    gm, gn = job.grid(384, 384)
    assert (gm, gn) == (3, 3)
    assert p.outputs == {0: [0, 4, 8], 1: [1, 5], 2: [2, 6], 3: [3, 7]}
    seen = {}
    for n, blob in p.segments.items():
        for i in cluster.segment_instrs(blob):
            if i["op"] == "STORE":
                seen[(i["row0"], i["col0"])] = (i["rows"], i["cols"])
    assert seen[(768, 768)] == (1000 - 768, 1100 - 768)
    assert sum(r * c for r, c in seen.values()) == 1000 * 1100
    # K chunks of 128, 128 and 44
    steps = [i for i in cluster.segment_instrs(p.segments[0]) if i["op"] == "ALLOC" and i["tensor"] == "A"]
    assert [s["cols"] for s in steps[:3]] == [128, 128, 44]


@pytest.mark.parametrize("beta", [0.0, 0.5])
def test_free_pass_and_dependencies(beta):
    job = job_of(700, 900, 500, beta=beta, lo=(256, 256, 192))
    p = cluster.plan(job, 3, budget=64 << 20)
    for blob in p.segments.values():
        ins = cluster.segment_instrs(blob)
        freed = {}
        allocated = set()
        for k, i in enumerate(ins):
            for d in i["deps"]:
                assert 0 <= d < k
            if i["op"] == "ALLOC":
                assert i["buf"] == k
                allocated.add(k)
                continue
            bufs = [b for b in (i["buf"], i["buf_a"], i["buf_b"]) if b >= 0]
            for b in bufs:
                assert b in allocated and b not in freed, (k, i)
            if i["op"] == "FREE":
                b = i["buf"]
                freed[b] = k
                users = [j for j, u in enumerate(ins[:k]) if u["op"] not in ("ALLOC", "FREE")
                         and b in (u["buf"], u["buf_a"], u["buf_b"])]
                # the FREE follows the last use at once and waits for every user
                assert sorted(i["deps"]) == users
                assert users[-1] == k - 1 or ins[k - 1]["op"] == "FREE"
            if i["op"] == "STEP":
                assert ins[i["buf_a"]]["tensor"] == "A" and ins[i["buf_b"]]["tensor"] == "B"
                loads = [d for d in i["deps"] if ins[d]["op"] == "LOAD"]
                assert len(loads) == 2
        assert set(freed) == allocated  # every buffer freed exactly once


def test_tile_ids_are_deterministic_across_replans():
    job = job_of(1024, 1024, 512, lo=(256, 256, 256))
    full = cluster.plan(job, 4, budget=64 << 20)
    ids = cluster.output_tile_ids(job, full.super)
    stores = {}
    for n, blob in full.segments.items():
        for i in cluster.segment_instrs(blob):
            if i["op"] == "STORE":
                stores[i["tile"]] = n
    assert set(stores) == set(ids.values())
    # node 1 lost: its outputs go round robin over 0, 2, 3 with the same ids
    lost = full.outputs[1]
    re = cluster.plan(job, 4, budget=64 << 20, outputs=lost, live=[0, 2, 3], super_sizes=full.super)
    assert cluster.segment_info(re.segments[1])["instrs"] == 0
    assert re.outputs == {0: [lost[0], lost[3]], 2: [lost[1]], 3: [lost[2]]}
    got = {i["tile"] for b in re.segments.values() for i in cluster.segment_instrs(b) if i["op"] == "STORE"}
    assert got == {ids[o] for o in lost}
    assert cluster.tile_id(cluster.TENSOR_C, 2, 3, 1) != cluster.tile_id(cluster.TENSOR_C, 2, 1, 3)


def test_autotune_ranks_by_model_and_respects_budget():
    job = job_of(8192, 8192, 8192, lo=(1024, 1024, 1024), hi=(4096, 4096, 4096))
    # a tight budget: C + A + B tiles of 2048^2 fp32 (48 MiB) fit, 4096^2 do not
    small = cluster.plan(job, 4, budget=64 << 20, autotune=True, storage_gbs=2.0)
    sm, sn, sk = small.super
    assert 4 * (sm * sn + sm * sk + sk * sn) <= 64 << 20
    for blob in small.segments.values():
        assert cluster.segment_info(blob)["peak_bytes"] <= 64 << 20
    # storage-bound model: larger output tiles reload less
    big = cluster.plan(job, 4, budget=2 * GiB, autotune=True, storage_gbs=0.5)
    assert big.super[0] * big.super[1] >= sm * sn
    # every node keeps a super-tile when a candidate allows it
    assert all(cluster.segment_info(b)["outputs"] > 0 for b in big.segments.values())


def test_errors():
    job = job_of(512, 512, 512, lo=(256, 256, 256))
    with pytest.raises(phobos.PhobosError) as e:
        cluster.plan(job, 2, budget=1024)  # nothing fits
    assert e.value.status == phobos.PHOBOS_ERR_OUT_OF_MEMORY
    with pytest.raises(phobos.PhobosError):
        cluster.plan(job, 2, budget=64 << 20, live=[0, 0])
    with pytest.raises(phobos.PhobosError):
        cluster.plan(job, 2, budget=64 << 20, live=[2])
    with pytest.raises(phobos.PhobosError):
        cluster.plan(job, 2, budget=64 << 20, outputs=[3, 1], super_sizes=(256, 256, 256))
    with pytest.raises(phobos.PhobosError):
        cluster.plan(job_of(512, 512, 512, lo=(256, 256, 256), hi=(128, 128, 128)), 2, budget=64 << 20)
    lib = cluster._lib()
    assert lib.phobos_cl_segment_info(b"junk", 4, None) != 0


def test_job_file_round_trip(tmp_path):
    job = job_of(300, 200, 100, beta=0.25, lo=(128, 64, 32), hi=(256, 128, 64))
    text = cluster.job_text(job)
    back = cluster.parse_job(text)
    assert (back.M, back.N, back.K, back.alpha, back.beta) == (300, 200, 100, 1.0, 0.25)
    assert back.super_lo == (128, 64, 32) and back.super_hi == (256, 128, 64)
    with pytest.raises(ValueError):
        cluster.parse_job(text.replace("readwrite", "write"))  # beta != 0 reads C
    with pytest.raises(ValueError):
        cluster.parse_job(text.replace("source = sgemm", "source = attention"))
    with pytest.raises(ValueError):
        cluster.parse_job(text.replace("300x100", "300x101"))
