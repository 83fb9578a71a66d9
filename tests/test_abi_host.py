"""Host-side checks of the C ABI: the library loads, exports what the header
declares, validates arguments and plans without touching a GPU."""
import os
import re
import subprocess

import pytest

import language_fp32_gemm_gb300 as phobos
from language_fp32_gemm_gb300 import build as lib_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "phobos_gemm.h")
CLUSTER_HEADER = os.path.join(ROOT, "include", "phobos_cluster.h")


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    return phobos.library()


def declared_functions(header=HEADER):
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"\(\*\w+\)\s*\(", "(", text)  # function-pointer members are not exports
    return sorted(set(re.findall(r"\b(phobos_\w+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    assert set(names) == set(phobos.ABI_FUNCTIONS), names


def test_cluster_header_declares_the_cluster_abi():
    from language_fp32_gemm_gb300 import cluster
    names = declared_functions(CLUSTER_HEADER)
    assert set(names) == set(cluster.CLUSTER_ABI_FUNCTIONS), names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", phobos.LIBRARY_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\s[TW]\s+(\w+)$", out, flags=re.M))
    for name in declared_functions() + declared_functions(CLUSTER_HEADER):
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_status_strings(lib):
    for code in range(6):
        assert phobos.status_string(code).startswith("PHOBOS_")
    assert "unknown" in phobos.status_string(99)


@pytest.mark.parametrize("args", [
    (-1, 4, 4, 4, 4, 4),      # negative M
    (4, -1, 4, 4, 4, 4),      # negative N
    (4, 4, -1, 4, 4, 4),      # negative K
    (4, 4, 8, 7, 4, 4),       # lda < K
    (4, 8, 4, 4, 7, 8),       # ldb < N
    (4, 8, 4, 4, 8, 7),       # ldc < N
])
def test_invalid_sizes_rejected_before_any_device_call(lib, args):
    M, N, K, lda, ldb, ldc = args
    st = phobos.phobos_sgemm(M, N, K, 1.0, 16, lda, 16, ldb, 0.0, 16, ldc, 0)
    assert st == phobos.PHOBOS_ERR_INVALID_VALUE
    with pytest.raises(phobos.PhobosError):
        phobos.phobos_gemm_plan(M, N, K, lda, ldb, ldc)


def test_null_pointers_rejected(lib):
    assert phobos.phobos_sgemm(4, 4, 4, 1.0, 0, 4, 16, 4, 0.0, 16, 4, 0) == phobos.PHOBOS_ERR_INVALID_VALUE
    assert phobos.phobos_sgemm(4, 4, 4, 1.0, 16, 4, 0, 4, 0.0, 16, 4, 0) == phobos.PHOBOS_ERR_INVALID_VALUE
    assert phobos.phobos_sgemm(4, 4, 4, 1.0, 16, 4, 16, 4, 0.0, 0, 4, 0) == phobos.PHOBOS_ERR_INVALID_VALUE
    assert phobos.phobos_sgemm_ex(4, 4, 4, 1.0, 16, 4, 16, 4, 0.0, 16, 4, 0, 7) == phobos.PHOBOS_ERR_INVALID_VALUE


def test_empty_output_is_a_no_op(lib):
    assert phobos.phobos_sgemm(0, 5, 5, 1.0, 0, 5, 0, 5, 0.0, 0, 5, 0) == phobos.PHOBOS_OK
    assert phobos.phobos_sgemm(5, 0, 5, 1.0, 0, 5, 0, 1, 0.0, 0, 1, 0) == phobos.PHOBOS_OK


def test_plan_paths(lib):
    p = phobos.phobos_gemm_plan(256, 256, 256, 256, 256, 256)
    assert p.path == phobos.PHOBOS_PATH_FFMA and p.workspace_bytes == 0
    p = phobos.phobos_gemm_plan(8192, 8192, 8192, 8192, 8192, 8192)
    assert p.path == phobos.PHOBOS_PATH_3XTF32
    assert p.tile_m == 256 and p.cluster_m == 2 and p.tile_n == 256 and p.tile_k == 32
    assert p.stages >= 2
    assert p.super_k == 8192 and p.super_m == 4096 and p.tail_split == 0
    # split operands: (Mp + Np) * Kp * 4 bytes, big and small
    assert p.workspace_bytes == 2 * (8192 + 8192) * 8192 * 4
    p = phobos.phobos_gemm_plan(8192, 8192, 8192, 8192, 8192, 8192, "tf32")
    assert p.path == phobos.PHOBOS_PATH_TF32 and p.workspace_bytes == (8192 + 8192) * 8192 * 4
    p = phobos.phobos_gemm_plan(3001, 5003, 1999, 1999, 5003, 5003)
    Mp, Np, Kp = 3072, 5120, 2016  # 256-row pair tiles, 256-column tiles, K blocks of 32
    assert p.workspace_bytes == 2 * (Mp * Kp * 4 + Np * Kp * 4)
    p = phobos.phobos_gemm_plan(65536, 256, 4096, 4096, 256, 256)
    assert p.tile_n == 256
    p = phobos.phobos_gemm_plan(4096, 100, 4096, 4096, 100, 100)
    assert p.tile_n == 128 and p.tile_m == 128 and p.cluster_m == 1
    p = phobos.phobos_gemm_plan(128, 4096, 4096, 4096, 4096, 4096)
    assert p.tile_m == 128 and p.cluster_m == 1
    p = phobos.phobos_gemm_plan(8, 4096, 4096, 4096, 4096, 4096)
    assert p.path == phobos.PHOBOS_PATH_FFMA


def test_plan_raster_groups(lib):
    # 4096-row raster groups, the pages' smallest super-tile; 2048 rows when
    # the kernel splits A and B itself (split TF32, CTA pairs, N > 1536) and a
    # 4096-row group would cover all of M.
    plan = lambda M, N, K, math="default": phobos.phobos_gemm_plan(M, N, K, K, N, N, math)
    assert plan(4096, 4096, 4096).super_m == 2048
    assert plan(3001, 5003, 1999).super_m == 2048
    assert plan(8192, 8192, 8192).super_m == 4096
    assert plan(16384, 16384, 16384).super_m == 4096
    assert plan(4096, 1024, 4096).super_m == 4096        # A split in shared memory
    assert plan(4096, 4096, 4096, "tf32").super_m == 4096
    assert plan(65536, 256, 4096).super_m == 4096


def test_kernel_clock_reader_rejects_null(lib):
    # argument checks before any device call
    assert lib.phobos_kernel_clock_mhz(None) == phobos.PHOBOS_ERR_INVALID_VALUE
    assert lib.phobos_kernel_clc_tiles(None) == phobos.PHOBOS_ERR_INVALID_VALUE


def test_plan_rejects_unknown_math(lib):
    with pytest.raises(phobos.PhobosError):
        phobos.phobos_gemm_plan(16, 16, 16, 16, 16, 16, 9)


def test_dimensions_beyond_the_kernels_int_range_are_refused(lib):
    big = 1 << 31  # the kernels index rows and columns with 32-bit ints
    with pytest.raises(phobos.PhobosError) as e:
        phobos.phobos_gemm_plan(big, 4, 4, 4, 4, 4)
    assert e.value.status == phobos.PHOBOS_ERR_UNSUPPORTED
    assert phobos.phobos_sgemm(4, big, 4, 1.0, 16, big, 16, big, 0.0, 16, big, 0) == \
        phobos.PHOBOS_ERR_UNSUPPORTED


def test_multicast_plans_are_validated_before_any_device_call(lib):
    M = N = K = 1024

    def run(plan, math=phobos.PHOBOS_MATH_3XTF32):
        return phobos.phobos_sgemm_ex(M, N, K, 1.0, 16, K, 16, N, 0.0, 16, N, 0, math, plan)

    def mc(math="3xtf32", **fields):
        p = phobos.phobos_gemm_plan(M, N, K, K, N, N, math)
        p.multicast, p.cluster_n = 1, 2
        for name, value in fields.items():
            setattr(p, name, value)
        return p

    assert run(mc(cluster_n=1)) == phobos.PHOBOS_ERR_UNSUPPORTED   # multicast needs 2 x 2
    assert run(mc(multicast=2)) == phobos.PHOBOS_ERR_INVALID_VALUE
    assert run(mc(a_split=2)) == phobos.PHOBOS_ERR_UNSUPPORTED     # A split inside the kernel
    p = mc()
    p.stages -= 1
    assert run(p) == phobos.PHOBOS_ERR_INVALID_VALUE               # the deepest ring only
    assert run(mc("bf16"), phobos.PHOBOS_MATH_BF16) == phobos.PHOBOS_ERR_UNSUPPORTED
    p = phobos.phobos_gemm_plan(M, N, K, K, N, N, "3xtf32")
    p.cluster_n = 2                                                 # 2 x 2 without multicast
    assert run(p) == phobos.PHOBOS_ERR_UNSUPPORTED
    single = phobos.phobos_gemm_plan(128, N, K, K, N, N, "3xtf32")
    assert single.cluster_m == 1
    single.multicast, single.cluster_n = 1, 2                      # single CTAs: no pairs
    assert phobos.phobos_sgemm_ex(128, N, K, 1.0, 16, K, 16, N, 0.0, 16, N, 0,
                                  phobos.PHOBOS_MATH_3XTF32, single) == phobos.PHOBOS_ERR_UNSUPPORTED


def test_cluster_launch_control_plans_are_validated_before_any_device_call(lib):
    # clc = 1: split-TF32 CTA pairs reading A from the workspace only
    M = N = K = 1024

    def run(plan, math=phobos.PHOBOS_MATH_3XTF32, m=M):
        return phobos.phobos_sgemm_ex(m, N, K, 1.0, 16, K, 16, N, 0.0, 16, N, 0, math, plan)

    def clc(math="3xtf32", m=M, **fields):
        p = phobos.phobos_gemm_plan(m, N, K, K, N, N, math)
        p.clc = 1
        for name, value in fields.items():
            setattr(p, name, value)
        return p

    assert phobos.phobos_gemm_plan(M, N, K, K, N, N, "3xtf32").clc == 0  # never chosen by itself
    assert run(clc(clc=2)) == phobos.PHOBOS_ERR_INVALID_VALUE
    assert run(clc(a_split=2)) == phobos.PHOBOS_ERR_UNSUPPORTED    # A split in shared memory
    assert run(clc(multicast=1, cluster_n=2)) == phobos.PHOBOS_ERR_UNSUPPORTED
    assert run(clc("tf32"), phobos.PHOBOS_MATH_TF32) == phobos.PHOBOS_ERR_UNSUPPORTED
    assert run(clc("bf16"), phobos.PHOBOS_MATH_BF16) == phobos.PHOBOS_ERR_UNSUPPORTED
    single = clc(m=128)
    assert single.cluster_m == 1
    assert run(single, m=128) == phobos.PHOBOS_ERR_UNSUPPORTED     # CTA pairs only
    ffma = clc("ffma")
    assert run(ffma, phobos.PHOBOS_MATH_FFMA) == phobos.PHOBOS_ERR_UNSUPPORTED


@pytest.mark.parametrize("var", ["WORLD_SIZE", "LOCAL_WORLD_SIZE"])
def test_multicast_refused_in_a_rank_of_a_multi_gpu_job(lib, monkeypatch, var):
    # TMA multicast is a one-GPU option: a process launched as one rank of a
    # multi-process job gets PHOBOS_ERR_UNSUPPORTED for a valid multicast plan,
    # before any device call; the same plan without multicast is not refused
    # by that rule (it fails later here only for want of a GPU).
    M = N = K = 1024
    p = phobos.phobos_gemm_plan(M, N, K, K, N, N, "3xtf32")
    p.multicast, p.cluster_n = 1, 2
    monkeypatch.setenv(var, "2")
    st = phobos.phobos_sgemm_ex(M, N, K, 1.0, 16, K, 16, N, 0.0, 16, N, 0,
                                phobos.PHOBOS_MATH_3XTF32, p)
    assert st == phobos.PHOBOS_ERR_UNSUPPORTED
    monkeypatch.setenv(var, "1")
    if var == "WORLD_SIZE":
        monkeypatch.delenv("LOCAL_WORLD_SIZE", raising=False)
    else:
        monkeypatch.delenv("WORLD_SIZE", raising=False)
    st = phobos.phobos_sgemm_ex(M, N, K, 1.0, 16, K, 16, N, 0.0, 16, N, 0,
                                phobos.PHOBOS_MATH_3XTF32, p)
    assert st != phobos.PHOBOS_ERR_UNSUPPORTED


def test_automatic_plans_never_choose_multicast(lib):
    for shape in [(256, 256, 256), (4096, 4096, 4096), (8192, 8192, 8192),
                  (3001, 5003, 1999), (65536, 256, 4096), (16384, 16384, 16384)]:
        M, N, K = shape
        for math in ("default", "3xtf32", "tf32", "fp16", "bf16", "ffma"):
            p = phobos.phobos_gemm_plan(M, N, K, K, N, N, math)
            assert p.multicast == 0 and p.cluster_n == 1


def test_noalloc_refuses_dimensions_beyond_the_kernels_int_range(lib):
    # Even with nothing to multiply (alpha = 0, then C = beta * C), M and N
    # beyond 2^31 - 1024 are refused before any size is narrowed or any
    # device call is made; C may then be any pointer.
    big = 1 << 31
    assert phobos.phobos_sgemm_noalloc(big, 4, 4, 0.0, 16, 4, 16, 4, 0.5, 16, 4, 0) == \
        phobos.PHOBOS_ERR_UNSUPPORTED
    assert phobos.phobos_sgemm_noalloc(4, big, 4, 0.0, 16, 4, 16, big, 0.5, 16, big, 0) == \
        phobos.PHOBOS_ERR_UNSUPPORTED
    assert phobos.phobos_sgemm_noalloc(4, 4, big, 1.0, 16, big, 16, 4, 0.5, 16, 4, 0) == \
        phobos.PHOBOS_ERR_UNSUPPORTED


def test_missing_library_raises_instead_of_falling_back():
    # No CPU fallback: without the built library every entry point raises.
    code = ("import language_fp32_gemm_gb300 as p\n"
            "p.LIBRARY_PATH = '/nonexistent/libphobos_gemm.so'\n"
            "try:\n"
            "    p.phobos_sgemm(4, 4, 4, 1.0, 16, 4, 16, 4, 0.0, 16, 4, 0)\n"
            "except ImportError as e:\n"
            "    print('raised:', e)\n")
    out = subprocess.run(["python", "-c", code], cwd=ROOT, capture_output=True, text=True,
                         timeout=120)
    assert out.returncode == 0, out.stderr
    assert "raised: libphobos_gemm.so is not built" in out.stdout


def test_binding_checks_tensors_before_any_call():
    torch = pytest.importorskip("torch")
    a = torch.zeros(4, 4)
    with pytest.raises(TypeError):  # host tensors: the library takes device memory only
        phobos.sgemm(a, a, a.clone())
    # leading dimensions of row-major views; anything else is refused
    big = torch.zeros(6, 10)
    assert phobos._ld(big[:, :7], "A") == 10
    assert phobos._ld(torch.zeros(1, 5), "A") == 5
    with pytest.raises(ValueError):
        phobos._ld(big.t(), "A")                      # column-major view
    with pytest.raises(ValueError):
        phobos._ld(torch.zeros(3), "A")               # not 2-D
    with pytest.raises(ValueError):
        phobos._ld(torch.zeros(16).as_strided((4, 4), (2, 1)), "A")  # overlapping rows
