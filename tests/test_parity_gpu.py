"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Bars (on the oracle's error scale den = |alpha| sum|a||b| + |beta||c_old|):
max |C - C_ref| / den <= 2^-20 for 3xTF32, FFMA and the K-chunked mode and
<= 2^-10 for single-pass TF32; bit-exact (C == float32(C_ref)) for integer
inputs and for the B = 0 closed form, in every mode.
"""
import numpy as np
import pytest

import language_fp32_gemm_gb300 as phobos
import oracle
import seeded_inputs as si
from gpu_util import padded, run_gemm, tolerance

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

MATHS = ["default", "3xtf32", "tf32", "ffma"]


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from language_fp32_gemm_gb300 import build as lib_build
    lib_build.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def check(dev, A, B, C0, alpha, beta, math, plan=None, offsets=(0, 0, 0)):
    C = run_gemm(torch, dev, A, B, C0, alpha, beta, math, plan=plan, offsets=offsets)
    ref, den = oracle.sgemm(A, B, C0, alpha, beta)
    err = oracle.max_rel_error(C, ref, den)
    assert err <= tolerance(math), "%s: max rel error %.3g" % (math, err)
    return C, ref, err


# ------------------------------------------------------------- config 1: 256^3

@pytest.mark.parametrize("math", MATHS)
def test_uniform_256(dev, math):
    w = si.workload("sgemm_256")
    check(dev, w.A(), w.B(), w.C_old(), w.alpha, w.beta, math)


@pytest.mark.parametrize("math", MATHS)
def test_integer_256_bit_exact(dev, math):
    w = si.workload("sgemm_256_int")
    A, B, C0 = w.A(), w.B(), w.C_old()
    C = run_gemm(torch, dev, A, B, C0, w.alpha, w.beta, math)
    ref, _ = oracle.sgemm(A, B, C0, w.alpha, w.beta)
    assert np.array_equal(C, oracle.ref32(ref))


# ------------------------------------------------------- edges and degenerates

EDGE_SHAPES = [(1, 1, 1), (1, 300, 17), (300, 1, 17), (7, 13, 5), (129, 257, 33),
               (128, 256, 32), (255, 129, 95), (300, 260, 200), (513, 384, 1000),
               (16, 520, 64), (130, 17, 260)]


@pytest.mark.parametrize("math", ["3xtf32", "tf32", "ffma"])
@pytest.mark.parametrize("shape", EDGE_SHAPES, ids=lambda s: "%dx%dx%d" % s)
def test_edge_shapes(dev, shape, math):
    M, N, K = shape
    seed = 1000 + M * 7 + N * 3 + K
    A = si.normal(seed, 0, (M, K))
    B = si.normal(seed, 1, (K, N))
    C0 = si.uniform_pm1(seed, 2, (M, N))
    check(dev, A, B, C0, 1.25, -0.5, math)


@pytest.mark.parametrize("math", ["3xtf32", "tf32", "ffma"])
def test_padded_leading_dimensions(dev, math):
    M, N, K = 200, 150, 90
    A = padded(si.normal(31, 0, (M, K)), 3)
    B = padded(si.normal(31, 1, (K, N)), 5)
    C0 = padded(si.uniform_pm1(31, 2, (M, N)), 1)
    check(dev, A, B, C0, 0.5, 2.0, math)


@pytest.mark.parametrize("math", ["3xtf32", "tf32", "ffma"])
def test_unaligned_pointers(dev, math):
    M, N, K = 190, 170, 120
    A = si.normal(32, 0, (M, K))
    B = si.normal(32, 1, (K, N))
    C0 = si.uniform_pm1(32, 2, (M, N))
    check(dev, A, B, C0, 1.0, 0.5, math, offsets=(1, 3, 1))


@pytest.mark.parametrize("pad", [1, 2, 3])
@pytest.mark.parametrize("c_offset", [0, 1, 2, 3])
@pytest.mark.parametrize("beta", [0.0, 0.5])
def test_misaligned_c_rows_bit_exact(dev, pad, c_offset, beta):
    # ldc = N + pad is not a multiple of 4, so consecutive rows of C start at
    # different offsets inside their 16-byte chunks (and the offset pointer
    # shifts them all): the tensor-core epilogue then moves each row through
    # its own aligned window of 16-byte chunks, with element-wise edges.
    # Integer inputs make every result exact, so any misplaced, dropped or
    # duplicated element fails; beta = 0 must not read C (NaN there).
    M, N, K = 300, 600, 64
    A = si.integers(40 + pad, 0, (M, K))
    B = si.integers(40 + pad, 1, (K, N))
    C0 = si.integers(40 + pad, 2, (M, N)) if beta else np.full((M, N), np.nan, np.float32)
    C0p = padded(C0, pad)
    C = run_gemm(torch, dev, A, B, C0p, 1.5, beta, "3xtf32", offsets=(0, 0, c_offset))
    ref, _ = oracle.sgemm(A, B, C0 if beta else None, 1.5, beta)
    assert np.array_equal(C, oracle.ref32(ref))


@pytest.mark.parametrize("math", MATHS)
def test_closed_form_zero_b_bit_exact(dev, math):
    M, N, K = 300, 270, 130
    A = si.normal(33, 0, (M, K))
    B = np.zeros((K, N), dtype=np.float32)
    C0 = si.uniform_pm1(33, 2, (M, N))
    C = run_gemm(torch, dev, A, B, C0, 1.5, -0.75, math)
    assert np.array_equal(C, np.float32(-0.75) * C0)


@pytest.mark.parametrize("math", MATHS)
def test_closed_form_identity(dev, math):
    M, N = 300, 260
    A = np.eye(M, dtype=np.float32)
    B = si.uniform_pm1(34, 1, (M, N))
    C0 = si.uniform_pm1(34, 2, (M, N))
    C, ref, _ = check(dev, A, B, C0, 0.75, 0.25, math)
    # A = I: C = alpha*B + beta*C0
    assert np.allclose(C, 0.75 * B.astype(np.float64) + 0.25 * C0, rtol=0,
                       atol=4 * tolerance(math))


@pytest.mark.parametrize("math", MATHS)
def test_beta_zero_ignores_nan(dev, math):
    M, N, K = 160, 140, 70
    A = si.normal(35, 0, (M, K))
    B = si.normal(35, 1, (K, N))
    C0 = np.full((M, N), np.nan, dtype=np.float32)
    C = run_gemm(torch, dev, A, B, C0, 1.0, 0.0, math)
    assert np.isfinite(C).all()
    ref, den = oracle.sgemm(A, B, None, 1.0, 0.0)
    assert oracle.max_rel_error(C, ref, den) <= tolerance(math)


@pytest.mark.parametrize("math", MATHS)
def test_alpha_zero_and_k_zero(dev, math):
    M, N = 100, 90
    C0 = si.uniform_pm1(36, 2, (M, N))
    A = si.normal(36, 0, (M, 40))
    B = si.normal(36, 1, (40, N))
    C = run_gemm(torch, dev, A, B, C0, 0.0, 0.5, math)
    assert np.array_equal(C, np.float32(0.5) * C0)
    C = run_gemm(torch, dev, np.zeros((M, 0), np.float32), np.zeros((0, N), np.float32), C0,
                 2.0, 0.5, math)
    assert np.array_equal(C, np.float32(0.5) * C0)


def test_empty_output_is_untouched(dev):
    for M, N in ((0, 10), (10, 0)):
        st = phobos.phobos_sgemm(M, N, 5, 1.0, 16, 5, 16, max(N, 1), 0.0, 16, max(N, 1), 0)
        assert st == phobos.PHOBOS_OK


# --------------------------------------------------------- K-chunked super-tiles

@pytest.mark.parametrize("math,super_k", [("3xtf32", 512), ("3xtf32", 96), ("tf32", 1024),
                                          ("ffma", 520)])
def test_k_chunked_cluster_split(dev, math, super_k):
    M, N, K = 520, 390, 2100
    plan = phobos.phobos_gemm_plan(M, N, K, K, N, N, math)
    plan.super_k = super_k
    A = si.uniform_pm1(37, 0, (M, K))
    B = si.uniform_pm1(37, 1, (K, N))
    C0 = si.normal(37, 2, (M, N))
    check(dev, A, B, C0, 0.75, 0.25, math, plan=plan)


def test_plan_validation_on_device(dev):
    plan = phobos.phobos_gemm_plan(256, 256, 256, 256, 256, 256, "3xtf32")
    plan.super_k = 33  # not a multiple of the K block
    A = torch.zeros(256, 256, device=dev)
    with pytest.raises(phobos.PhobosError):
        phobos.sgemm(A, A, A.clone(), 1.0, 0.0, math="3xtf32", plan=plan)
    plan = phobos.phobos_gemm_plan(256, 256, 256, 256, 256, 256, "3xtf32")
    with pytest.raises(phobos.PhobosError):
        phobos.sgemm(A, A, A.clone(), 1.0, 0.0, math="ffma", plan=plan)


def test_host_buffer_entry_point(dev):
    M, N, K = 333, 222, 111
    A = si.normal(38, 0, (M, K))
    B = si.normal(38, 1, (K, N))
    C0 = si.uniform_pm1(38, 2, (M, N))
    C = C0.copy()
    st = phobos.phobos_sgemm_host(M, N, K, 1.5, A.ctypes.data, K, B.ctypes.data, N, 0.5,
                                  C.ctypes.data, N, 0, phobos.PHOBOS_MATH_3XTF32)
    assert st == phobos.PHOBOS_OK
    ref, den = oracle.sgemm(A, B, C0, 1.5, 0.5)
    assert oracle.max_rel_error(C, ref, den) <= oracle.TOL_FP32


def test_timing_events_and_launch_count(dev):
    M = N = K = 512
    A = torch.randn(M, K, device=dev)
    B = torch.randn(K, N, device=dev)
    C = torch.zeros(M, N, device=dev)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()  # torch creates the CUDA events lazily, on first record
    stop.record()
    # one pre-pass launch (split A and/or B, zero the tail flags), then the
    # main kernel; with the in-kernel panel split the main kernel alone
    for a_split, launches in ((1, 2), (2, 2), (3, 1)):
        plan = phobos.phobos_gemm_plan(M, N, K, K, N, N, "3xtf32")
        plan.a_split = a_split
        n0 = phobos.phobos_kernel_launches()
        phobos.phobos_set_timing_events(start.cuda_event, stop.cuda_event)
        try:
            phobos.sgemm(A, B, C, 1.0, 0.0, math="3xtf32", plan=plan)
        finally:
            phobos.phobos_set_timing_events(None, None)
        torch.cuda.synchronize()
        assert phobos.phobos_kernel_launches() - n0 == launches
        assert start.elapsed_time(stop) > 0


# ------------------------------------------------------- tail split along K

@pytest.mark.parametrize("math", ["3xtf32", "tf32"])
@pytest.mark.parametrize("shape,split,super_k", [
    ((512, 512, 2048), 0, None),     # 4 pair tiles: automatic split over idle SMs
    ((512, 512, 2048), 1, None),     # split switched off
    ((512, 512, 2048), 3, None),     # forced, uneven K pieces
    ((1000, 100, 1024), 0, None),    # single-CTA tiles (N <= 128)
    ((520, 390, 2100), 0, 512),      # split inside every K chunk of the cluster split
    ((777, 1290, 333), 0, None),     # ragged edges, short K: pieces of at least 4 blocks
    # 100 pair tiles: 24 tail tiles; 8 pieces each would need 192 pairs, so the
    # tail's K blocks are dealt evenly to all of them (shares across tiles)
    ((2560, 2560, 2048), 8, None),
    ((2500, 2510, 1100), 8, 512),    # the same inside K chunks, ragged edges
], ids=lambda v: str(v))
def test_tail_split(dev, math, shape, split, super_k):
    M, N, K = shape
    plan = phobos.phobos_gemm_plan(M, N, K, K, N, N, math)
    plan.tail_split = split
    if super_k is not None:
        plan.super_k = super_k
    A = si.normal(81, 0, (M, K))
    B = si.normal(81, 1, (K, N))
    C0 = si.uniform_pm1(81, 2, (M, N))
    C1, _, _ = check(dev, A, B, C0, 0.5, 1.5, math, plan=plan)
    # deterministic: the same call again gives the same bits
    C2 = run_gemm(torch, dev, A, B, C0, 0.5, 1.5, math, plan=plan)
    assert np.array_equal(C1, C2)


def test_tail_split_rejects_bad_values(dev):
    plan = phobos.phobos_gemm_plan(512, 512, 512, 512, 512, 512, "3xtf32")
    plan.tail_split = 9
    A = torch.zeros(512, 512, device=dev)
    with pytest.raises(phobos.PhobosError):
        phobos.sgemm(A, A, A.clone(), 1.0, 0.0, math="3xtf32", plan=plan)


# ---------------------------------------------- A split inside the kernel

@pytest.mark.parametrize("math", ["3xtf32", "tf32"])
@pytest.mark.parametrize("shape", [(300, 260, 200), (1000, 700, 332), (4096, 256, 1000),
                                   (129, 100, 36), (640, 1024, 4), (333, 257, 68), (77, 900, 4)],
                         ids=lambda s: "%dx%dx%d" % s)
def test_a_split_in_kernel_matches_prepass(dev, math, shape):
    M, N, K = shape
    A = si.normal(91, 0, (M, K))
    B = si.normal(91, 1, (K, N))
    C0 = si.uniform_pm1(91, 2, (M, N))
    out = {}
    for mode in (1, 2):
        plan = phobos.phobos_gemm_plan(M, N, K, K, N, N, math)
        plan.a_split = mode
        out[mode], _, _ = check(dev, A, B, C0, 1.25, 0.75, math, plan=plan)
    # the same tf32 rounding of A either way: identical bits
    assert np.array_equal(out[1], out[2])


def test_a_split_in_kernel_needs_aligned_rows(dev):
    M, N, K = 64, 64, 33  # lda = 33 is not a multiple of 4
    plan = phobos.phobos_gemm_plan(M, N, K, K, N, N, "3xtf32")
    plan.a_split = 2
    A = torch.zeros(M, K, device=dev)
    B = torch.zeros(K, N, device=dev)
    with pytest.raises(phobos.PhobosError) as e:
        phobos.sgemm(A, B, torch.zeros(M, N, device=dev), 1.0, 0.0, math="3xtf32", plan=plan)
    assert e.value.status == phobos.PHOBOS_ERR_UNSUPPORTED


# --------------------------------------- FFMA split-K over a cluster (DSMEM)

@pytest.mark.parametrize("shape,split", [((256, 256, 256), 0), ((256, 256, 256), 1),
                                         ((100, 70, 1000), 0), ((64, 64, 8), 0),
                                         ((130, 129, 300), 3), ((200, 300, 77), 8)],
                         ids=lambda v: str(v))
def test_ffma_cluster_split_k(dev, shape, split):
    M, N, K = shape
    plan = phobos.phobos_gemm_plan(M, N, K, K, N, N, "ffma")
    assert plan.tile_m == 64
    plan.tail_split = split
    A = si.normal(95, 0, (M, K))
    B = si.normal(95, 1, (K, N))
    C0 = si.uniform_pm1(95, 2, (M, N))
    C1, _, _ = check(dev, A, B, C0, 0.5, -1.5, "ffma", plan=plan)
    C2 = run_gemm(torch, dev, A, B, C0, 0.5, -1.5, "ffma", plan=plan)
    assert np.array_equal(C1, C2)  # deterministic


# 128 x 128 FFMA tiles: interior K tiles load without bounds checks; the
# last partial K tile, ragged edge tiles, unaligned bases and leading
# dimensions that are not multiples of 4 take the checked loads.
@pytest.mark.parametrize("shape,pads,offsets,super_k", [
    ((384, 384, 200), (0, 0, 0), (0, 0, 0), None),   # all tiles interior, K tail of 8
    ((300, 260, 203), (0, 0, 0), (0, 0, 0), None),   # ragged M, N and K
    ((384, 256, 256), (1, 0, 0), (0, 0, 0), None),   # lda = K + 1: A on the checked loads
    ((384, 256, 256), (0, 0, 0), (0, 1, 0), None),   # B base not 16-byte aligned
    ((256, 384, 1000), (0, 0, 0), (0, 0, 0), 520),   # K chunks starting at 8 mod 16
], ids=lambda v: str(v))
def test_ffma_128_interior_and_edges(dev, shape, pads, offsets, super_k):
    M, N, K = shape
    plan = phobos.phobos_gemm_plan(M, N, K, K + pads[0], N + pads[1], N + pads[2], "ffma")
    plan.tile_m, plan.tile_n = 128, 128
    if super_k is not None:
        plan.super_k = super_k
    A = padded(si.normal(96, 0, (M, K)), pads[0])
    B = padded(si.normal(96, 1, (K, N)), pads[1])
    C0 = padded(si.uniform_pm1(96, 2, (M, N)), pads[2])
    check(dev, A, B, C0, 1.25, 0.5, "ffma", plan=plan, offsets=offsets)


@pytest.mark.parametrize("beta", [0.0, 0.5])
def test_host_buffer_entry_point_in_bands(dev, beta):
    # M >= 2048 on the tensor-core path: row bands with overlapped copies;
    # padded leading dimensions on every operand
    M, N, K = 4100, 300, 200
    A = padded(si.normal(96, 0, (M, K)), 3)
    B = padded(si.normal(96, 1, (K, N)), 1)
    C0 = si.uniform_pm1(96, 2, (M, N))
    C = padded(C0, 2)  # a copy of C0 inside a wider buffer (ldc = N + 2)
    lda, ldb, ldc = A.strides[0] // 4, B.strides[0] // 4, C.strides[0] // 4
    st = phobos.phobos_sgemm_host(M, N, K, 1.5, A.ctypes.data, lda, B.ctypes.data, ldb, beta,
                                  C.ctypes.data, ldc, 0, phobos.PHOBOS_MATH_3XTF32)
    assert st == phobos.PHOBOS_OK
    ref, den = oracle.sgemm(A, B, C0, 1.5, beta)
    assert oracle.max_rel_error(C, ref, den) <= oracle.TOL_FP32


# ----------------------------- split-TF32 accuracy where it is tightest

@pytest.mark.parametrize("K", [32, 64, 128, 256, 512, 1025, 1100, 2000, 2048])
def test_split_tf32_short_k_stress(dev, K):
    # The tensor core truncates while it accumulates a TMEM partial sum; the
    # error relative to sum|a||b| is largest when K spans few partials.  Two
    # million normal-distributed outputs per K, all checked against the oracle.
    M, N = 1024, 2048
    A = si.normal(97, 0, (M, K))
    B = si.normal(97, 1, (K, N))
    check(dev, A, B, np.zeros((M, N), np.float32), 1.0, 0.0, "3xtf32")


# ------------------------------- inputs of one sign: the bound's other side

def promote_blocks(K):
    """K blocks (of 32) per TMEM partial sum of split TF32 for this K."""
    return 1 if K <= 128 else 2 if K <= 512 else 4 if K <= 1024 else 8


@pytest.mark.parametrize("K", [256, 1024, 4096])
@pytest.mark.parametrize("math", ["3xtf32", "ffma"])
def test_same_sign_inputs_within_their_accumulation_bound(dev, math, K):
    # The 2^-20 bound holds for zero-mean data, as in every workload.  When all
    # products share a sign, the running sum grows like sum|a||b| and every
    # fp32 addition rounds relative to it, so no fp32 accumulation meets 2^-20
    # at large K.  Each path must still stay inside the error of its own
    # arithmetic:
    #  - FFMA: K additions, each rounded to nearest (2^-24 of the running sum);
    #  - split TF32: the tensor core truncates each of the U = 3 passes x 4
    #    MMAs x (blocks per partial) updates of a TMEM partial sum towards
    #    zero.  Measured on GB300 over K = 128 .. 8192, the loss averages
    #    0.15 - 0.19 U 2^-23 of the partial's sum|a||b| and its largest value
    #    over these 0.5 M outputs stays below U 2^-23 / 4; 2^-21 covers the
    #    split's dropped a_small*b_small and rounded small parts and the
    #    rounded register additions.  The measured worst cases (8.1e-7,
    #    1.4e-6, 2.5e-6 at K = 256, 1024, 4096) sit 1.3 - 1.5x below the
    #    bound, and a build with partials twice as long (1.7e-6, 3.0e-6,
    #    5.0e-6), a missing promotion (8.6e-5 at K = 8192) or a dropped split
    #    pass (about 2^-11) exceeds it.
    M, N = 512, 1024
    A = np.abs(si.uniform_pm1(98, 0, (M, K)))
    B = np.abs(si.uniform_pm1(98, 1, (K, N)))
    C0 = np.zeros((M, N), np.float32)
    C = run_gemm(torch, dev, A, B, C0, 1.0, 0.0, math)
    ref, den = oracle.sgemm(A, B, C0, 1.0, 0.0)
    err = oracle.max_rel_error(C, ref, den)
    if math == "ffma":
        bound = K * 2.0 ** -24
    else:
        U = 3 * 4 * promote_blocks(K)
        bound = U * 2.0 ** -23 / 4 + 2.0 ** -21
    assert err <= bound, "max rel error %.3g > %.3g" % (err, bound)


def test_kernels_count_their_sm_clock_only_while_timed(dev):
    # phobos_kernel_clock_mhz: the tensor-core kernels add their SM cycles and
    # global-timer nanoseconds to a device sum while timing events are set.
    M = N = K = 2048
    dA = torch.from_numpy(si.normal(97, 0, (M, K))).to(dev)
    dB = torch.from_numpy(si.normal(97, 1, (K, N))).to(dev)
    dC = torch.zeros((M, N), dtype=torch.float32, device=dev)
    phobos.phobos_kernel_clock_mhz()  # clear
    phobos.sgemm(dA, dB, dC, 1.0, 0.0)
    assert phobos.phobos_kernel_clock_mhz() == 0.0  # not timed: nothing counted
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()  # torch creates the CUDA events on their first record
    stop.record()
    torch.cuda.synchronize()
    assert start.cuda_event and stop.cuda_event
    phobos.phobos_set_timing_events(start.cuda_event, stop.cuda_event)
    try:
        for _ in range(3):
            phobos.sgemm(dA, dB, dC, 1.0, 0.0)
    finally:
        phobos.phobos_set_timing_events(None, None)
    mhz = phobos.phobos_kernel_clock_mhz()
    assert 300.0 < mhz < 2500.0, mhz
    assert phobos.phobos_kernel_clock_mhz() == 0.0  # the read cleared the sum
    assert start.elapsed_time(stop) > 0.0
    assert phobos.phobos_check_device(0) == phobos.PHOBOS_OK
