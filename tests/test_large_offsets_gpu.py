"""Matrices of more than 2^31 elements, on the GPU through the C ABI.

The library accepts M, N and K up to 2^31 - 1024 with 64-bit leading
dimensions, so an element offset (row * ld + column) can pass 2^31; 32-bit
index arithmetic anywhere on the path (kernels, split pre-pass, in-kernel
split, tensor maps, workspace layout) would wrap there.  Each case makes one
matrix larger than 2^31 elements (8 GiB):

* C: 65 600 x 33 000 with K = 64, at ldc = 33 000 (16-byte rows) and at
  ldc = 33 001 (the 4-byte epilogue, with NaN in the padding column, which
  must stay untouched).  Checked on whole rows at both ends and around the
  row where the offset passes 2^31, on seeded rows, and on the first and last
  columns.
* A: 2 200 003 x 1001 with N = 40.  At lda = 1004 (NaN padding), TMA reads
  the caller's A and the kernel splits it in shared memory; at lda = 1001 the
  pre-pass splits it.  Every output is checked.
* B: 1 100 003 x 2001, with M = 40 (one CTA per tile, split pre-pass: every
  output checked) and M = 512 (CTA pairs splitting A and B inside the kernel:
  whole rows checked at both ends of both pair rows).  The split workspace
  also holds more than 2^31 elements here.

The large matrix is drawn and copied block by block (`integer_rows`), so the
host holds one block at a time.  A case is skipped when the device or the
host lacks room for it.

Entries are small integers, and every sum stays below 2^23 in magnitude, so
every path computes each output exactly in fp32; results are compared bit for
bit with the oracle.  In the B case the oracle runs once per block of K rows,
and the test adds the blocks' results: with integer entries each block's
result is an exact integer, so their fp64 sum is exactly the oracle's result
over all of K.
"""
import math

import numpy as np
import pytest

import language_fp32_gemm_gb300 as phobos
import oracle
import seeded_inputs as si

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

GIB = 1 << 30
BLOCK_BYTES = 512 << 20  # host block of the large matrix
LIMIT = 2 ** 31          # the element offset each case passes
C_SHAPE = (65600, 33000, 64)     # M, N, K
A_SHAPE = (2200003, 40, 1001)
B_SHAPE = (1100003, 2001)        # K, N; M is 40 and 512


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from language_fp32_gemm_gb300 import build as lib_build
    lib_build.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    yield d
    phobos.phobos_release()
    torch.cuda.empty_cache()


def host_available():
    avail = None
    with open("/proc/meminfo") as f:
        for line in f:
            if line.startswith("MemAvailable:"):
                avail = int(line.split()[1]) * 1024
    try:
        with open("/sys/fs/cgroup/memory.max") as f:
            limit = f.read().strip()
        with open("/sys/fs/cgroup/memory.current") as f:
            current = int(f.read())
        if limit != "max":
            avail = min(avail, int(limit) - current)
    except OSError:
        pass
    return avail


def need_room(device_bytes, host_bytes=6 * GIB):
    phobos.phobos_release()
    torch.cuda.empty_cache()
    free, _ = torch.cuda.mem_get_info()
    if free < device_bytes + 4 * GIB:
        pytest.skip("needs %.1f GiB free on the device" % (device_bytes / GIB))
    host = host_available()
    if host is not None and host < host_bytes:
        pytest.skip("needs %.1f GiB of host memory" % (host_bytes / GIB))


def device_matrix(dev, rows, cols, ld, fill=float("nan")):
    """A rows x cols view with leading dimension ld; padding holds ``fill``."""
    backing = torch.full(((rows - 1) * ld + cols,), fill, dtype=torch.float32, device=dev)
    return torch.as_strided(backing, (rows, cols), (ld, 1)), backing


def upload(view, seed, stream, lo, hi, visit=None):
    """Draw the integer matrix (seed, stream) of view's shape block by block into view."""
    rows, cols = view.shape
    step = max(1, BLOCK_BYTES // (4 * cols))
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        blk = si.integer_rows(seed, stream, (rows, cols), r0, r1, lo, hi)
        view[r0:r1].copy_(torch.from_numpy(blk))
        if visit is not None:
            visit(r0, r1, blk)
    torch.cuda.synchronize()


def run(dA, dB, dC, alpha, beta):
    phobos.sgemm(dA, dB, dC, alpha, beta)
    torch.cuda.synchronize()
    st = phobos.phobos_check_device(0)
    assert st == phobos.PHOBOS_OK, phobos.status_string(st)


def exact(ref64):
    out = ref64.astype(np.float32)
    assert np.array_equal(out.astype(np.float64), ref64)  # the bound above holds
    return out


def assert_bits(got, want):
    bad = np.argwhere(got.view(np.uint32) != want.view(np.uint32))
    assert bad.size == 0, "%d outputs differ, first at %s: %r vs %r" % (
        len(bad), tuple(bad[0]), got[tuple(bad[0])], want[tuple(bad[0])])


@pytest.mark.parametrize("pad", [0, 1], ids=["aligned_rows", "unaligned_rows"])
def test_result_beyond_2_31_elements(dev, pad):
    (M, N, K), seed = C_SHAPE, 301
    ldc = N + pad
    alpha, beta = 1.5, 0.5
    need_room(M * ldc * 4)
    A = si.integers(seed, 0, (M, K))
    B = si.integers(seed, 1, (K, N))
    dC, backing = device_matrix(dev, M, N, ldc)
    cross = math.ceil(LIMIT / ldc)  # first row whose offset passes 2^31
    assert (cross - 1) * ldc < LIMIT <= cross * ldc and cross < M
    rows = sorted(set([0, 1, cross - 1, cross, cross + 1, M - 257, M - 256, M - 2, M - 1] +
                      si.sample_indices(seed, 9, M, N, 24, edges=False)[0].tolist()))
    cols = [0, 1, N - 2, N - 1]
    c0_rows, c0_cols = {}, np.empty((M, len(cols)), dtype=np.float32)

    def keep(r0, r1, blk):
        c0_cols[r0:r1] = blk[:, cols]
        for r in rows:
            if r0 <= r < r1:
                c0_rows[r] = blk[r - r0].copy()

    upload(dC, seed, 2, -4, 4, keep)
    run(torch.from_numpy(A).to(dev), torch.from_numpy(B).to(dev), dC, alpha, beta)

    ri = torch.tensor(rows, device=dev)
    got_rows = dC.index_select(0, ri).cpu().numpy()
    got_cols = dC.index_select(1, torch.tensor(cols, device=dev)).cpu().numpy()
    C0r = np.stack([c0_rows[r] for r in rows])
    ref_rows, _ = oracle.sgemm(A[rows], B, C0r, alpha, beta, want_den=False)
    ref_cols, _ = oracle.sgemm(A, np.ascontiguousarray(B[:, cols]), c0_cols, alpha, beta,
                               want_den=False)
    assert_bits(got_rows, exact(ref_rows))
    assert_bits(got_cols, exact(ref_cols))
    if ldc > N:  # the padding after every row but the last is untouched
        gap = torch.as_strided(backing, (M - 1, ldc - N), (ldc, 1), N)
        assert bool(torch.isnan(gap).all())
    del dC, backing
    phobos.phobos_release()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("pad", [3, 0], ids=["tma_rows", "prepass_rows"])
def test_a_beyond_2_31_elements(dev, pad):
    (M, N, K), seed = A_SHAPE, 302
    lda = K + pad
    alpha, beta = 1.0, 0.5
    need_room(M * lda * 4 + 20 * GIB)
    B = si.integers(seed, 1, (K, N))
    C0 = si.integers(seed, 2, (M, N))
    dA, _backing = device_matrix(dev, M, K, lda)
    assert (M - 1) * lda + K > LIMIT
    ref = np.empty((M, N), dtype=np.float64)

    def check(r0, r1, blk):
        ref[r0:r1], _ = oracle.sgemm(blk, B, C0[r0:r1], alpha, beta, want_den=False)

    upload(dA, seed, 0, -4, 4, check)
    dC = torch.from_numpy(C0).to(dev)
    run(dA, torch.from_numpy(B).to(dev), dC, alpha, beta)
    assert_bits(dC.cpu().numpy(), exact(ref))
    del dA, _backing, dC
    phobos.phobos_release()
    torch.cuda.empty_cache()


def test_b_beyond_2_31_elements(dev):
    (K, N), seed = B_SHAPE, 303
    alpha, beta = 1.0, 0.5
    need_room(K * N * 4 + 24 * GIB)
    assert K * N > LIMIT
    # M = 40: all of C; M = 512: whole rows at both ends of both 256-row pair tiles
    cases = {40: list(range(40)), 512: [0, 1, 127, 128, 255, 256, 257, 383, 384, 510, 511]}
    A = {m: si.integers(seed, 10 + m, (m, K), -2, 2) for m in cases}
    C0 = {m: si.integers(seed, 20 + m, (m, N), -2, 2) for m in cases}
    P = {m: None for m in cases}
    dB = torch.empty((K, N), dtype=torch.float32, device=dev)

    def check(r0, r1, blk):
        for m, rows in cases.items():
            a = np.ascontiguousarray(A[m][rows, r0:r1])
            if P[m] is None:
                P[m], _ = oracle.sgemm(a, blk, C0[m][rows], alpha, beta, want_den=False)
            else:
                part, _ = oracle.sgemm(a, blk, None, alpha, 0.0, want_den=False)
                P[m] += part

    upload(dB, seed, 1, -2, 2, check)
    for m, rows in cases.items():
        dC = torch.from_numpy(C0[m]).to(dev)
        run(torch.from_numpy(A[m]).to(dev), dB, dC, alpha, beta)
        assert_bits(dC.cpu().numpy()[rows], exact(P[m]))
        del dC
    del dB
    phobos.phobos_release()
    torch.cuda.empty_cache()
