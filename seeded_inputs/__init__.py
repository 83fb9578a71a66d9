"""Seeded synthetic inputs for the fp32 GEMM workloads.

This module serves both the CUDA path's tests/benchmark and the oracle; it
holds none of the GEMM's arithmetic, only random numbers.

Generator: SplitMix64 (G. L. Steele, D. Lea, C. H. Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014), used counter-based: the n-th
draw (n = 0, 1, ...) of a stream is ``mix64(base + (n + 1) * GAMMA)`` with
``GAMMA = 0x9E3779B97F4A7C15`` and ``mix64`` the generator's finaliser.  A
stream's ``base`` is ``mix64(seed * 2**20 + stream)``, so every matrix of every
workload draws from its own stream and any element can be generated without
the ones before it.

Value maps (all results are float32):
  uniform[-1, 1):  2 * (x >> 40) * 2**-24 - 1      (exact in fp32)
  normal(0, sd):   Box-Muller in float64 on draws 2n, 2n+1, times sd, rounded
  integers lo..hi: (x >> 32) % (hi - lo + 1) + lo

Workloads: the five fp32 SGEMM shapes with their distributions, scalars and
seeds; matrices are stream 0 (A), 1 (B), 2 (C_old) and 3 (sampled indices),
plus 10 for the tall-skinny shape that shares seed 3 with the unaligned one.
"""
import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def mix64(z):
    """SplitMix64 finaliser on a uint64 ndarray (wrapping arithmetic)."""
    z = np.asarray(z, dtype=np.uint64)
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64_sequence(state, count):
    """The classic sequential SplitMix64 outputs for a given 64-bit state."""
    n = np.arange(1, count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return mix64(np.uint64(state) + n * GAMMA)


def stream_base(seed, stream):
    with np.errstate(over="ignore"):
        key = np.uint64(seed) * np.uint64(1 << 20) + np.uint64(stream)
    return mix64(np.array([key], dtype=np.uint64))[0]


def stream_bits(seed, stream, count, offset=0):
    """``count`` raw 64-bit draws of stream ``(seed, stream)`` from ``offset``."""
    base = stream_base(seed, stream)
    n = np.arange(offset + 1, offset + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return mix64(base + n * GAMMA)


def _threads():
    try:
        return max(1, min(16, len(os.sched_getaffinity(0))))
    except AttributeError:  # pragma: no cover
        return 4


def _fill(out, fn):
    """Fill the flat float32 array ``out`` chunk by chunk with ``fn(lo, hi)``."""
    total = out.size
    spans = [(lo, min(total, lo + _CHUNK)) for lo in range(0, total, _CHUNK)]
    if len(spans) <= 1:
        for lo, hi in spans:
            out[lo:hi] = fn(lo, hi)
        return out

    def work(span):
        lo, hi = span
        out[lo:hi] = fn(lo, hi)

    with ThreadPoolExecutor(_threads()) as pool:
        list(pool.map(work, spans))
    return out


def uniform_pm1(seed, stream, shape):
    """iid uniform on [-1, 1) with 24-bit resolution, exact in float32."""
    out = np.empty(int(np.prod(shape)), dtype=np.float32)

    def fn(lo, hi):
        x = stream_bits(seed, stream, hi - lo, lo)
        u = (x >> np.uint64(40)).astype(np.float64) * 2.0 ** -24
        return (2.0 * u - 1.0).astype(np.float32)

    return _fill(out, fn).reshape(shape)


def normal(seed, stream, shape, sd=1.0):
    """iid normal(0, sd) by Box-Muller on draws 2n and 2n+1."""
    out = np.empty(int(np.prod(shape)), dtype=np.float32)

    def fn(lo, hi):
        x = stream_bits(seed, stream, 2 * (hi - lo), 2 * lo)
        u1 = ((x[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
        u2 = (x[1::2] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
        z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)
        return (z * sd).astype(np.float32)

    return _fill(out, fn).reshape(shape)


def integers(seed, stream, shape, lo=-4, hi=4):
    """iid integers uniform on lo..hi, as float32."""
    shape = tuple(shape)
    return integer_rows(seed, stream, shape, 0, shape[0], lo, hi)


def integer_rows(seed, stream, shape, r0, r1, lo=-4, hi=4):
    """Rows r0 .. r1-1 of ``integers(seed, stream, shape, lo, hi)``.

    Draw n of the stream is element n of the row-major matrix, so a block of
    rows is drawn on its own: a matrix larger than host memory can be made and
    copied block by block.
    """
    span = hi - lo + 1
    cols = int(np.prod(shape[1:])) if len(shape) > 1 else 1
    out = np.empty((r1 - r0) * cols, dtype=np.float32)
    first = r0 * cols

    def fn(a, b):
        x = stream_bits(seed, stream, b - a, first + a)
        return ((x >> np.uint64(32)) % np.uint64(span)).astype(np.int64).astype(np.float32) + lo

    return _fill(out, fn).reshape((r1 - r0,) + tuple(shape[1:]))


def sample_indices(seed, stream, M, N, count, edges=True):
    """Seeded output positions for sampled checks.

    ``count`` uniform draws over [0, M) x [0, N); with ``edges`` the four
    corners and a stripe along the last row and last column are added, so the
    ragged edge tiles are always covered.  Returns int64 ``(rows, cols)``.
    """
    x = stream_bits(seed, stream, 2 * count)
    rows = (x[0::2] % np.uint64(max(M, 1))).astype(np.int64)
    cols = (x[1::2] % np.uint64(max(N, 1))).astype(np.int64)
    if edges and M > 0 and N > 0:
        extra_r = [0, 0, M - 1, M - 1]
        extra_c = [0, N - 1, 0, N - 1]
        for t in range(0, 32):
            extra_r += [M - 1, (t * 7919) % M]
            extra_c += [(t * 104729) % N, N - 1]
        rows = np.concatenate([rows, np.array(extra_r, dtype=np.int64)])
        cols = np.concatenate([cols, np.array(extra_c, dtype=np.int64)])
    return rows, cols


# --------------------------------------------------------------- workloads

class Workload:
    """One GEMM problem: shape, scalars and how each matrix is drawn."""

    def __init__(self, name, M, N, K, alpha, beta, seed, a, b, c, streams=(0, 1, 2, 3),
                 sample_count=0, note=""):
        self.name, self.M, self.N, self.K = name, M, N, K
        self.alpha, self.beta, self.seed = alpha, beta, seed
        self.a, self.b, self.c = a, b, c          # (kind, parameter) per matrix
        self.streams = streams
        self.sample_count = sample_count
        self.note = note

    def flops(self):
        return 2.0 * self.M * self.N * self.K

    def _draw(self, spec, stream, shape):
        kind, param = spec
        if kind == "uniform":
            return uniform_pm1(self.seed, stream, shape)
        if kind == "normal":
            return normal(self.seed, stream, shape, param)
        if kind == "int":
            return integers(self.seed, stream, shape, -param, param)
        if kind == "zeros":
            return np.zeros(shape, dtype=np.float32)
        raise ValueError(kind)

    def A(self):
        return self._draw(self.a, self.streams[0], (self.M, self.K))

    def B(self):
        return self._draw(self.b, self.streams[1], (self.K, self.N))

    def C_old(self):
        return self._draw(self.c, self.streams[2], (self.M, self.N))

    def samples(self, count=None):
        return sample_indices(self.seed, self.streams[3], self.M, self.N,
                              count if count is not None else self.sample_count)

    def with_beta(self, beta, name=None):
        w = Workload(name or self.name, self.M, self.N, self.K, self.alpha, beta, self.seed,
                     self.a, self.b, self.c, self.streams, self.sample_count, self.note)
        return w


def _sd_inv_sqrt(K):
    return 1.0 / math.sqrt(K)


WORKLOADS = {
    "sgemm_256": Workload("sgemm_256", 256, 256, 256, 1.5, 0.5, 0,
                          ("uniform", None), ("uniform", None), ("uniform", None)),
    "sgemm_256_int": Workload("sgemm_256_int", 256, 256, 256, 1.5, 0.5, 0,
                              ("int", 4), ("int", 4), ("int", 4), streams=(4, 5, 6, 7),
                              note="entries in -4..4; every result is exact in fp32"),
    "sgemm_4096_beta0": Workload("sgemm_4096_beta0", 4096, 4096, 4096, 1.0, 0.0, 1,
                                 ("normal", 1.0), ("normal", 1.0), ("uniform", None),
                                 sample_count=4096),
    "sgemm_4096_beta1": Workload("sgemm_4096_beta1", 4096, 4096, 4096, 1.0, 1.0, 1,
                                 ("normal", 1.0), ("normal", 1.0), ("uniform", None),
                                 sample_count=4096),
    "sgemm_8192": Workload("sgemm_8192", 8192, 8192, 8192, 0.75, 0.25, 2,
                           ("uniform", None), ("uniform", None), ("normal", 1.0),
                           sample_count=4096),
    "sgemm_3001x5003x1999": Workload("sgemm_3001x5003x1999", 3001, 5003, 1999, 1.0, 0.5, 3,
                                     ("normal", _sd_inv_sqrt(1999)),
                                     ("normal", _sd_inv_sqrt(1999)), ("uniform", None),
                                     sample_count=4096),
    "sgemm_65536x256x4096": Workload("sgemm_65536x256x4096", 65536, 256, 4096, 1.0, 0.5, 3,
                                     ("normal", _sd_inv_sqrt(4096)),
                                     ("normal", _sd_inv_sqrt(4096)), ("uniform", None),
                                     streams=(10, 11, 12, 13), sample_count=4096),
    "sgemm_16384": Workload("sgemm_16384", 16384, 16384, 16384, 1.0, 0.0, 4,
                            ("uniform", None), ("uniform", None), ("zeros", None),
                            sample_count=4096),
}


def workload(name):
    return WORKLOADS[name]
