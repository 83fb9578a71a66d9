"""Python binding of libphobos_gemm: fp32 GEMM C = alpha*A*B + beta*C on GB300.

Argument marshalling only.  Every step of the GEMM runs in the CUDA kernels
of ``libphobos_gemm.so`` (built in-tree by ``build.py``); importing a function
from here never computes anything on the CPU, and a missing library raises
instead of falling back.

The names mirror the C ABI in ``include/phobos_gemm.h``:

* ``phobos_sgemm``, ``phobos_sgemm_ex``, ``phobos_sgemm_host`` take raw
  pointers (Python ints), sizes and leading dimensions, and return the
  status code;
* ``phobos_gemm_plan`` returns a ``PhobosGemmPlan`` (or raises);
* ``sgemm`` is the same call for torch tensors: it reads pointers, leading
  dimensions and the current CUDA stream from the tensors and raises
  ``PhobosError`` on a non-zero status.
"""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY_PATH = os.path.join(HERE, "libphobos_gemm.so")

PHOBOS_OK = 0
PHOBOS_ERR_INVALID_VALUE = 1
PHOBOS_ERR_UNSUPPORTED = 2
PHOBOS_ERR_CUDA = 3
PHOBOS_ERR_OUT_OF_MEMORY = 4
PHOBOS_ERR_TIMEOUT = 5

PHOBOS_MATH_DEFAULT = 0
PHOBOS_MATH_3XTF32 = 1
PHOBOS_MATH_TF32 = 2
PHOBOS_MATH_FFMA = 3
PHOBOS_MATH_FP16 = 4
PHOBOS_MATH_BF16 = 5

PHOBOS_PATH_FFMA = 1
PHOBOS_PATH_TF32 = 2
PHOBOS_PATH_3XTF32 = 3
PHOBOS_PATH_FP16 = 4
PHOBOS_PATH_BF16 = 5

MATH_NAMES = {"default": PHOBOS_MATH_DEFAULT, "3xtf32": PHOBOS_MATH_3XTF32,
              "tf32": PHOBOS_MATH_TF32, "ffma": PHOBOS_MATH_FFMA,
              "fp16": PHOBOS_MATH_FP16, "bf16": PHOBOS_MATH_BF16}

ABI_FUNCTIONS = ("phobos_gemm_plan", "phobos_sgemm", "phobos_sgemm_ex", "phobos_sgemm_host",
                 "phobos_check_device", "phobos_set_timing_events", "phobos_kernel_launches",
                 "phobos_release", "phobos_status_string", "phobos_sgemm_noalloc",
                 "phobos_kernel_clock_mhz", "phobos_kernel_clc_tiles")

# Split operands the no-allocation entry point can hold (bytes).
PHOBOS_NOALLOC_SCRATCH_BYTES = 64 << 20


class PhobosGemmPlan(ctypes.Structure):
    """Mirror of ``phobos_gemm_plan_t``."""
    _fields_ = [("path", ctypes.c_int32), ("tile_m", ctypes.c_int32),
                ("tile_n", ctypes.c_int32), ("tile_k", ctypes.c_int32),
                ("cluster_m", ctypes.c_int32), ("cluster_n", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("multicast", ctypes.c_int32),
                ("super_m", ctypes.c_int64), ("super_n", ctypes.c_int64),
                ("super_k", ctypes.c_int64), ("workspace_bytes", ctypes.c_size_t),
                ("tail_split", ctypes.c_int32), ("a_split", ctypes.c_int32),
                ("clc", ctypes.c_int32)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}

    def copy(self):
        p = PhobosGemmPlan()
        ctypes.pointer(p)[0] = self
        return p


class PhobosError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        msg = status_string(status)
        super().__init__("%s%s" % (what + ": " if what else "", msg))


_lib = None


def library():
    """The loaded ``libphobos_gemm.so`` (ctypes handle); raises if it is not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIBRARY_PATH):
            raise ImportError("libphobos_gemm.so is not built; run "
                              "language_fp32_gemm_gb300.build.build() first "
                              "(there is no CPU fallback)")
        lib = ctypes.CDLL(LIBRARY_PATH)
        i64, f32, i32, vp = ctypes.c_int64, ctypes.c_float, ctypes.c_int, ctypes.c_void_p
        plan_p = ctypes.POINTER(PhobosGemmPlan)
        gemm = [i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, vp]
        lib.phobos_gemm_plan.argtypes = [i64, i64, i64, i64, i64, i64, i32, plan_p]
        lib.phobos_sgemm.argtypes = gemm
        lib.phobos_sgemm_ex.argtypes = gemm + [i32, plan_p]
        lib.phobos_sgemm_host.argtypes = gemm + [i32]
        lib.phobos_sgemm_noalloc.argtypes = gemm
        lib.phobos_check_device.argtypes = [vp]
        lib.phobos_release.argtypes = []
        lib.phobos_set_timing_events.argtypes = [vp, vp]
        lib.phobos_kernel_clock_mhz.argtypes = [ctypes.POINTER(ctypes.c_double)]
        lib.phobos_kernel_clc_tiles.argtypes = [ctypes.POINTER(ctypes.c_uint64)]
        lib.phobos_kernel_launches.argtypes = []
        lib.phobos_kernel_launches.restype = ctypes.c_uint64
        lib.phobos_status_string.argtypes = [i32]
        lib.phobos_status_string.restype = ctypes.c_char_p
        for name in ("phobos_gemm_plan", "phobos_sgemm", "phobos_sgemm_ex", "phobos_sgemm_host",
                     "phobos_check_device", "phobos_release", "phobos_set_timing_events",
                     "phobos_sgemm_noalloc", "phobos_kernel_clock_mhz",
                     "phobos_kernel_clc_tiles"):
            getattr(lib, name).restype = i32
        _lib = lib
    return _lib


def status_string(status):
    return library().phobos_status_string(int(status)).decode()


def _math(math):
    if isinstance(math, str):
        return MATH_NAMES[math.lower()]
    return int(math)


# ------------------------------------------------------------- raw C ABI

def phobos_gemm_plan(M, N, K, lda, ldb, ldc, math=PHOBOS_MATH_DEFAULT):
    plan = PhobosGemmPlan()
    st = library().phobos_gemm_plan(M, N, K, lda, ldb, ldc, _math(math), ctypes.byref(plan))
    if st != PHOBOS_OK:
        raise PhobosError(st, "phobos_gemm_plan")
    return plan


def phobos_sgemm(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0):
    return library().phobos_sgemm(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream)


def phobos_sgemm_ex(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0,
                    math=PHOBOS_MATH_DEFAULT, plan=None):
    return library().phobos_sgemm_ex(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream,
                                     _math(math), ctypes.byref(plan) if plan is not None else None)


def phobos_sgemm_host(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0,
                      math=PHOBOS_MATH_DEFAULT):
    return library().phobos_sgemm_host(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream,
                                       _math(math))


def phobos_sgemm_noalloc(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0):
    """Split-TF32 GEMM whose scratch is a fixed array inside the library: no
    device allocation, for callers that cannot allocate (see the C header)."""
    return library().phobos_sgemm_noalloc(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream)


def phobos_check_device(stream=0):
    return library().phobos_check_device(stream)


def phobos_release():
    return library().phobos_release()


def phobos_set_timing_events(start, stop):
    """``start``/``stop``: cudaEvent_t handles as ints (e.g. torch.cuda.Event().cuda_event)."""
    return library().phobos_set_timing_events(start, stop)


def phobos_kernel_launches():
    return library().phobos_kernel_launches()


def phobos_kernel_clc_tiles():
    """Tiles that Cluster Launch Control launches took from cancelled pair
    launches while timing events were set, since the last call; clears it."""
    n = ctypes.c_uint64(0)
    st = library().phobos_kernel_clc_tiles(ctypes.byref(n))
    if st != PHOBOS_OK:
        raise PhobosError(st, "phobos_kernel_clc_tiles")
    return n.value


def phobos_kernel_clock_mhz():
    """Average SM clock (MHz) of the tensor-core kernels launched while timing
    events were set, since the last call (0.0 if none); clears the sum."""
    mhz = ctypes.c_double(0.0)
    st = library().phobos_kernel_clock_mhz(ctypes.byref(mhz))
    if st != PHOBOS_OK:
        raise PhobosError(st, "phobos_kernel_clock_mhz")
    return mhz.value


# ----------------------------------------------------------- torch tensors

def _ld(t, name):
    """Leading dimension (elements) of a row-major 2-D tensor view."""
    if t.dim() != 2:
        raise ValueError("%s must be 2-D" % name)
    rows, cols = t.shape
    if cols > 1 and t.stride(1) != 1:
        raise ValueError("%s must have unit inner stride (row-major)" % name)
    if rows > 1:
        if t.stride(0) < max(cols, 1):
            raise ValueError("%s has overlapping rows" % name)
        return t.stride(0)
    return max(cols, 1)


def _stream(t, stream):
    if stream is not None:
        return int(getattr(stream, "cuda_stream", stream))
    import torch
    return torch.cuda.current_stream(t.device).cuda_stream


def sgemm(A, B, C, alpha=1.0, beta=0.0, math=PHOBOS_MATH_DEFAULT, plan=None, stream=None):
    """C = alpha*A@B + beta*C in place for float32 CUDA tensors (row-major views).

    Enqueued on ``stream`` (default: torch's current stream for C's device).
    Returns C.  Raises ``PhobosError`` on a non-zero status.
    """
    import torch
    for t, n in ((A, "A"), (B, "B"), (C, "C")):
        if t.dtype != torch.float32 or not t.is_cuda:
            raise TypeError("%s must be a float32 CUDA tensor" % n)
    M, K = A.shape
    K2, N = B.shape
    if K2 != K or tuple(C.shape) != (M, N):
        raise ValueError("shape mismatch: A %s, B %s, C %s" % (tuple(A.shape), tuple(B.shape),
                                                               tuple(C.shape)))
    st = phobos_sgemm_ex(M, N, K, float(alpha), A.data_ptr(), _ld(A, "A"), B.data_ptr(),
                         _ld(B, "B"), float(beta), C.data_ptr(), _ld(C, "C"), _stream(C, stream),
                         math, plan)
    if st != PHOBOS_OK:
        raise PhobosError(st, "phobos_sgemm_ex")
    return C
