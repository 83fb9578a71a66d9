"""Shared helpers of the GPU parity tests: run the library through its C ABI on
torch device buffers and compare with the CPU oracle."""
import numpy as np

import language_fp32_gemm_gb300 as phobos
import oracle


def padded(x, extra_cols):
    """A view of ``x`` inside a wider row-major buffer (leading dimension grows)."""
    if extra_cols == 0:
        return x
    buf = np.full((x.shape[0], x.shape[1] + extra_cols), np.float32(7.0), dtype=np.float32)
    buf[:, :x.shape[1]] = x
    return buf[:, :x.shape[1]]


def to_device(x, torch, dev, offset=0):
    """Copy a (possibly padded) numpy view to the device, keeping its leading dimension.

    ``offset`` shifts the data by that many floats inside the allocation, so a
    non-zero odd offset gives a pointer that is not 16-byte aligned.  Returns
    (tensor view, backing tensor).
    """
    rows, cols = x.shape
    ld = max(x.strides[0] // 4, cols, 1) if rows > 1 else max(cols, 1)
    total = (rows - 1) * ld + cols if rows > 0 and cols > 0 else 0
    flat = np.zeros(offset + max(total, 1), dtype=np.float32)
    if total:
        base = np.lib.stride_tricks.as_strided(flat[offset:], shape=(rows, cols), strides=(4 * ld, 4))
        base[...] = x
    backing = torch.from_numpy(flat).to(dev)
    view = torch.as_strided(backing, (rows, cols), (ld, 1), offset)
    return view, backing


def run_gemm(torch, dev, A, B, C0, alpha, beta, math, plan=None, offsets=(0, 0, 0)):
    """Run C = alpha*A*B + beta*C0 on the GPU; return C as a numpy array."""
    dA, _ka = to_device(A, torch, dev, offsets[0])
    dB, _kb = to_device(B, torch, dev, offsets[1])
    dC, _kc = to_device(C0, torch, dev, offsets[2])
    phobos.sgemm(dA, dB, dC, alpha, beta, math=math, plan=plan)
    torch.cuda.synchronize()
    st = phobos.phobos_check_device(0)
    assert st == phobos.PHOBOS_OK, phobos.status_string(st)
    return dC.cpu().numpy()


def tolerance(math):
    return oracle.TOL_TF32 if math == "tf32" else oracle.TOL_FP32
