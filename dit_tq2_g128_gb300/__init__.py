"""Python binding of the GB300 TQ2_0_g128 ternary matmul library.

Argument marshalling only: every entry point forwards raw device pointers,
sizes and a CUDA stream to the C ABI declared in ``include/tq2.h`` (loaded
from ``libtq2_gb300.so`` next to this file) and turns a non-zero status into
``TQ2Error``.  All arithmetic runs in the library's CUDA kernels; there is no
Python or CPU fallback, and importing this package fails loudly when the
library has not been built.

Arguments that take device memory accept a torch CUDA tensor or a raw integer
pointer.  ``stream`` accepts a ``torch.cuda.Stream``, a raw ``cudaStream_t``
integer, or None (the current torch stream when torch is importable, else the
legacy default stream).
"""

from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtq2_gb300.so")

TQ2_OK = 0
TQ2_ERR_INVALID_ARG = 1
TQ2_ERR_BAD_K = 2
TQ2_ERR_MISALIGNED = 3
TQ2_ERR_UNSUPPORTED_DEVICE = 4
TQ2_ERR_CUDA = 5
TQ2_ERR_TIMEOUT = 6
TQ2_ERR_TOO_LARGE = 7
TQ2_NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024

TQ2_KERNEL_AUTO = 0
TQ2_KERNEL_GEMV = 1
TQ2_KERNEL_SKINNY = 2
TQ2_KERNEL_TC = 3
TQ2_KERNEL_F32REF = 4
TQ2_KERNEL_TC_DIRECT = 5
TQ2_KERNEL_SKINNY_MMA = 6
KERNEL_NAMES = {0: "auto", 1: "gemv", 2: "skinny", 3: "tc", 4: "f32ref", 5: "tc_direct", 6: "skinny_mma"}

# Every symbol include/tq2.h declares.
EXPORTS = (
    "tq2_soa_bytes", "tq2_status_string", "tq2_reformat_aos_to_soa", "tq2_gemv", "tq2_gemv_resident",
    "tq2_gemm",
    "tq2_gemm_f32ref", "tq2_gemm_with", "tq2_select_kernel", "tq2_set_wait_timeout_ns",
    "tq2_device_status", "tq2_version", "tq2_gemm_workspace_bytes", "tq2_gemm_ws",
    "tq2_gemm_noalloc", "tq2_quantize_f32", "tq2_gate_up_swiglu", "tq2_gate_up_swiglu_resident",
    "tq2_act16_from_f32",
    "tq2_act16_to_f32", "tq2_gemm_act16", "tq2_attention_f32",
)


class TQ2Error(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}" if what else status_string(status))


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build the CUDA library first "
            "(python -m dit_tq2_g128_gb300.build, or __graft_entry__.build())")
    L = ctypes.CDLL(LIB_PATH)
    i64, vp, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    L.tq2_soa_bytes.restype = ctypes.c_size_t
    L.tq2_soa_bytes.argtypes = [i64, i64]
    L.tq2_status_string.restype = ctypes.c_char_p
    L.tq2_status_string.argtypes = [i32]
    L.tq2_reformat_aos_to_soa.restype = i32
    L.tq2_reformat_aos_to_soa.argtypes = [vp, vp, i64, i64, vp]
    for name in ("tq2_gemv", "tq2_gemv_resident"):
        f = getattr(L, name)
        f.restype = i32
        f.argtypes = [vp, vp, vp, vp, i64, i64, vp]
    for name in ("tq2_gemm", "tq2_gemm_f32ref"):
        f = getattr(L, name)
        f.restype = i32
        f.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp]
    L.tq2_gemm_with.restype = i32
    L.tq2_gemm_with.argtypes = [i32, vp, vp, vp, vp, i64, i64, i64, vp]
    L.tq2_select_kernel.restype = i32
    L.tq2_select_kernel.argtypes = [i64, i64, i64]
    L.tq2_set_wait_timeout_ns.restype = ctypes.c_uint64
    L.tq2_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
    L.tq2_device_status.restype = i32
    L.tq2_device_status.argtypes = [vp]
    L.tq2_version.restype = i32
    L.tq2_version.argtypes = []
    L.tq2_gemm_workspace_bytes.restype = ctypes.c_size_t
    L.tq2_gemm_workspace_bytes.argtypes = [i64, i64, i64]
    L.tq2_gemm_ws.restype = i32
    L.tq2_gemm_ws.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp, ctypes.c_size_t, vp]
    L.tq2_quantize_f32.restype = i32
    L.tq2_quantize_f32.argtypes = [vp, vp, i64, i64, vp]
    L.tq2_act16_from_f32.restype = i32
    L.tq2_act16_from_f32.argtypes = [vp, vp, i64, i64, vp]
    L.tq2_act16_to_f32.restype = i32
    L.tq2_act16_to_f32.argtypes = [vp, vp, i64, i64, vp]
    L.tq2_gemm_act16.restype = i32
    L.tq2_gemm_act16.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp]
    L.tq2_attention_f32.restype = i32
    L.tq2_attention_f32.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp]
    for name in ("tq2_gate_up_swiglu", "tq2_gate_up_swiglu_resident"):
        f = getattr(L, name)
        f.restype = i32
        f.argtypes = [vp, vp, vp, i64, i64, i64, vp]
    L.tq2_gemm_noalloc.restype = i32
    L.tq2_gemm_noalloc.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp]
    return L


lib = _load()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        try:
            import torch
            if torch.cuda.is_available() and torch.cuda.is_initialized():
                return torch.cuda.current_stream().cuda_stream
        except ImportError:  # pragma: no cover
            pass
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, what: str):
    if status != TQ2_OK:
        raise TQ2Error(status, what)


def status_string(status: int) -> str:
    return lib.tq2_status_string(int(status)).decode()


tq2_status_string = status_string


def tq2_soa_bytes(n: int, k: int) -> int:
    return int(lib.tq2_soa_bytes(n, k))


def tq2_version() -> int:
    return int(lib.tq2_version())


def tq2_select_kernel(m: int, n: int, k: int) -> int:
    return int(lib.tq2_select_kernel(m, n, k))


def tq2_set_wait_timeout_ns(ns: int) -> int:
    return int(lib.tq2_set_wait_timeout_ns(int(ns)))


def tq2_device_status(stream=None) -> int:
    """Synchronise ``stream`` and return (and clear) the device status word."""
    return int(lib.tq2_device_status(_stream(stream)))


def tq2_reformat_aos_to_soa(w_aos, w_soa, n: int, k: int, stream=None) -> None:
    _check(lib.tq2_reformat_aos_to_soa(_ptr(w_aos), _ptr(w_soa), n, k, _stream(stream)),
           "tq2_reformat_aos_to_soa")


def tq2_quantize_f32(w, w_aos, n: int, k: int, stream=None) -> None:
    _check(lib.tq2_quantize_f32(_ptr(w), _ptr(w_aos), n, k, _stream(stream)), "tq2_quantize_f32")


def tq2_act16_from_f32(x, x16, m: int, k: int, stream=None) -> None:
    _check(lib.tq2_act16_from_f32(_ptr(x), _ptr(x16), m, k, _stream(stream)), "tq2_act16_from_f32")


def tq2_act16_to_f32(x16, x, m: int, k: int, stream=None) -> None:
    _check(lib.tq2_act16_to_f32(_ptr(x16), _ptr(x), m, k, _stream(stream)), "tq2_act16_to_f32")


def tq2_gemm_act16(w_soa, x16, residual16, out16, m: int, n: int, k: int, stream=None) -> None:
    _check(lib.tq2_gemm_act16(_ptr(w_soa), _ptr(x16), _ptr(residual16), _ptr(out16), m, n, k,
                              _stream(stream)), "tq2_gemm_act16")


def tq2_attention_f32(q, k, v, out, heads: int, seq: int, dim: int, stream=None) -> None:
    _check(lib.tq2_attention_f32(_ptr(q), _ptr(k), _ptr(v), _ptr(out), heads, seq, dim, _stream(stream)),
           "tq2_attention_f32")


def tq2_gate_up_swiglu(w_soa, x, out, m: int, f: int, k: int, stream=None) -> None:
    _check(lib.tq2_gate_up_swiglu(_ptr(w_soa), _ptr(x), _ptr(out), m, f, k, _stream(stream)),
           "tq2_gate_up_swiglu")


def tq2_gate_up_swiglu_resident(w_soa, x, out, m: int, f: int, k: int, stream=None) -> None:
    _check(lib.tq2_gate_up_swiglu_resident(_ptr(w_soa), _ptr(x), _ptr(out), m, f, k, _stream(stream)),
           "tq2_gate_up_swiglu_resident")


def tq2_gemv(w_soa, x, residual, out, n: int, k: int, stream=None) -> None:
    _check(lib.tq2_gemv(_ptr(w_soa), _ptr(x), _ptr(residual), _ptr(out), n, k, _stream(stream)),
           "tq2_gemv")


def tq2_gemv_resident(w_soa, x, residual, out, n: int, k: int, stream=None) -> None:
    _check(lib.tq2_gemv_resident(_ptr(w_soa), _ptr(x), _ptr(residual), _ptr(out), n, k,
                                 _stream(stream)), "tq2_gemv_resident")


def tq2_gemm(w_soa, x, residual, out, m: int, n: int, k: int, stream=None) -> None:
    _check(lib.tq2_gemm(_ptr(w_soa), _ptr(x), _ptr(residual), _ptr(out), m, n, k,
                        _stream(stream)), "tq2_gemm")


def tq2_gemm_f32ref(w_soa, x, residual, out, m: int, n: int, k: int, stream=None) -> None:
    _check(lib.tq2_gemm_f32ref(_ptr(w_soa), _ptr(x), _ptr(residual), _ptr(out), m, n, k,
                               _stream(stream)), "tq2_gemm_f32ref")


def tq2_gemm_workspace_bytes(m: int, n: int, k: int) -> int:
    return int(lib.tq2_gemm_workspace_bytes(m, n, k))


def tq2_gemm_ws(w_soa, x, residual, out, m: int, n: int, k: int, workspace, workspace_bytes: int,
                stream=None) -> None:
    _check(lib.tq2_gemm_ws(_ptr(w_soa), _ptr(x), _ptr(residual), _ptr(out), m, n, k,
                           _ptr(workspace), int(workspace_bytes), _stream(stream)), "tq2_gemm_ws")


def tq2_gemm_noalloc(w_soa, x, residual, out, m: int, n: int, k: int, stream=None) -> None:
    """tq2_gemm without any device allocation (fixed library scratch; see include/tq2.h)."""
    _check(lib.tq2_gemm_noalloc(_ptr(w_soa), _ptr(x), _ptr(residual), _ptr(out), m, n, k,
                                _stream(stream)), "tq2_gemm_noalloc")


def tq2_gemm_with(kernel: int, w_soa, x, residual, out, m: int, n: int, k: int,
                  stream=None) -> None:
    _check(lib.tq2_gemm_with(int(kernel), _ptr(w_soa), _ptr(x), _ptr(residual), _ptr(out), m, n,
                             k, _stream(stream)), f"tq2_gemm_with({KERNEL_NAMES.get(kernel)})")


# ---------------------------------------------------------------------------
# Tensor-level conveniences (shape and dtype checks, then the calls above).


def _check_tensor(t, name, dtype, numel):
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if str(t.dtype) != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.numel() != numel:
        raise ValueError(f"{name} has {t.numel()} elements, expected {numel}")


def upload_weight(w_aos_host, n: int, k: int, stream=None):
    """Copy AoS blocks (numpy uint8 or torch CPU tensor) to the device and
    relayout them to SoA; returns the SoA uint8 CUDA tensor (caller-owned)."""
    import numpy as np
    import torch
    nbytes = tq2_soa_bytes(n, k)
    if nbytes == 0 and n:
        raise TQ2Error(TQ2_ERR_BAD_K, "upload_weight")
    src = torch.from_numpy(np.ascontiguousarray(w_aos_host, dtype=np.uint8).reshape(-1)) \
        if not isinstance(w_aos_host, torch.Tensor) else w_aos_host.reshape(-1)
    if src.numel() != nbytes:
        raise ValueError(f"weight has {src.numel()} bytes, expected {nbytes}")
    aos = src.to("cuda", non_blocking=False)
    soa = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    tq2_reformat_aos_to_soa(aos, soa, n, k, stream)
    return soa


def workspace(m: int, n: int, k: int, device="cuda"):
    """A device workspace for tq2_gemm_ws (torch uint8 tensor; None if not needed)."""
    import torch
    nbytes = tq2_gemm_workspace_bytes(m, n, k)
    return torch.empty(nbytes, dtype=torch.uint8, device=device) if nbytes else None


def matmul(w_soa, x, residual=None, *, n: int, k: int, out=None, kernel: int = TQ2_KERNEL_AUTO,
           workspace=None, stream=None):
    """out[M, N] = x[M, K] . dequant(W)^T (+ residual) on torch CUDA tensors.

    With ``workspace`` (see ``workspace()``) and kernel AUTO, runs tq2_gemm_ws."""
    import torch
    m = x.numel() // k if k else 0
    _check_tensor(w_soa, "w_soa", "torch.uint8", tq2_soa_bytes(n, k))
    _check_tensor(x, "x", "torch.float32", m * k)
    if residual is not None:
        _check_tensor(residual, "residual", "torch.float32", m * n)
    if out is None:
        out = torch.empty((m, n), dtype=torch.float32, device=x.device)
    _check_tensor(out, "out", "torch.float32", m * n)
    if workspace is not None and kernel == TQ2_KERNEL_AUTO:
        tq2_gemm_ws(w_soa, x, residual, out, m, n, k, workspace, workspace.numel(), stream)
    else:
        tq2_gemm_with(kernel, w_soa, x, residual, out, m, n, k, stream)
    return out
