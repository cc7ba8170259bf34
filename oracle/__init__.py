"""CPU oracle for the TQ2_0_g128 ternary matmul -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or runs anything here, and this
package imports nothing from the product.

The arithmetic lives in ``tq2_oracle.c`` (plain C, double precision, a naive
loop per output element); this module compiles it with the host C compiler on
first use and marshals numpy arrays to it.  See that file's header for the
definition it restates and the passages it follows.

Pins (all in ``tests/test_oracle.py``): the binary16 decoder against numpy's
float16 for all 65536 bit patterns; hand-built blocks whose results are short
closed forms (all +1, all 0, all -1, alternating signs, every single-code
position); the contraction against ``numpy.matmul`` of the dequantised matrix;
invariants (linearity, negation, exact doubling under d*2, row-wise equals
batched, residual passthrough) and the SoA layout on a hand-built example plus
the AoS->SoA->AoS round trip.  The gate/up SwiGLU (``swiglu``) is pinned by
the closed form silu(ln 3) = 0.75 ln 3, the odd identity silu(z) - silu(-z) = z
(flipping every gate code), zero gate or up rows, exact linearity in the up
rows and the limits silu(z) -> z and -> 0.  The DiT joint attention
(``attention``) is pinned by closed forms (identical keys give the mean of v,
one key gives v, a two-key case is a logistic weight), a dominant key, and
permutation equivariance over keys and queries.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tq2_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libtq2_oracle.so")
_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_p = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile ``tq2_oracle.c`` into ``_build/libtq2_oracle.so`` (OpenMP if available)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            L.tq2o_half_to_double.restype = ctypes.c_double
            L.tq2o_half_to_double.argtypes = [ctypes.c_uint16]
            L.tq2o_dequant.restype = ctypes.c_int
            L.tq2o_dequant.argtypes = [_p, _i64, _i64, _p]
            L.tq2o_matmul.restype = ctypes.c_int
            L.tq2o_matmul.argtypes = [_p, _p, _p, _i64, _i64, _i64, _p, _i64, _p, _p]
            L.tq2o_weight_bytes.restype = _i64
            L.tq2o_weight_bytes.argtypes = [_i64, _i64]
            L.tq2o_aos_to_soa.restype = ctypes.c_int
            L.tq2o_aos_to_soa.argtypes = [_p, _p, _i64, _i64]
            L.tq2o_soa_to_aos.restype = ctypes.c_int
            L.tq2o_soa_to_aos.argtypes = [_p, _p, _i64, _i64]
            L.tq2o_threads.restype = ctypes.c_int
            L.tq2o_set_threads.argtypes = [ctypes.c_int]
            L.tq2o_double_to_half.restype = ctypes.c_uint16
            L.tq2o_double_to_half.argtypes = [ctypes.c_double]
            L.tq2o_quantize.restype = ctypes.c_int
            L.tq2o_quantize.argtypes = [_p, _i64, _i64, _p]
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def threads() -> int:
    return lib().tq2o_threads()


def set_threads(t: int) -> None:
    lib().tq2o_set_threads(int(t))


def half_to_double(bits: int) -> float:
    return lib().tq2o_half_to_double(int(bits) & 0xFFFF)


def _aos(w_aos, n, k):
    w = np.ascontiguousarray(w_aos, dtype=np.uint8)
    assert w.size == weight_bytes(n, k), (w.size, n, k)
    return w


def weight_bytes(n: int, k: int) -> int:
    return int(lib().tq2o_weight_bytes(n, k))


def dequant(w_aos, n: int, k: int) -> np.ndarray:
    """Dense float64 [n, k] weight: (code - 1) * d for every weight."""
    w = _aos(w_aos, n, k)
    out = np.empty((n, k), dtype=np.float64)
    rc = lib().tq2o_dequant(_ptr(w), n, k, _ptr(out))
    if rc:
        raise ValueError(f"tq2o_dequant: k={k} is not a positive multiple of 128")
    return out


def matmul(w_aos, x, residual=None, *, n: int, k: int, rows=None):
    """float64 (out, absdot), each [len(rows) or M, N].

    out = x[rows] . dequant(W)^T (+ residual[rows]);
    absdot = sum_k |x[rows, k] * dequant(W)[:, k]|, the per-element scale of the
    tolerance bounds.
    """
    w = _aos(w_aos, n, k)
    x = np.ascontiguousarray(x, dtype=np.float32)
    m = x.shape[0] if x.ndim == 2 else 1
    assert x.size == m * k
    r = None if residual is None else np.ascontiguousarray(residual, dtype=np.float32)
    if r is not None:
        assert r.size == m * n
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        assert rows.ndim == 1 and (rows.size == 0 or (rows.min() >= 0 and rows.max() < m))
        n_rows = rows.size
    else:
        n_rows = m
    out = np.empty((n_rows, n), dtype=np.float64)
    absdot = np.empty((n_rows, n), dtype=np.float64)
    if n_rows and n:
        rc = lib().tq2o_matmul(_ptr(w), _ptr(x), _ptr(r), m, n, k, _ptr(rows), n_rows,
                               _ptr(out), _ptr(absdot))
        if rc == -1:
            raise ValueError(f"tq2o_matmul: k={k} is not a positive multiple of 128")
        if rc:
            raise MemoryError("tq2o_matmul: allocation failed")
    return out, absdot


def aos_to_soa(w_aos, n: int, k: int) -> np.ndarray:
    w = _aos(w_aos, n, k)
    out = np.empty(w.size, dtype=np.uint8)
    if lib().tq2o_aos_to_soa(_ptr(w), _ptr(out), n, k):
        raise ValueError("bad k")
    return out


def soa_to_aos(w_soa, n: int, k: int) -> np.ndarray:
    s = np.ascontiguousarray(w_soa, dtype=np.uint8).reshape(-1)
    assert s.size == weight_bytes(n, k)
    out = np.empty(s.size, dtype=np.uint8)
    if lib().tq2o_soa_to_aos(_ptr(s), _ptr(out), n, k):
        raise ValueError("bad k")
    return out.reshape(n, k // 128, 34)


def double_to_half(v: float) -> int:
    """binary16 bits of v, round to nearest even (the oracle's own conversion)."""
    return int(lib().tq2o_double_to_half(float(v)))


def quantize(w, n: int, k: int) -> np.ndarray:
    """Encoder: f32 weights [n, k] -> uint8 AoS blocks [n, k/128, 34] (absmean
    scale per 128-weight block, binary16 round to nearest even, codes
    clamp(rint(w / d), -1, 1) + 1 in binary32)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    assert w.size == n * k
    out = np.zeros((n, k // 128 if k > 0 else 0, 34), dtype=np.uint8)
    if lib().tq2o_quantize(_ptr(w), n, k, _ptr(out)) == -1:
        raise ValueError(f"tq2o_quantize: k={k} is not a positive multiple of 128")
    return out


def silu(z):
    """SiLU in float64: z * sigmoid(z) = z / (1 + exp(-z)) (the element-wise
    activation the pages dispatch as ``silu_f32``, "oxibonsai-kernels 0.1.5
    src/gpu_backend/metal_graph/pipelines.rs", FLUX.2 VAE primitives)."""
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def swiglu(w_aos, x, *, f: int, k: int, rows=None):
    """Fused gate/up projection with the SwiGLU activation, float64.

    The TQ2 analogue of the pages' ``fused_gate_up_swiglu_q1`` /
    ``fused_gate_up_swiglu_gemm_q1`` pipelines ("oxibonsai-kernels 0.1.5
    src/gpu_backend/metal_graph/pipelines.rs", decode and prefill fields),
    which the pages name without a listing.  Reading: the weight holds 2f rows,
    the gate projection in rows [0, f) and the up projection in rows [f, 2f);
    for each input row, g = x . W_gate^T, u = x . W_up^T and
    h = silu(g) * u, f values.

    Returns (h, g, u, absdot_g, absdot_u), each [len(rows) or M, f]; the
    absdot arrays are sum_k |x w| of the gate and up rows (the tolerance scales).
    """
    out, absdot = matmul(w_aos, x, n=2 * f, k=k, rows=rows)
    g, u = out[:, :f], out[:, f:]
    return silu(g) * u, g, u, absdot[:, :f], absdot[:, f:]


def attention(q, k, v, *, heads: int, seq: int, dim: int, rows=None):
    """DiT joint multi-head attention, float64: the contract of the pages'
    ``joint_attention_gpu`` ("oxibonsai-image 0.2.2 src/gpu.rs", its doc
    comment; kernel ``joint_attention_flash_f32`` of "oxibonsai-kernels 0.1.5
    src/gpu_backend/metal_graph/pipelines.rs", FLUX.2 DiT joint attention).

    q, k, v: head-major [heads, seq, dim] (float32 inputs);
    out[t, h*dim + d] = sum_j p[h, t, j] v[h, j, d] with
    p[h, t, :] = softmax_j(q[h, t] . k[h, j] / sqrt(dim)) over all keys
    (non-causal).  Token-major output [seq, heads*dim] (or the token rows
    `rows`).  The softmax subtracts the row maximum before exponentiating.

    Returns (out, absv): absv[t, h*dim + d] = sum_j p[h, t, j] |v[h, j, d]|, the
    scale of the tolerance bounds.
    """
    q = np.asarray(q, dtype=np.float64).reshape(heads, seq, dim)
    k = np.asarray(k, dtype=np.float64).reshape(heads, seq, dim)
    v = np.asarray(v, dtype=np.float64).reshape(heads, seq, dim)
    t = np.arange(seq) if rows is None else np.asarray(rows, dtype=np.int64)
    out = np.empty((t.size, heads * dim))
    absv = np.empty((t.size, heads * dim))
    scale = 1.0 / np.sqrt(dim)
    for h in range(heads):
        s = (q[h, t] @ k[h].T) * scale               # [rows, seq]
        s -= s.max(axis=1, keepdims=True)
        e = np.exp(s)
        p = e / e.sum(axis=1, keepdims=True)
        out[:, h * dim:(h + 1) * dim] = p @ v[h]
        absv[:, h * dim:(h + 1) * dim] = p @ np.abs(v[h])
    return out, absv
