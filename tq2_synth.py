"""Seeded synthetic inputs for the TQ2_0_g128 ternary matmul.

This module is shared by the CPU oracle's tests and by the CUDA path's tests
and benchmark.  It only draws random numbers and lays them out as the raw
input buffers the method consumes; it holds none of the method's arithmetic
(no decode, no contraction, no relayout).

Inputs follow the workloads of the DiT ternary Linears described on the
"oxibonsai-image 0.2.2 src/gpu.rs" page (module doc: row-major f32
``input[M, K]``, out-major ``BlockTQ2_0_g128`` weight blocks ``[N, K/128]``,
f32 ``out[M, N]``):

* ``x``        : float32 ``[M, K]``, i.i.d. N(0, 1); optionally a set of
                 outlier channels (columns) multiplied by a factor.
* weight AoS   : uint8 ``[N, K/128, 34]``: 32 bytes of 2-bit codes followed by
                 the little-endian binary16 scale ``d``.  Each byte carries four
                 i.i.d. codes drawn from {0, 1, 2} with the requested
                 probabilities, packed into its four 2-bit fields.  Because the
                 four fields are i.i.d., the byte distribution does not depend on
                 which field holds which weight.
* ``d``        : binary16 of ``|N(0, sigma)| + 1e-4`` (round to nearest even).
* ``residual`` : float32 ``[M, N]``, i.i.d. N(0, 1), or None.

Draw order for one problem (one ``numpy.random.default_rng(seed)``):
x, outlier channel choice (if any), codes, d, residual.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

BLOCK_WEIGHTS = 128
BLOCK_BYTES = 34
QS_BYTES = 32


@dataclass
class Problem:
    """One seeded matmul problem: all host arrays, numpy-owned."""

    m: int
    n: int
    k: int
    x: np.ndarray  # float32 [m, k]
    w_aos: np.ndarray  # uint8 [n, k/128, 34]
    residual: np.ndarray | None  # float32 [m, n] or None
    seed: int
    name: str = ""


def draw_codes(rng: np.random.Generator, shape, p_zero_code: float, p_one_code: float,
               p_two_code: float) -> np.ndarray:
    """Draw i.i.d. 2-bit code values in {0, 1, 2} with the given probabilities."""
    return rng.choice(np.arange(3, dtype=np.uint8), size=shape,
                      p=[p_zero_code, p_one_code, p_two_code]).astype(np.uint8)


def pack_fields(fields: np.ndarray) -> np.ndarray:
    """Pack a trailing axis of four 2-bit fields into one byte (field f at bits 2f)."""
    assert fields.shape[-1] == 4
    f = fields.astype(np.uint8)
    return (f[..., 0] | (f[..., 1] << 2) | (f[..., 2] << 4) | (f[..., 3] << 6)).astype(np.uint8)


def make_weight_aos(rng: np.random.Generator, n: int, k: int, *, d_sigma: float,
                    code_probs=(1 / 3, 1 / 3, 1 / 3)) -> np.ndarray:
    """uint8 [n, k/128, 34] AoS weight blocks with i.i.d. codes and random scales."""
    assert k % BLOCK_WEIGHTS == 0
    kb = k // BLOCK_WEIGHTS
    fields = draw_codes(rng, (n, kb, QS_BYTES, 4), *code_probs)
    qs = pack_fields(fields)
    d = (np.abs(rng.normal(0.0, d_sigma, size=(n, kb))) + 1e-4).astype(np.float16)
    out = np.empty((n, kb, BLOCK_BYTES), dtype=np.uint8)
    out[:, :, :QS_BYTES] = qs
    out[:, :, QS_BYTES:] = d.astype("<f2").view(np.uint8).reshape(n, kb, 2)
    return out


def make_problem(m: int, n: int, k: int, *, seed: int = 0, d_sigma: float = 0.02,
                 code_probs=(1 / 3, 1 / 3, 1 / 3), outlier_frac: float = 0.0,
                 outlier_scale: float = 20.0, residual: bool = False, name: str = "") -> Problem:
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((m, k), dtype=np.float64).astype(np.float32)
    if outlier_frac > 0.0:
        n_out = int(round(outlier_frac * k))
        ch = rng.choice(k, size=n_out, replace=False)
        x[:, ch] *= np.float32(outlier_scale)
    w = make_weight_aos(rng, n, k, d_sigma=d_sigma, code_probs=code_probs)
    r = rng.standard_normal((m, n), dtype=np.float64).astype(np.float32) if residual else None
    return Problem(m=m, n=n, k=k, x=x, w_aos=w, residual=r, seed=seed, name=name)


# ----------------------------------------------------------------------------
# The five workloads.  Sizes and distributions are the stated benchmark
# configurations; only their seeds and draw order are this module's choice.
# ----------------------------------------------------------------------------

SMALL = dict(m=8, k=1024, n=1024, d_sigma=0.02)
DECODE_GATE_UP = dict(m=1, k=4096, n=12288, d_sigma=0.02, code_probs=(0.3, 0.4, 0.3))
DECODE_DOWN = dict(m=1, k=12288, n=4096, d_sigma=0.02, code_probs=(0.3, 0.4, 0.3), residual=True)
SKINNY_MS = (1, 7, 8, 9, 16, 64, 100)
SKINNY = dict(k=4096, n=4096, d_sigma=0.02)
DIT_NS = (3072, 9216, 12288)
DIT = dict(m=1536, k=3072, d_sigma=0.01, outlier_frac=0.01)

# Full DiT forward linear set: 100 layers at M=4096, in this order.
DIT_FORWARD_M = 4096
DIT_FORWARD_SHAPES = ([(3072, 3072)] * 40 + [(3072, 9216)] * 20 + [(3072, 12288)] * 20
                      + [(12288, 3072)] * 20)  # (K, N) per layer index


def small(seed: int = 0) -> Problem:
    return make_problem(**SMALL, seed=seed, name="small_m8_k1024_n1024")


def decode_gate_up(seed: int = 0) -> Problem:
    return make_problem(**DECODE_GATE_UP, seed=seed, name="decode_gemv_m1_k4096_n12288")


def decode_down(seed: int = 0) -> Problem:
    return make_problem(**DECODE_DOWN, seed=seed, name="decode_gemv_m1_k12288_n4096_res")


def skinny(m: int, seed: int = 0) -> Problem:
    return make_problem(m=m, **SKINNY, seed=seed, name=f"skinny_m{m}_k4096_n4096")


def dit(n: int, seed: int = 0) -> Problem:
    return make_problem(n=n, **DIT, seed=seed, name=f"dit_m1536_k3072_n{n}")


def dit_forward_layer(index: int, *, dist: str = "dit", m: int = DIT_FORWARD_M) -> Problem:
    """Layer ``index`` (0..99) of the 100-linear DiT forward set, seeded by its index.

    ``dist="dit"`` uses the large-M DiT distributions (1% outlier channels x20,
    sigma_d=0.01); ``dist="skinny"`` uses the skinny-sweep ones (no outliers,
    sigma_d=0.02).  Odd layer indices carry the residual epilogue.
    """
    k, n = DIT_FORWARD_SHAPES[index]
    if dist == "dit":
        kw = dict(d_sigma=0.01, outlier_frac=0.01)
    elif dist == "skinny":
        kw = dict(d_sigma=0.02)
    else:
        raise ValueError(dist)
    return make_problem(m=m, n=n, k=k, seed=index, residual=bool(index % 2), **kw,
                        name=f"dit_forward_l{index}_m{m}_k{k}_n{n}")
