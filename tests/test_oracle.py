"""Pins for the CPU oracle (no GPU).

The oracle is checked against things other than itself: numpy's binary16
decoder, closed-form results on hand-built blocks (bytes written literally),
numpy.matmul on the dequantised matrix, algebraic invariants, and the one
worked example the pages print (two all-zero blocks are 68 bytes).
"""

import os

import numpy as np
import pytest

import oracle
import tq2_synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

HALF_0_5 = 0x3800  # binary16 bits of 0.5
HALF_0_375 = 0x3600  # 0.375
HALF_3 = 0x4200  # 3.0


def block(qs_byte_values, d_bits):
    """One 34-byte block from 32 literal qs bytes and the 16-bit scale bits."""
    qs = np.asarray(qs_byte_values, dtype=np.uint8)
    assert qs.shape == (32,)
    return np.concatenate([qs, np.array([d_bits & 0xFF, d_bits >> 8], dtype=np.uint8)])


def weight(blocks, n, k):
    return np.concatenate(blocks).reshape(n, k // 128, 34)


def rand_x(m, k, seed=1):
    return np.random.default_rng(seed).standard_normal((m, k)).astype(np.float32)


# --------------------------------------------------------------------------
# binary16 decoding


def test_half_decoder_matches_numpy_for_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint32)
    ref = bits.astype(np.uint16).view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signs of zeros, too
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


# --------------------------------------------------------------------------
# the pages' worked example


def test_golden_two_zero_blocks():
    vals = {}
    blocks = []
    with open(os.path.join(GOLDEN, "two_zero_blocks.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            parts = line.split()
            if parts[0].startswith("block") and parts[0] != "block_bytes":
                blocks.append(bytes.fromhex(parts[1] + parts[2]))
            else:
                vals[parts[0]] = int(parts[1])
    assert all(len(b) == vals["block_bytes"] for b in blocks)
    raw = np.frombuffer(b"".join(blocks), dtype=np.uint8)
    assert raw.size == vals["total_bytes"] == 68
    # as one weight row of K=256 (two blocks)
    assert oracle.weight_bytes(1, 256) == vals["total_bytes"]
    w = oracle.dequant(raw, 1, 256)
    assert np.all(w == 0.0)
    out, absdot = oracle.matmul(raw, rand_x(3, 256), n=1, k=256)
    assert np.all(out == 0.0) and np.all(absdot == 0.0)


# --------------------------------------------------------------------------
# hand-built blocks with closed-form results


@pytest.mark.parametrize("k", [128, 256])
def test_all_plus_one(k):
    # byte 0xAA = fields 2,2,2,2 -> every weight +1; d = 0.5
    blk = block([0xAA] * 32, HALF_0_5)
    w = weight([blk] * (k // 128), 1, k)
    x = rand_x(2, k)
    out, absdot = oracle.matmul(w, x, n=1, k=k)
    ref = 0.5 * x.astype(np.float64).sum(axis=1)
    np.testing.assert_allclose(out[:, 0], ref, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(absdot[:, 0], 0.5 * np.abs(x.astype(np.float64)).sum(axis=1),
                               rtol=1e-13)


def test_all_zero_weight_gives_residual_exactly():
    # byte 0x55 = fields 1,1,1,1 -> every weight 0
    k, n, m = 256, 3, 4
    w = weight([block([0x55] * 32, HALF_3)] * (n * k // 128), n, k)
    x = rand_x(m, k)
    res = rand_x(m, n, seed=5)
    out, absdot = oracle.matmul(w, x, res, n=n, k=k)
    assert np.array_equal(out, res.astype(np.float64))
    assert np.all(absdot == 0.0)
    out0, _ = oracle.matmul(w, x, n=n, k=k)
    assert np.all(out0 == 0.0)


def test_all_minus_one():
    # byte 0x00 = fields 0,0,0,0 -> every weight -1
    k = 128
    w = weight([block([0x00] * 32, HALF_0_375)], 1, k)
    x = rand_x(3, k)
    out, _ = oracle.matmul(w, x, n=1, k=k)
    np.testing.assert_allclose(out[:, 0], -0.375 * x.astype(np.float64).sum(axis=1),
                               rtol=1e-13, atol=1e-13)


def test_field_order_within_byte():
    # 0x88 = 0b10_00_10_00: field0=0 (-1), field1=2 (+1), field2=0 (-1), field3=2 (+1)
    # so weight j is +1 for j%4 in {1,3}, -1 for j%4 in {0,2}
    k = 128
    x = rand_x(2, k).astype(np.float64)
    j = np.arange(k)
    w = weight([block([0x88] * 32, HALF_0_5)], 1, k)
    out, _ = oracle.matmul(w, x.astype(np.float32), n=1, k=k)
    ref = 0.5 * (x[:, j % 2 == 1].sum(1) - x[:, j % 2 == 0].sum(1))
    np.testing.assert_allclose(out[:, 0], ref, rtol=1e-12, atol=1e-12)
    # 0x06 = 0b00_00_01_10: field0=2 (+1), field1=1 (0), field2=0 (-1), field3=0 (-1)
    w = weight([block([0x06] * 32, HALF_0_5)], 1, k)
    out, _ = oracle.matmul(w, x.astype(np.float32), n=1, k=k)
    ref = 0.5 * (x[:, j % 4 == 0].sum(1) - x[:, j % 4 >= 2].sum(1))
    np.testing.assert_allclose(out[:, 0], ref, rtol=1e-12, atol=1e-12)


def test_every_single_code_position_selects_one_input():
    # All fields 1 (weight 0) except weight j set to field value 2 (+1):
    # out[:, 0] must be x[:, j] * d exactly, for every j of the block, in the
    # second block of the row (so the block index is exercised too).
    k = 256
    x = rand_x(3, k)
    for j in range(128):
        qs = np.full(32, 0x55, dtype=np.uint8)
        s = 2 * (j % 4)
        qs[j // 4] = (0x55 & ~(3 << s)) | (2 << s)
        w = weight([block([0x55] * 32, HALF_0_5), block(qs, HALF_3)], 1, k)
        dense = oracle.dequant(w, 1, k)
        expect = np.zeros(k)
        expect[128 + j] = 3.0
        assert np.array_equal(dense[0], expect), j
        out, _ = oracle.matmul(w, x, n=1, k=k)
        assert np.array_equal(out[:, 0], 3.0 * x[:, 128 + j].astype(np.float64)), j


def test_tiny_multi_row_hand_values():
    # N=3 rows, K=128, M=2; x = ones for row 0 and ramp for row 1.
    k = 128
    x = np.stack([np.ones(k), np.arange(k)]).astype(np.float32)
    rows = [block([0xAA] * 32, HALF_0_5),   # +0.5 everywhere
            block([0x00] * 32, HALF_3),     # -3 everywhere
            block([0x55] * 32, HALF_3)]     # 0 everywhere
    w = weight(rows, 3, k)
    out, _ = oracle.matmul(w, x, n=3, k=k)
    s = k * (k - 1) / 2
    expect = np.array([[0.5 * k, -3.0 * k, 0.0], [0.5 * s, -3.0 * s, 0.0]])
    assert np.array_equal(out, expect)


def test_code3_decodes_arithmetically_to_plus_two():
    k = 128
    w = weight([block([0xFF] * 32, HALF_0_5)], 1, k)
    assert np.all(oracle.dequant(w, 1, k) == 1.0)


# --------------------------------------------------------------------------
# the contraction against a library matmul on the dequantised matrix


@pytest.mark.parametrize("m,n,k", [(1, 7, 128), (5, 3, 384), (8, 64, 1024)])
def test_contraction_matches_numpy_matmul(m, n, k):
    p = tq2_synth.make_problem(m, n, k, seed=m + n + k, residual=True, outlier_frac=0.02)
    W = oracle.dequant(p.w_aos, n, k)
    x64 = p.x.astype(np.float64)
    ref = np.matmul(x64, W.T) + p.residual.astype(np.float64)
    out, absdot = oracle.matmul(p.w_aos, p.x, p.residual, n=n, k=k)
    scale = np.matmul(np.abs(x64), np.abs(W).T)
    np.testing.assert_allclose(absdot, scale, rtol=1e-12)
    assert np.all(np.abs(out - ref) <= 1e-12 * (scale + np.abs(ref) + 1e-300))


# --------------------------------------------------------------------------
# invariants


def test_linearity_in_x():
    n, k, m = 16, 256, 3
    p = tq2_synth.make_problem(m, n, k, seed=3)
    rng = np.random.default_rng(11)
    # integer-valued inputs so that 3x - 2y is exact in float32
    x = rng.integers(-8, 9, size=(m, k)).astype(np.float32)
    y = rng.integers(-8, 9, size=(m, k)).astype(np.float32)
    fx, sx = oracle.matmul(p.w_aos, x, n=n, k=k)
    fy, sy = oracle.matmul(p.w_aos, y, n=n, k=k)
    fz, _ = oracle.matmul(p.w_aos, 3 * x - 2 * y, n=n, k=k)
    tol = 1e-13 * (3 * sx + 2 * sy)
    assert np.all(np.abs(fz - (3 * fx - 2 * fy)) <= tol)


def test_negation_and_scale_doubling_are_exact():
    n, k, m = 8, 384, 4
    p = tq2_synth.make_problem(m, n, k, seed=4)
    f, _ = oracle.matmul(p.w_aos, p.x, n=n, k=k)
    fneg, _ = oracle.matmul(p.w_aos, -p.x, n=n, k=k)
    assert np.array_equal(fneg, -f)
    w2 = p.w_aos.copy()
    d = w2[:, :, 32:].copy().view("<f2")
    w2[:, :, 32:] = (d.astype(np.float32) * 2).astype("<f2").view(np.uint8)
    f2, _ = oracle.matmul(w2, p.x, n=n, k=k)
    assert np.array_equal(f2, 2 * f)


def test_rows_equal_batched_and_subset():
    n, k, m = 12, 256, 6
    p = tq2_synth.make_problem(m, n, k, seed=6, residual=True)
    full, _ = oracle.matmul(p.w_aos, p.x, p.residual, n=n, k=k)
    for r in range(m):
        one, _ = oracle.matmul(p.w_aos, p.x[r:r + 1], p.residual[r:r + 1], n=n, k=k)
        assert np.array_equal(one[0], full[r])
    sub, _ = oracle.matmul(p.w_aos, p.x, p.residual, n=n, k=k, rows=[5, 0, 3])
    assert np.array_equal(sub, full[[5, 0, 3]])


def test_bad_k_is_rejected():
    L = oracle.lib()
    for k in (0, -128, 64, 200):
        assert L.tq2o_dequant(None, 1, k, None) == -1
        assert L.tq2o_matmul(None, None, None, 1, 1, k, None, 0, None, None) == -1
        assert L.tq2o_aos_to_soa(None, None, 1, k) == -1
        assert L.tq2o_soa_to_aos(None, None, 1, k) == -1


# --------------------------------------------------------------------------
# SoA layout


def test_soa_layout_hand_example():
    n, k = 2, 256  # 4 blocks in row-major (n, b) order
    blocks = []
    for i in range(4):
        qs = (np.arange(32) + 32 * i).astype(np.uint8)
        blocks.append(block(qs, 0x1100 + i))  # d bytes: low = i, high = 0x11
    w = weight(blocks, n, k)
    soa = oracle.aos_to_soa(w, n, k)
    assert soa.size == 4 * 34
    assert np.array_equal(soa[:128], np.arange(128, dtype=np.uint8))
    assert np.array_equal(soa[128:], np.array([0, 0x11, 1, 0x11, 2, 0x11, 3, 0x11], np.uint8))


@pytest.mark.parametrize("n,k", [(1, 128), (3, 384), (17, 1024)])
def test_soa_round_trip(n, k):
    p = tq2_synth.make_problem(1, n, k, seed=n * k)
    soa = oracle.aos_to_soa(p.w_aos, n, k)
    assert soa.size == p.w_aos.size
    back = oracle.soa_to_aos(soa, n, k)
    assert np.array_equal(back, p.w_aos)


# --------------------------------------------------------------------------
# the input generator (draws only; checked here so both sides can trust it)


def test_generator_distributions():
    p = tq2_synth.decode_gate_up()
    assert p.x.shape == (1, 4096) and p.w_aos.shape == (12288, 32, 34)
    qs = p.w_aos[:, :, :32].reshape(-1)
    fields = np.stack([(qs >> s) & 3 for s in (0, 2, 4, 6)]).reshape(-1)
    frac = np.bincount(fields, minlength=4) / fields.size
    assert frac[3] == 0.0
    np.testing.assert_allclose(frac[:3], [0.3, 0.4, 0.3], atol=2e-3)
    d = p.w_aos[:, :, 32:].copy().view("<f2").astype(np.float64)
    assert d.min() >= 1e-4 * 0.999
    np.testing.assert_allclose(np.mean(d - 1e-4), 0.02 * np.sqrt(2 / np.pi), rtol=0.02)
    q = tq2_synth.dit(3072)
    col_absmax = np.abs(q.x).max(axis=0)
    assert (col_absmax > 10).sum() == round(0.01 * 3072)


# ---------------------------------------------------------------------------
# Encoder (f32 -> blocks): this library's absmean reading, pinned to closed
# forms and to numpy's own binary16 conversion.


def _codes(blk):
    """The 128 codes of one 34-byte block."""
    b = np.asarray(blk, dtype=np.uint8)
    return np.array([(b[j // 4] >> (2 * (j % 4))) & 3 for j in range(128)])


def _d_bits(blk):
    return int(blk[32]) | (int(blk[33]) << 8)


def test_double_to_half_matches_numpy():
    rng = np.random.default_rng(5)
    vals = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.uniform(-9, 5, 20000),
        [0.0, -0.0, 1.0, -1.0, 65504.0, 65519.999, 65520.0, 1e30, -1e30,
         2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0000001, 3 * 2.0 ** -26, 2.0 ** -14,
         2.0 ** -14 - 2.0 ** -25, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 2049.0, 2051.0]])
    for v in vals:
        with np.errstate(over="ignore"):
            want = int(np.array([v], dtype=np.float64).astype(np.float16).view(np.uint16)[0])
        assert oracle.double_to_half(v) == want, (v, hex(want))


def test_quantize_constant_block():
    # gamma = |a|; a exactly representable: w / d = +-1 -> codes 2 (positive), 0 (negative)
    for a in (1.0, 0.375, -2.5, 2.0 ** -10):
        blk = oracle.quantize(np.full((1, 128), a, np.float32), 1, 128)[0, 0]
        assert oracle.half_to_double(_d_bits(blk)) == abs(a)
        assert np.all(_codes(blk) == (2 if a > 0 else 0))


def test_quantize_alternating_and_spike():
    w = np.tile(np.array([0.75, -0.75], np.float32), 64).reshape(1, 128)
    blk = oracle.quantize(w, 1, 128)[0, 0]
    assert oracle.half_to_double(_d_bits(blk)) == 0.75
    assert np.array_equal(_codes(blk), np.tile([2, 0], 64))
    # a single spike: gamma = 3/128 (exact in binary16); the spike clips to +1, zeros stay 0
    w = np.zeros((1, 128), np.float32)
    w[0, 5] = 3.0
    blk = oracle.quantize(w, 1, 128)[0, 0]
    assert oracle.half_to_double(_d_bits(blk)) == 3.0 / 128
    want = np.ones(128, int)
    want[5] = 2
    assert np.array_equal(_codes(blk), want)


def test_quantize_ties_round_to_even():
    # 64 x 1.5 and 64 x 0.5: gamma = 1 exactly; rint(1.5) = 2 -> clipped to +1,
    # rint(0.5) = 0 (ties to even), rint(-0.5) = -0 -> code 1
    w = np.array([1.5] * 64 + [0.5] * 32 + [-0.5] * 32, np.float32).reshape(1, 128)
    blk = oracle.quantize(w, 1, 128)[0, 0]
    assert _d_bits(blk) == 0x3C00
    assert np.array_equal(_codes(blk), np.array([2] * 64 + [1] * 64))


def test_quantize_zero_and_huge_blocks():
    blk = oracle.quantize(np.zeros((1, 128), np.float32), 1, 128)[0, 0]
    assert _d_bits(blk) == 0 and np.all(_codes(blk) == 1)
    # gamma above the binary16 range: d = Inf, every code 1
    blk = oracle.quantize(np.full((1, 128), 1e6, np.float32), 1, 128)[0, 0]
    assert _d_bits(blk) == 0x7C00 and np.all(_codes(blk) == 1)


def test_quantize_scaling_and_layout():
    rng = np.random.default_rng(11)
    n, k = 3, 384
    w = rng.standard_normal((n, k)).astype(np.float32)
    a = oracle.quantize(w, n, k)
    b = oracle.quantize(w * np.float32(4.0), n, k)
    for r in range(n):
        for blk in range(k // 128):
            assert np.array_equal(_codes(a[r, blk]), _codes(b[r, blk]))
            assert oracle.half_to_double(_d_bits(b[r, blk])) == 4 * oracle.half_to_double(_d_bits(a[r, blk]))
            # each block is quantised on its own
            one = oracle.quantize(w[r:r + 1, blk * 128:(blk + 1) * 128], 1, 128)[0, 0]
            assert np.array_equal(one, a[r, blk])
    # reconstruction: |w - (c-1) d| <= d/2 where |w| <= 1.5 d, else the clip error |w| - d
    wd = oracle.dequant(a, n, k)
    for r in range(n):
        for blk in range(k // 128):
            d = oracle.half_to_double(_d_bits(a[r, blk]))
            seg = slice(blk * 128, (blk + 1) * 128)
            err = np.abs(w[r, seg].astype(np.float64) - wd[r, seg])
            bound = np.where(np.abs(w[r, seg]) <= 1.5 * d, 0.5 * d * (1 + 1e-6),
                             np.abs(w[r, seg]) - d + 1e-12)
            assert np.all(err <= bound)


def test_quantize_bad_k():
    with pytest.raises(ValueError):
        oracle.quantize(np.zeros((1, 100), np.float32), 1, 100)


# --------------------------------------------------------------------------
# gate/up SwiGLU

HALF_1 = 0x3C00  # 1.0


def _one_hot_block(pos, d_bits, code=2):
    """A block whose weight `pos` has code `code` and every other weight code 1 (zero)."""
    qs = np.full(32, 0x55, dtype=np.uint8)
    byte, shift = pos // 4, 2 * (pos % 4)
    qs[byte] = np.uint8(((int(qs[byte]) & ~(3 << shift)) & 0xFF) | (code << shift))
    return block(qs, d_bits)


def test_silu_closed_form_ln3():
    # sigmoid(ln 3) = 3/4
    z = np.log(3.0)
    assert abs(float(oracle.silu(z)) - 0.75 * z) < 1e-15
    assert abs(float(oracle.silu(-z)) - (-0.25 * z)) < 1e-15


def test_swiglu_hand_built_ln3():
    # f = 1, k = 128: gate row selects x[0] (d = 1), up row selects x[1] (d = 1)
    w = weight([_one_hot_block(0, HALF_1), _one_hot_block(1, HALF_1)], 2, 128)
    x = np.zeros((1, 128), dtype=np.float32)
    x[0, 0] = np.float32(np.log(3.0))
    x[0, 1] = 2.5
    h, g, u, _, _ = oracle.swiglu(w, x, f=1, k=128)
    assert g[0, 0] == float(np.float32(np.log(3.0))) and u[0, 0] == 2.5
    # silu(z) for z within 2^-24 relative of ln 3: 0.75 * ln 3 * 2.5 to ~1e-7
    assert abs(h[0, 0] - 0.75 * np.log(3.0) * 2.5) < 1e-7 * abs(h[0, 0])


def test_swiglu_odd_identity_pins_gate_and_up_roles():
    # flipping every gate code (c -> 2 - c) negates g exactly; since
    # silu(z) - silu(-z) = z, h(W) - h(W') = g * u.  Swapped gate/up roles or a
    # different activation break this.
    f, k = 24, 384
    p = tq2_synth.make_problem(3, 2 * f, k, seed=11)
    w = np.array(p.w_aos, copy=True).reshape(2 * f, k // 128, 34)
    w_flip = w.copy()
    qs = w_flip[:f, :, :32]
    c = np.stack([(qs >> (2 * t)) & 3 for t in range(4)], axis=-1)
    c = 2 - c
    w_flip[:f, :, :32] = (c[..., 0] | (c[..., 1] << 2) | (c[..., 2] << 4) | (c[..., 3] << 6)).astype(np.uint8)
    h, g, u, sg, su = oracle.swiglu(w, p.x, f=f, k=k)
    h2, g2, u2, _, _ = oracle.swiglu(w_flip, p.x, f=f, k=k)
    assert np.array_equal(g2, -g) and np.array_equal(u2, u)
    assert np.allclose(h - h2, g * u, rtol=1e-12, atol=1e-12 * np.max(np.abs(g * u)))


def test_swiglu_zero_rows_and_linearity_in_up():
    f, k = 8, 256
    p = tq2_synth.make_problem(2, 2 * f, k, seed=12)
    w = np.array(p.w_aos, copy=True).reshape(2 * f, k // 128, 34)
    z_up = w.copy()
    z_up[f:, :, :32] = 0x55
    assert np.array_equal(oracle.swiglu(z_up, p.x, f=f, k=k)[0], np.zeros((2, f)))
    z_gate = w.copy()
    z_gate[:f, :, :32] = 0x55
    assert np.array_equal(np.abs(oracle.swiglu(z_gate, p.x, f=f, k=k)[0]), np.zeros((2, f)))
    # doubling every up scale (exact in binary16) doubles h exactly
    dbl = w.copy()
    d = dbl[f:, :, 32].astype(np.uint16) | (dbl[f:, :, 33].astype(np.uint16) << 8)
    d2 = (d.view(np.float16).astype(np.float32) * 2).astype(np.float16).view(np.uint16)
    dbl[f:, :, 32] = (d2 & 0xFF).astype(np.uint8)
    dbl[f:, :, 33] = (d2 >> 8).astype(np.uint8)
    h = oracle.swiglu(w, p.x, f=f, k=k)[0]
    assert np.array_equal(oracle.swiglu(dbl, p.x, f=f, k=k)[0], 2 * h)


def test_swiglu_limits():
    # gate = +-40 (x = 40, d = 1): h = 40 u (sigmoid(40) = 1 - 4e-18) and |h| < 1e-15 |u|
    w = weight([_one_hot_block(0, HALF_1), _one_hot_block(1, HALF_1)], 2, 128)
    x = np.zeros((2, 128), dtype=np.float32)
    x[:, 1] = 3.0
    x[0, 0], x[1, 0] = 40.0, -40.0
    h = oracle.swiglu(w, x, f=1, k=128)[0]
    assert abs(h[0, 0] - 120.0) < 1e-12
    assert abs(h[1, 0]) < 1e-15 * 3.0


# --------------------------------------------------------------------------
# DiT joint attention


def test_attention_identical_keys_give_mean_of_v():
    rng = np.random.default_rng(3)
    h, n, d = 2, 7, 16
    q = rng.standard_normal((h, n, d))
    k = np.repeat(rng.standard_normal((h, 1, d)), n, axis=1)
    v = rng.standard_normal((h, n, d))
    out, _ = oracle.attention(q, k, v, heads=h, seq=n, dim=d)
    for hh in range(h):
        assert np.allclose(out[:, hh * d:(hh + 1) * d], v[hh].mean(axis=0)[None, :], rtol=0, atol=1e-14)


def test_attention_single_key_and_token_major_layout():
    rng = np.random.default_rng(4)
    h, d = 3, 8
    q, k, v = (rng.standard_normal((h, 1, d)) for _ in range(3))
    out, _ = oracle.attention(q, k, v, heads=h, seq=1, dim=d)
    assert np.array_equal(out[0], v[:, 0, :].reshape(-1))   # heads concatenated along features


def test_attention_two_keys_logistic():
    # dim 4, q = (a, 0, 0, 0), keys 0 and (b, 0, 0, 0): scores 0 and a b / 2, so
    # the weight of key 1 is the logistic 1 / (1 + exp(-a b / 2))
    a, b = 1.5, 0.8
    q = np.array([[[a, 0, 0, 0]]])
    k = np.array([[[0, 0, 0, 0], [b, 0, 0, 0]]], dtype=np.float64)
    v = np.array([[[1.0, 2.0, 3.0, 4.0], [-5.0, 0.5, 7.0, 1.0]]])
    q2 = np.concatenate([q, q], axis=1)  # two identical queries
    out, _ = oracle.attention(q2, k, v, heads=1, seq=2, dim=4)
    w1 = 1.0 / (1.0 + np.exp(-a * b / 2.0))
    ref = (1 - w1) * v[0, 0] + w1 * v[0, 1]
    assert np.allclose(out, ref[None, :], rtol=0, atol=1e-14)


def test_attention_dominant_key():
    rng = np.random.default_rng(5)
    h, n, d = 1, 6, 8
    q = np.zeros((h, n, d)); q[..., 0] = 1.0
    k = rng.standard_normal((h, n, d)) * 0.1
    k[0, 3, 0] = 200.0   # score 200/sqrt(8) above the rest: weight 1 - e^-70
    v = rng.standard_normal((h, n, d))
    out, _ = oracle.attention(q, k, v, heads=h, seq=n, dim=d)
    assert np.allclose(out, v[0, 3][None, :], rtol=0, atol=1e-12)


def test_attention_permutation_equivariance():
    rng = np.random.default_rng(6)
    h, n, d = 2, 9, 16
    q, k, v = (rng.standard_normal((h, n, d)) for _ in range(3))
    out, absv = oracle.attention(q, k, v, heads=h, seq=n, dim=d)
    pk = rng.permutation(n)
    out_k, _ = oracle.attention(q, k[:, pk], v[:, pk], heads=h, seq=n, dim=d)
    assert np.allclose(out_k, out, rtol=0, atol=1e-13)
    pq = rng.permutation(n)
    out_q, _ = oracle.attention(q[:, pq], k, v, heads=h, seq=n, dim=d)
    assert np.allclose(out_q, out[pq], rtol=0, atol=1e-13)
    assert np.all(absv >= np.abs(out) - 1e-13)
    sub, _ = oracle.attention(q, k, v, heads=h, seq=n, dim=d, rows=[4, 0])
    assert np.array_equal(sub, out[[4, 0]])
