"""Host-side tests of the C ABI (no GPU): the library loads, exports every
declared symbol, and rejects bad arguments before touching the device."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def tq2():
    import __graft_entry__
    __graft_entry__.build()
    import dit_tq2_g128_gb300 as m
    return m


def declared_functions():
    src = open(os.path.join(ROOT, "include", "tq2.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tq2_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(tq2):
    names = declared_functions()
    assert len(names) >= 11, names
    raw = ctypes.CDLL(tq2.LIB_PATH)
    for name in names:
        assert hasattr(raw, name), name
    assert sorted(tq2.EXPORTS) == names


def test_soa_bytes(tq2):
    assert tq2.tq2_soa_bytes(12288, 4096) == 13369344
    assert tq2.tq2_soa_bytes(4096, 12288) == 13369344
    assert tq2.tq2_soa_bytes(1, 128) == 34
    assert tq2.tq2_soa_bytes(0, 128) == 0
    for bad_k in (0, -128, 100, 129):
        assert tq2.tq2_soa_bytes(3, bad_k) == 0
    assert tq2.tq2_soa_bytes(-1, 128) == 0


def test_status_strings(tq2):
    for s in range(8):
        assert tq2.status_string(s).startswith("TQ2_")
    assert "unknown" in tq2.status_string(99)


def test_kernel_selection(tq2):
    assert tq2.tq2_select_kernel(1, 12288, 4096) == tq2.TQ2_KERNEL_GEMV
    assert tq2.tq2_select_kernel(1, 4096, 12288) == tq2.TQ2_KERNEL_GEMV
    assert tq2.tq2_select_kernel(1536, 3072, 3072) == tq2.TQ2_KERNEL_TC
    assert tq2.tq2_select_kernel(4096, 3072, 12288) == tq2.TQ2_KERNEL_TC
    for m in (2, 3, 7, 8, 9, 16, 32):
        assert tq2.tq2_select_kernel(m, 4096, 4096) == tq2.TQ2_KERNEL_SKINNY_MMA
        assert tq2.tq2_select_kernel(m, 1024, 1024) == tq2.TQ2_KERNEL_SKINNY_MMA
    for m in (33, 64, 100):
        assert tq2.tq2_select_kernel(m, 4096, 4096) == tq2.TQ2_KERNEL_TC
    # rows too long for the skinny kernel's K slices go to the tcgen05 kernel
    assert tq2.tq2_select_kernel(32, 4096, 1 << 17) == tq2.TQ2_KERNEL_TC


def rc_gemm(tq2, w, x, r, o, m, n, k, kernel=0):
    return tq2.lib.tq2_gemm_with(kernel, w, x, r, o, m, n, k, None)


def test_argument_errors_are_returned_before_any_launch(tq2):
    A = 1 << 20  # fake, 16-byte aligned, non-overlapping "device" addresses
    W, X, O, R = A, 64 * A, 128 * A, 192 * A
    # K must be a positive multiple of 128
    for k in (0, -128, 64, 130):
        assert rc_gemm(tq2, W, X, None, O, 4, 4, k) == tq2.TQ2_ERR_BAD_K
        assert tq2.lib.tq2_gemv(W, X, None, O, 4, k, None) == tq2.TQ2_ERR_BAD_K
        assert tq2.lib.tq2_gemv_resident(W, X, None, O, 4, k, None) == tq2.TQ2_ERR_BAD_K
        assert tq2.lib.tq2_reformat_aos_to_soa(W, O, 4, k, None) == tq2.TQ2_ERR_BAD_K
    # negative sizes
    assert rc_gemm(tq2, W, X, None, O, -1, 4, 128) == tq2.TQ2_ERR_INVALID_ARG
    assert rc_gemm(tq2, W, X, None, O, 4, -1, 128) == tq2.TQ2_ERR_INVALID_ARG
    assert tq2.lib.tq2_reformat_aos_to_soa(W, O, -1, 128, None) == tq2.TQ2_ERR_INVALID_ARG
    # size overflow
    assert rc_gemm(tq2, W, X, None, O, 1 << 40, 1 << 40, 128) == tq2.TQ2_ERR_INVALID_ARG
    # empty problems are no-ops even with null pointers
    assert rc_gemm(tq2, None, None, None, None, 0, 4, 128) == tq2.TQ2_OK
    assert rc_gemm(tq2, None, None, None, None, 4, 0, 128) == tq2.TQ2_OK
    assert tq2.lib.tq2_reformat_aos_to_soa(None, None, 0, 128, None) == tq2.TQ2_OK
    # null pointers
    assert rc_gemm(tq2, None, X, None, O, 4, 4, 128) == tq2.TQ2_ERR_INVALID_ARG
    assert rc_gemm(tq2, W, None, None, O, 4, 4, 128) == tq2.TQ2_ERR_INVALID_ARG
    assert rc_gemm(tq2, W, X, None, None, 4, 4, 128) == tq2.TQ2_ERR_INVALID_ARG
    assert tq2.lib.tq2_reformat_aos_to_soa(None, O, 4, 128, None) == tq2.TQ2_ERR_INVALID_ARG
    # misalignment
    assert rc_gemm(tq2, W + 4, X, None, O, 4, 4, 128) == tq2.TQ2_ERR_MISALIGNED
    assert rc_gemm(tq2, W, X + 8, None, O, 4, 4, 128) == tq2.TQ2_ERR_MISALIGNED
    assert rc_gemm(tq2, W, X, None, O + 4, 4, 4, 128) == tq2.TQ2_ERR_MISALIGNED
    assert rc_gemm(tq2, W, X, R + 4, O, 4, 4, 128) == tq2.TQ2_ERR_MISALIGNED
    assert tq2.lib.tq2_reformat_aos_to_soa(W + 1, O + 4, 4, 128, None) == tq2.TQ2_ERR_MISALIGNED
    # overlaps: out over x, out over w, partial residual overlap; exact alias is fine
    assert rc_gemm(tq2, W, X, None, X + 16, 4, 4, 128) == tq2.TQ2_ERR_INVALID_ARG
    assert rc_gemm(tq2, W, X, None, W, 4, 4, 128) == tq2.TQ2_ERR_INVALID_ARG
    assert rc_gemm(tq2, W, X, O + 16, O, 4, 4, 128) == tq2.TQ2_ERR_INVALID_ARG
    assert tq2.lib.tq2_reformat_aos_to_soa(W, W + 16, 4, 128, None) == tq2.TQ2_ERR_INVALID_ARG
    # kernel choice constraints
    assert rc_gemm(tq2, W, X, None, O, 2, 4, 128, tq2.TQ2_KERNEL_GEMV) == tq2.TQ2_ERR_INVALID_ARG
    assert rc_gemm(tq2, W, X, None, O, 17, 4, 128, tq2.TQ2_KERNEL_SKINNY) == tq2.TQ2_ERR_INVALID_ARG
    assert rc_gemm(tq2, W, X, None, O, 4, 4, 128, 9) == tq2.TQ2_ERR_INVALID_ARG
    assert rc_gemm(tq2, W, X, None, O, 4, 4, 128, 7) == tq2.TQ2_ERR_INVALID_ARG
    assert rc_gemm(tq2, W, X, None, O, 33, 4, 128, tq2.TQ2_KERNEL_SKINNY_MMA) == tq2.TQ2_ERR_INVALID_ARG
    assert rc_gemm(tq2, W, X, None, O, 1, 4, 128, tq2.TQ2_KERNEL_SKINNY_MMA) == tq2.TQ2_ERR_INVALID_ARG
    assert rc_gemm(tq2, W, X, None, O, 4, 4, 128, -1) == tq2.TQ2_ERR_INVALID_ARG


def test_workspace_size_and_errors(tq2):
    # binary16 copy of x padded to 128 rows, only for tensor-core shapes
    assert tq2.tq2_gemm_workspace_bytes(1536, 3072, 3072) == 1536 * 3072 * 2
    assert tq2.tq2_gemm_workspace_bytes(130, 64, 256) == 256 * 256 * 2
    assert tq2.tq2_gemm_workspace_bytes(1, 4096, 4096) == 0
    assert tq2.tq2_gemm_workspace_bytes(0, 4096, 4096) == 0
    assert tq2.tq2_gemm_workspace_bytes(64, 64, 100) == 0
    assert tq2.tq2_gemm_workspace_bytes(4096, 3072, 12288) == 4096 * 12288 * 2
    A = 1 << 20
    W, X, O, WS = A, 64 * A, 128 * A, 256 * A
    need = tq2.tq2_gemm_workspace_bytes(128, 256, 1024)
    f = tq2.lib.tq2_gemm_ws
    assert f(W, X, None, O, 128, 256, 1024, None, 0, None) == tq2.TQ2_ERR_INVALID_ARG
    assert f(W, X, None, O, 128, 256, 1024, WS, need - 1, None) == tq2.TQ2_ERR_INVALID_ARG
    assert f(W, X, None, O, 128, 256, 1024, WS + 16, need, None) == tq2.TQ2_ERR_MISALIGNED
    assert f(W, X, None, O, 128, 256, 1024, X, need, None) == tq2.TQ2_ERR_INVALID_ARG
    assert f(W, X, None, O, 128, 256, 1000, WS, need, None) == tq2.TQ2_ERR_BAD_K
    assert f(None, None, None, None, 0, 256, 1024, None, 0, None) == tq2.TQ2_OK


def test_python_wrapper_raises(tq2):
    with pytest.raises(tq2.TQ2Error) as e:
        tq2.tq2_gemm(1 << 20, 2 << 20, None, 3 << 20, 4, 4, 100)
    assert e.value.status == tq2.TQ2_ERR_BAD_K


def test_wait_timeout_setter_round_trips(tq2):
    old = tq2.tq2_set_wait_timeout_ns(12345)
    assert tq2.tq2_set_wait_timeout_ns(old) == 12345


def test_argument_errors_of_the_next_row_entry_points(tq2):
    # every check below returns before any device work (no GPU needed)
    A = 1 << 20  # fake, 16-byte aligned, non-overlapping "device" addresses
    W, X, O, R = A, 64 * A, 128 * A, 192 * A
    L = tq2.lib
    # encoder f32 -> blocks
    assert L.tq2_quantize_f32(X, O, 4, 100, None) == tq2.TQ2_ERR_BAD_K
    assert L.tq2_quantize_f32(X, O, -1, 128, None) == tq2.TQ2_ERR_INVALID_ARG
    assert L.tq2_quantize_f32(None, None, 0, 128, None) == tq2.TQ2_OK
    assert L.tq2_quantize_f32(None, O, 4, 128, None) == tq2.TQ2_ERR_INVALID_ARG
    assert L.tq2_quantize_f32(X + 4, O, 4, 128, None) == tq2.TQ2_ERR_MISALIGNED
    assert L.tq2_quantize_f32(X, X + 16, 4, 128, None) == tq2.TQ2_ERR_INVALID_ARG
    # fused gate/up + SwiGLU
    f = L.tq2_gate_up_swiglu
    assert f(W, X, O, 4, 8, 100, None) == tq2.TQ2_ERR_BAD_K
    assert f(W, X, O, -1, 8, 128, None) == tq2.TQ2_ERR_INVALID_ARG
    assert f(W, X, O, 4, -8, 128, None) == tq2.TQ2_ERR_INVALID_ARG
    assert f(None, None, None, 0, 8, 128, None) == tq2.TQ2_OK
    assert f(None, None, None, 4, 0, 128, None) == tq2.TQ2_OK
    assert f(None, X, O, 4, 8, 128, None) == tq2.TQ2_ERR_INVALID_ARG
    assert f(W, X, O + 4, 4, 8, 128, None) == tq2.TQ2_ERR_MISALIGNED
    assert f(W, X, X + 16, 4, 8, 128, None) == tq2.TQ2_ERR_INVALID_ARG
    assert f(W, X, W, 4, 8, 128, None) == tq2.TQ2_ERR_INVALID_ARG
    # binary16 activation GEMM and converters
    g = L.tq2_gemm_act16
    assert g(W, X, None, O, 4, 32, 100, None) == tq2.TQ2_ERR_BAD_K
    assert g(W, X, None, O, 4, 40, 128, None) == tq2.TQ2_ERR_INVALID_ARG   # n % 16
    assert g(None, None, None, None, 0, 32, 128, None) == tq2.TQ2_OK
    assert g(W, None, None, O, 4, 32, 128, None) == tq2.TQ2_ERR_INVALID_ARG
    assert g(W, X + 2, None, O, 4, 32, 128, None) == tq2.TQ2_ERR_MISALIGNED
    assert g(W, X, R + 2, O, 4, 32, 128, None) == tq2.TQ2_ERR_MISALIGNED
    assert g(W, X, None, X + 16, 4, 32, 128, None) == tq2.TQ2_ERR_INVALID_ARG
    assert g(W, X, O + 16, O, 4, 32, 128, None) == tq2.TQ2_ERR_INVALID_ARG  # partial residual overlap
    for conv in (L.tq2_act16_from_f32, L.tq2_act16_to_f32):
        assert conv(X, O, 4, 24, None) == tq2.TQ2_ERR_INVALID_ARG            # k % 16
        assert conv(X, O, -1, 32, None) == tq2.TQ2_ERR_INVALID_ARG
        assert conv(None, None, 0, 32, None) == tq2.TQ2_OK
        assert conv(None, O, 4, 32, None) == tq2.TQ2_ERR_INVALID_ARG
        assert conv(X + 8, O, 4, 32, None) == tq2.TQ2_ERR_MISALIGNED
        assert conv(X, X + 16, 4, 32, None) == tq2.TQ2_ERR_INVALID_ARG
    # DiT joint attention
    a = L.tq2_attention_f32
    for bad in (100, 4, 136):                                                  # dim not 8 * j <= 128
        assert a(X, R, W, O, 2, 128, bad, None) == tq2.TQ2_ERR_INVALID_ARG
    assert a(X, R, W, O, -1, 128, 128, None) == tq2.TQ2_ERR_INVALID_ARG
    assert a(X, R, W, O, 70000, 128, 128, None) == tq2.TQ2_ERR_INVALID_ARG   # heads > 65535
    assert a(None, None, None, None, 0, 128, 128, None) == tq2.TQ2_OK
    assert a(None, None, None, None, 2, 0, 128, None) == tq2.TQ2_OK
    assert a(None, R, W, O, 2, 128, 128, None) == tq2.TQ2_ERR_INVALID_ARG
    assert a(X, R + 4, W, O, 2, 128, 128, None) == tq2.TQ2_ERR_MISALIGNED
    assert a(X, R, W, X, 2, 128, 128, None) == tq2.TQ2_ERR_INVALID_ARG       # out over q
