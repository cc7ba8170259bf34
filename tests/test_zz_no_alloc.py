"""tq2_gemm_noalloc: the entry point for callers that cannot allocate device
memory.  It must give the same results as tq2_gemm_ws (which takes a
caller-provided workspace) without allocating anything, call after call: the
test also watches torch's allocator and the device's stream-ordered memory
pool around each call.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.  It passes on its own in a
fresh process as well as after the other tests.
"""

import ctypes

import numpy as np
import pytest

import oracle
import tq2_synth

TOL_TC = 4e-3


@pytest.fixture(scope="module")
def tq2():
    import __graft_entry__
    __graft_entry__.build()
    import dit_tq2_g128_gb300 as m
    return m


def test_noalloc_rejects_oversize_before_any_work(tq2):
    # ceil(4096/128)*128 * 12288 * 2 bytes = 96 MiB > the 32 MiB scratch
    A = 1 << 20
    rc = tq2.lib.tq2_gemm_noalloc(A, 1024 * A, None, 2048 * A, 4096, 3072, 12288, None)
    assert rc == tq2.TQ2_ERR_TOO_LARGE
    assert "TOO_LARGE" in tq2.status_string(rc)
    # shape errors keep their usual codes
    assert tq2.lib.tq2_gemm_noalloc(A, 2 * A, None, 3 * A, 8, 8, 100, None) == tq2.TQ2_ERR_BAD_K


def _default_pool_usage():
    """(reserved bytes, used high-water mark) of the device's default
    stream-ordered memory pool, the one cudaMallocAsync draws from, with the
    high-water mark reset to zero first; None where the CUDA runtime library
    cannot be loaded by path."""
    import os
    for path in ("/usr/local/cuda/lib64/libcudart.so", "libcudart.so.13", "libcudart.so"):
        try:
            rt = ctypes.CDLL(path)
            break
        except OSError:
            rt = None
    if rt is None:
        return None
    pool = ctypes.c_void_p()
    if rt.cudaDeviceGetDefaultMemPool(ctypes.byref(pool), 0) != 0:
        return None
    reserved_current, used_high = 5, 8  # cudaMemPoolAttr enumerators
    val = ctypes.c_uint64(0)
    rt.cudaMemPoolGetAttribute(pool, reserved_current, ctypes.byref(val))
    reserved = val.value
    rt.cudaMemPoolGetAttribute(pool, used_high, ctypes.byref(val))
    return rt, pool, reserved, val.value


def _reset_pool_high(state):
    rt, pool = state[0], state[1]
    zero = ctypes.c_uint64(0)
    rt.cudaMemPoolSetAttribute(pool, 8, ctypes.byref(zero))


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice(tq2):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA GPU visible")
    stream = torch.cuda.current_stream().cuda_stream
    # two calls in a row, different shapes and data (the second also exercises
    # the residual epilogue and a ragged tile)
    cases = [dict(m=1536, n=3072, k=3072, seed=0, residual=False),
             dict(m=300, n=700, k=1024, seed=1, residual=True)]
    for case in cases:
        p = tq2_synth.make_problem(case["m"], case["n"], case["k"], seed=case["seed"],
                                   residual=case["residual"], outlier_frac=0.01, d_sigma=0.01)
        assert tq2.tq2_select_kernel(p.m, p.n, p.k) == tq2.TQ2_KERNEL_TC
        w = tq2.upload_weight(p.w_aos, p.n, p.k)
        x = torch.from_numpy(p.x).cuda()
        r = None if p.residual is None else torch.from_numpy(p.residual).cuda()
        want = torch.full((p.m, p.n), float("nan"), device="cuda")
        ws = tq2.workspace(p.m, p.n, p.k)
        tq2.tq2_gemm_ws(w, x, r, want, p.m, p.n, p.k, ws, ws.numel())
        got = torch.full((p.m, p.n), float("nan"), device="cuda")
        torch.cuda.synchronize()
        # nothing may be allocated by the call: neither through torch's
        # allocator nor from the stream-ordered pool (used high-water mark
        # reset to zero just before)
        pool = _default_pool_usage()
        if pool is not None:
            _reset_pool_high(pool)
        torch_before = (torch.cuda.memory_allocated(), torch.cuda.memory_reserved())
        rc = tq2.lib.tq2_gemm_noalloc(w.data_ptr(), x.data_ptr(),
                                      None if r is None else r.data_ptr(), got.data_ptr(),
                                      p.m, p.n, p.k, ctypes.c_void_p(stream))
        assert rc == tq2.TQ2_OK, tq2.status_string(rc)
        torch.cuda.synchronize()
        assert (torch.cuda.memory_allocated(), torch.cuda.memory_reserved()) == torch_before
        if pool is not None:
            after = _default_pool_usage()
            assert after[3] == 0, "the call drew memory from the stream-ordered pool"
            assert after[2] == pool[2]
        assert tq2.tq2_device_status() == tq2.TQ2_OK
        g = got.cpu().numpy().astype(np.float64)
        e = want.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(g))
        rows = np.unique(np.linspace(0, p.m - 1, 24).astype(np.int64))
        _, scale = oracle.matmul(p.w_aos, p.x, p.residual, n=p.n, k=p.k, rows=rows)
        res = 0.0 if p.residual is None else np.abs(p.residual[rows].astype(np.float64))
        bound = TOL_TC * scale + 2.0 ** -23 * res + 1e-30
        assert np.all(np.abs(g[rows] - e[rows]) <= bound)
        # the kernels are the same, so in fact every element agrees exactly
        assert np.array_equal(g, e)
