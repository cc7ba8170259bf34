"""GPU parity: every CUDA entry point against the CPU oracle, through the C ABI.

Bars (per element, Sigma|xw| computed by the oracle in f64):
  * reformat and encoder: bit-exact;
  * f32 kernels (GEMV, small-M, f32ref): |out - ref| <= 1e-5 * Sigma|xw| + 2^-23 |residual|;
  * tensor-core kernel: |out - ref| <= 4e-3 * Sigma|xw| + 2^-23 |residual|, and the
    cosine between each output row and the oracle's row >= 0.9999.
Large problems run in full on the GPU and are checked on sampled rows (all N
columns of each sampled row) that the oracle computes one by one.
"""

import numpy as np
import pytest

import oracle
import tq2_synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL_F32 = 1e-5
TOL_TC = 4e-3
COS_MIN = 0.9999


@pytest.fixture(scope="module")
def tq2():
    import dit_tq2_g128_gb300 as m
    return m


def tol_for(tq2, kernel):
    tc = (tq2.TQ2_KERNEL_TC, tq2.TQ2_KERNEL_TC_DIRECT, tq2.TQ2_KERNEL_SKINNY_MMA)
    return TOL_TC if kernel in tc else TOL_F32


def upload(tq2, p):
    return tq2.upload_weight(p.w_aos, p.n, p.k)


def sample_rows(m, extra=12, seed=0):
    base = {0, 1, m - 1, m // 2}
    for r in (127, 128, 129, 255, 256, m - 128, m - 129):
        if 0 <= r < m:
            base.add(r)
    rng = np.random.default_rng(seed)
    base.update(rng.integers(0, m, size=min(extra, m)).tolist())
    return np.array(sorted(base), dtype=np.int64)


def check(out, p, kernel_tol, *, rows=None, cos=False, what=""):
    out = np.asarray(out, dtype=np.float64).reshape(-1, p.n)
    ref, scale = oracle.matmul(p.w_aos, p.x, p.residual, n=p.n, k=p.k, rows=rows)
    got = out if rows is None else out[rows]
    res = 0.0 if p.residual is None else np.abs(p.residual.reshape(-1, p.n)[
        slice(None) if rows is None else rows].astype(np.float64))
    bound = kernel_tol * scale + 2.0 ** -23 * res + 1e-30
    err = np.abs(got - ref)
    worst = float(np.max(err / bound)) if err.size else 0.0
    assert np.all(err <= bound), f"{what}: max err/bound {worst:.3g}"
    if cos:
        num = np.sum(got * ref, axis=1)
        den = np.linalg.norm(got, axis=1) * np.linalg.norm(ref, axis=1)
        c = np.where(den > 0, num / np.where(den > 0, den, 1), 1.0)
        assert np.all(c >= COS_MIN), f"{what}: min row cosine {c.min()}"
    return worst


def run(tq2, kernel, w, p, *, out=None, inplace=False):
    x = torch.from_numpy(p.x).cuda()
    r = None if p.residual is None else torch.from_numpy(p.residual).cuda()
    if inplace:
        out = r.clone()
        r = out
    elif out is None:
        out = torch.full((p.m, p.n), float("nan"), dtype=torch.float32, device="cuda")
    tq2.tq2_gemm_with(kernel, w, x, r, out, p.m, p.n, p.k)
    torch.cuda.synchronize()
    return out.cpu().numpy()


# ---------------------------------------------------------------------------
# AoS -> SoA


@pytest.mark.parametrize("n,k", [(1, 128), (3, 384), (17, 1024), (257, 256), (1000, 1152),
                                 (12288, 4096)])
@pytest.mark.parametrize("offset", [0, 1])
def test_reformat_bit_exact(tq2, n, k, offset):
    p = tq2_synth.make_problem(1, n, k, seed=n + k)
    nbytes = tq2.tq2_soa_bytes(n, k)
    raw = torch.zeros(nbytes + 64, dtype=torch.uint8, device="cuda")
    raw[offset:offset + nbytes] = torch.from_numpy(p.w_aos.reshape(-1)).cuda()
    soa = torch.full((nbytes + 32,), 0xA5, dtype=torch.uint8, device="cuda")
    tq2.tq2_reformat_aos_to_soa(raw[offset:].data_ptr(), soa, n, k)
    torch.cuda.synchronize()
    got = soa.cpu().numpy()
    assert np.array_equal(got[:nbytes], oracle.aos_to_soa(p.w_aos, n, k))
    assert np.all(got[nbytes:] == 0xA5)  # nothing written past the end


# ---------------------------------------------------------------------------
# M = 1 decode GEMV


def test_gemv_gate_up_full(tq2):
    p = tq2_synth.decode_gate_up()
    w = upload(tq2, p)
    x = torch.from_numpy(p.x[0]).cuda()
    out = torch.full((p.n,), float("nan"), device="cuda")
    tq2.tq2_gemv(w, x, None, out, p.n, p.k)
    torch.cuda.synchronize()
    check(out.cpu().numpy(), p, TOL_F32, what="gemv gate/up")


def test_gemv_down_residual_full(tq2):
    p = tq2_synth.decode_down()
    w = upload(tq2, p)
    x = torch.from_numpy(p.x[0]).cuda()
    r = torch.from_numpy(p.residual[0]).cuda()
    out = torch.full((p.n,), float("nan"), device="cuda")
    tq2.tq2_gemv(w, x, r, out, p.n, p.k)
    torch.cuda.synchronize()
    check(out.cpu().numpy(), p, TOL_F32, what="gemv down+res")
    # in place: residual and out are the same buffer
    tq2.tq2_gemv(w, x, r, r, p.n, p.k)
    torch.cuda.synchronize()
    check(r.cpu().numpy(), p, TOL_F32, what="gemv in-place")


@pytest.mark.parametrize("n,k", [(1, 128), (129, 128), (7, 1152), (300, 3072), (33, 20480),
                                 (5, 65536), (30400, 4096), (250000, 512), (2000, 16384),
                                 # 64-weight lanes: one to four 2048-weight chunks
                                 (1, 2048), (77, 2048), (3, 6144), (1000, 8192), (153, 4096)])
def test_gemv_edge_shapes(tq2, n, k):
    p = tq2_synth.make_problem(1, n, k, seed=n * 7 + k, residual=(n % 2 == 1))
    w = upload(tq2, p)
    check(run(tq2, tq2.TQ2_KERNEL_GEMV, w, p), p, TOL_F32, what=f"gemv n={n} k={k}")


@pytest.mark.parametrize("n,k", [(12288, 4096), (4096, 12288), (153, 4096), (1, 2048), (3, 6144),
                                 (7, 1152), (33, 20480), (30400, 4096)])
def test_gemv_resident_equals_gemv_bit_for_bit(tq2, n, k):
    # the resident-weights entry only moves the weight copies before the
    # dependency wait: the same arithmetic, so the same bits as tq2_gemv
    p = tq2_synth.make_problem(1, n, k, seed=n * 3 + k, residual=(n % 2 == 0))
    w = upload(tq2, p)
    torch.cuda.synchronize()  # the contract: the weights are complete before the call
    x = torch.from_numpy(p.x[0]).cuda()
    r = None if p.residual is None else torch.from_numpy(p.residual[0]).cuda()
    a = torch.full((n,), float("nan"), device="cuda")
    b = torch.full((n,), float("nan"), device="cuda")
    tq2.tq2_gemv(w, x, r, a, n, k)
    tq2.tq2_gemv_resident(w, x, r, b, n, k)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    check(b.cpu().numpy(), p, TOL_F32, what=f"gemv resident n={n} k={k}")


@pytest.mark.parametrize("k", [4096, 3072])
def test_gemv_resident_chain_reads_x_after_the_previous_call(tq2, k):
    # a chain of dependent calls with no synchronisation in between: call i+1
    # reads the x that call i writes (and adds the residual call i-1 wrote), so
    # reading x or the residual before the dependency wait would show up as a
    # difference from the same chain through tq2_gemv
    n = k
    ws = []
    for i in range(3):
        p = tq2_synth.make_problem(1, n, k, seed=500 + i + k)
        ws.append(upload(tq2, p))
    torch.cuda.synchronize()
    x0 = torch.from_numpy(tq2_synth.make_problem(1, n, k, seed=600 + k).x[0]).cuda()

    def chain(fn):
        bufs = [x0.clone()] + [torch.full((n,), float("nan"), device="cuda") for _ in range(12)]
        for i in range(12):
            res = bufs[i - 1] if i >= 1 else None
            fn(ws[i % 3], bufs[i], res, bufs[i + 1], n, k)
        torch.cuda.synchronize()
        return torch.stack(bufs[1:])

    a = chain(tq2.tq2_gemv)
    b = chain(tq2.tq2_gemv_resident)
    assert torch.isfinite(a).all()
    assert torch.equal(a, b)


def test_gemv_quantisation_bound_with_wide_dynamic_range(tq2):
    # one huge activation per 64 elements next to tiny ones: the GEMV's
    # documented bound (2^-22 * max|x_block| * sum_block |w| per 128-weight
    # block, the granularity of its x scale) must hold, and so must the
    # contract's 1e-5 * sum|x w|
    n, k = 512, 4096
    p = tq2_synth.make_problem(1, n, k, seed=17)
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(k) * 1e-3).astype(np.float32)
    x[::64] = 1e3 * np.sign(rng.standard_normal(k // 64)).astype(np.float32)
    p.x = x[None, :]
    w = upload(tq2, p)
    out = run(tq2, tq2.TQ2_KERNEL_GEMV, w, p)[0].astype(np.float64)
    ref, scale = oracle.matmul(p.w_aos, p.x, n=n, k=k)
    W = np.abs(oracle.dequant(p.w_aos, n, k))
    smax = np.abs(x.astype(np.float64)).reshape(-1, 128).max(axis=1)
    bound = (W.reshape(n, -1, 128).sum(axis=2) * smax[None, :]).sum(axis=1) * 2.0 ** -22
    bound += 1e-6 * scale[0]
    assert np.all(np.abs(out - ref[0]) <= bound)
    assert np.all(np.abs(out - ref[0]) <= TOL_F32 * scale[0])


# ---------------------------------------------------------------------------
# all kernels on the small configuration and on ragged shapes

KERNELS = ["TQ2_KERNEL_TC", "TQ2_KERNEL_TC_DIRECT", "TQ2_KERNEL_F32REF", "TQ2_KERNEL_SKINNY",
           "TQ2_KERNEL_SKINNY_MMA"]


@pytest.mark.parametrize("kname", KERNELS)
@pytest.mark.parametrize("residual", [False, True])
def test_small_config_each_kernel(tq2, kname, residual):
    p = tq2_synth.make_problem(8, 1024, 1024, seed=0, residual=residual)
    w = upload(tq2, p)
    kernel = getattr(tq2, kname)
    check(run(tq2, kernel, w, p), p, tol_for(tq2, kernel), cos=tol_for(tq2, kernel) == TOL_TC,
          what=kname)


@pytest.mark.parametrize("m,n,k", [(1, 1, 128), (2, 129, 256), (3, 7, 128), (17, 257, 384),
                                   (129, 300, 640), (130, 255, 128), (5, 1000, 1024),
                                   (256, 512, 256), (200, 33, 1280)])
@pytest.mark.parametrize("kname", KERNELS + ["TQ2_KERNEL_AUTO"])
def test_ragged_shapes(tq2, m, n, k, kname):
    kernel = getattr(tq2, kname)
    if kernel == tq2.TQ2_KERNEL_SKINNY and m > 16:
        pytest.skip("small-M kernel is limited to M <= 16")
    if kernel == tq2.TQ2_KERNEL_SKINNY_MMA and not 2 <= m <= 32:
        pytest.skip("skinny tensor-core kernel is limited to 2 <= M <= 32")
    p = tq2_synth.make_problem(m, n, k, seed=m * 1000 + n + k, residual=(m + n) % 2 == 0,
                               outlier_frac=0.01)
    w = upload(tq2, p)
    eff = tq2.tq2_select_kernel(m, n, k) if kernel == tq2.TQ2_KERNEL_AUTO else kernel
    out = run(tq2, kernel, w, p)
    check(out, p, tol_for(tq2, eff), cos=(tol_for(tq2, eff) == TOL_TC and n >= 16),
          what=f"{kname} {m}x{n}x{k}")


@pytest.mark.parametrize("kname", KERNELS)
def test_inplace_residual(tq2, kname):
    kernel = getattr(tq2, kname)
    p = tq2_synth.make_problem(9, 300, 512, seed=5, residual=True)
    w = upload(tq2, p)
    check(run(tq2, kernel, w, p, inplace=True), p, tol_for(tq2, kernel), what=f"{kname} in-place")


def test_code3_decodes_to_plus_two_everywhere(tq2):
    # code 3 is never generated; every kernel still decodes it as c - 1 = +2
    m, n, k = 4, 64, 256
    p = tq2_synth.make_problem(m, n, k, seed=3)
    p.w_aos[:, :, :32] = 0xFF
    w = upload(tq2, p)
    for kernel in (tq2.TQ2_KERNEL_TC, tq2.TQ2_KERNEL_TC_DIRECT, tq2.TQ2_KERNEL_F32REF,
                   tq2.TQ2_KERNEL_SKINNY, tq2.TQ2_KERNEL_SKINNY_MMA):
        check(run(tq2, kernel, w, p), p, tol_for(tq2, kernel), what=f"code3 {kernel}")
    p1 = tq2_synth.make_problem(1, n, k, seed=3)
    p1.w_aos[:] = p.w_aos
    check(run(tq2, tq2.TQ2_KERNEL_GEMV, w, p1), p1, TOL_F32, what="code3 gemv")


def test_zero_weights_give_residual(tq2):
    m, n, k = 130, 260, 384
    p = tq2_synth.make_problem(m, n, k, seed=9, residual=True)
    p.w_aos[:, :, :32] = 0x55
    w = upload(tq2, p)
    for kernel in (tq2.TQ2_KERNEL_TC, tq2.TQ2_KERNEL_TC_DIRECT, tq2.TQ2_KERNEL_F32REF):
        out = run(tq2, kernel, w, p)
        assert np.array_equal(out, p.residual), kernel


def test_empty_problems_are_noops(tq2):
    w = torch.zeros(34, dtype=torch.uint8, device="cuda")
    x = torch.zeros(128, device="cuda")
    out = torch.full((4,), 7.0, device="cuda")
    for kernel in (0, 1, 2, 3, 4, 5):
        tq2.tq2_gemm_with(kernel, w, x, None, out, 0, 1, 128)
        tq2.tq2_gemm_with(kernel, w, x, None, out, 1, 0, 128)
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)


# ---------------------------------------------------------------------------
# the benchmark configurations


@pytest.mark.parametrize("m", tq2_synth.SKINNY_MS)
def test_skinny_sweep_auto(tq2, m):
    p = tq2_synth.skinny(m)
    w = upload(tq2, p)
    kernel = tq2.tq2_select_kernel(m, p.n, p.k)
    out = run(tq2, tq2.TQ2_KERNEL_AUTO, w, p)
    check(out, p, tol_for(tq2, kernel), cos=tol_for(tq2, kernel) == TOL_TC, what=f"skinny m={m}")


@pytest.mark.parametrize("m", [2, 3, 7, 8, 9, 15, 16, 17, 24, 31, 32])
@pytest.mark.parametrize("n,k,res", [(4096, 4096, False), (1000, 1152, True), (12288, 4096, False),
                                     (300, 12288, True)])
def test_skinny_mma(tq2, m, n, k, res):
    p = tq2_synth.make_problem(m, n, k, seed=31 * m + n, residual=res, outlier_frac=0.01)
    w = upload(tq2, p)
    assert tq2.tq2_select_kernel(m, n, k) == tq2.TQ2_KERNEL_SKINNY_MMA
    a = run(tq2, tq2.TQ2_KERNEL_SKINNY_MMA, w, p)
    check(a, p, TOL_TC, cos=True, what=f"skinny mma {m}x{n}x{k}")
    b = run(tq2, tq2.TQ2_KERNEL_SKINNY_MMA, w, p)
    assert np.array_equal(a, b)  # same bits on every call (fixed reduction order)


@pytest.mark.parametrize("m", [7, 8, 9, 16])
def test_skinny_sweep_tc(tq2, m):
    p = tq2_synth.skinny(m)
    w = upload(tq2, p)
    check(run(tq2, tq2.TQ2_KERNEL_TC, w, p), p, TOL_TC, cos=True, what=f"tc m={m}")


def test_dit_large_m_tc_direct(tq2):
    p = tq2_synth.dit(3072)
    w = upload(tq2, p)
    out = run(tq2, tq2.TQ2_KERNEL_TC_DIRECT, w, p)
    check(out, p, TOL_TC, rows=sample_rows(p.m), cos=True, what="dit n=3072 tc_direct")


def test_dit_large_m_f32ref(tq2):
    p = tq2_synth.dit(3072)
    w = upload(tq2, p)
    check(run(tq2, tq2.TQ2_KERNEL_F32REF, w, p), p, TOL_F32, rows=sample_rows(p.m, extra=6),
          what="f32ref dit")


# ---------------------------------------------------------------------------
# tensor-core kernel fed from the workspace (tq2_gemm_ws)


def run_ws(tq2, w, p, *, inplace=False):
    x = torch.from_numpy(p.x).cuda()
    r = None if p.residual is None else torch.from_numpy(p.residual).cuda()
    out = r.clone() if inplace else torch.full((p.m, p.n), float("nan"), device="cuda")
    if inplace:
        r = out
    ws = tq2.workspace(p.m, p.n, p.k)
    nbytes = 0 if ws is None else ws.numel()
    tq2.tq2_gemm_ws(w, x, r, out, p.m, p.n, p.k, ws, nbytes)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("m,n,k", [(8, 1024, 1024), (4, 7, 128), (17, 257, 384), (129, 300, 640),
                                   (130, 255, 128), (256, 512, 256), (200, 33, 1280),
                                   (300, 700, 4096), (5, 1000, 1152)])
@pytest.mark.parametrize("residual", [False, True])
def test_ws_ragged(tq2, m, n, k, residual):
    p = tq2_synth.make_problem(m, n, k, seed=m + n + k, residual=residual, outlier_frac=0.01)
    w = upload(tq2, p)
    eff = tq2.tq2_select_kernel(m, n, k)
    check(run_ws(tq2, w, p), p, tol_for(tq2, eff), cos=(tol_for(tq2, eff) == TOL_TC and n >= 16),
          what=f"ws {m}x{n}x{k}")


def test_ws_inplace_and_repeat(tq2):
    p = tq2_synth.make_problem(260, 520, 768, seed=7, residual=True)
    w = upload(tq2, p)
    a = run_ws(tq2, w, p, inplace=True)
    check(a, p, TOL_TC, cos=True, what="ws in-place")
    b = run_ws(tq2, w, p, inplace=True)
    assert np.array_equal(a, b)  # deterministic


@pytest.mark.parametrize("m,n,k", [(300, 100, 640), (129, 36, 128), (513, 1028, 256), (77, 4, 384)])
def test_ws_inplace_ragged(tq2, m, n, k):
    # in-place residual with a 16-byte row pitch: the reduce-add epilogue,
    # including boxes clipped at the M and N edges
    p = tq2_synth.make_problem(m, n, k, seed=3 * m + n, residual=True)
    w = upload(tq2, p)
    eff = tq2.tq2_select_kernel(m, n, k)
    check(run_ws(tq2, w, p, inplace=True), p, tol_for(tq2, eff),
          cos=(tol_for(tq2, eff) == TOL_TC and n >= 16), what=f"ws in-place {m}x{n}x{k}")


@pytest.mark.parametrize("n", tq2_synth.DIT_NS)
def test_ws_dit_large_m(tq2, n):
    p = tq2_synth.dit(n)
    w = upload(tq2, p)
    check(run_ws(tq2, w, p), p, TOL_TC, rows=sample_rows(p.m), cos=True, what=f"ws dit n={n}")


@pytest.mark.parametrize("layer", [0, 41, 60, 81])
def test_ws_dit_forward_layers(tq2, layer):
    p = tq2_synth.dit_forward_layer(layer)
    w = upload(tq2, p)
    check(run_ws(tq2, w, p), p, TOL_TC, rows=sample_rows(p.m, extra=4, seed=layer), cos=True,
          what=f"ws dit forward layer {layer}")


@pytest.mark.parametrize("m", [7, 8, 9, 16, 64, 100])
def test_ws_skinny(tq2, m):
    p = tq2_synth.skinny(m)
    w = upload(tq2, p)
    check(run_ws(tq2, w, p), p, TOL_TC, cos=True, what=f"ws skinny m={m}")


# ---------------------------------------------------------------------------
# bounded device waits


@pytest.mark.parametrize("kname", ["TQ2_KERNEL_TC", "TQ2_KERNEL_TC_DIRECT"])
def test_wait_timeout_is_reported_and_context_survives(tq2, kname):
    kernel = getattr(tq2, kname)
    p = tq2_synth.make_problem(128, 256, 2048, seed=1)
    w = upload(tq2, p)
    assert tq2.tq2_device_status() == tq2.TQ2_OK
    old = tq2.tq2_set_wait_timeout_ns(0)
    try:
        run(tq2, kernel, w, p)
        st = tq2.tq2_device_status()
    finally:
        tq2.tq2_set_wait_timeout_ns(old)
    assert st == tq2.TQ2_ERR_TIMEOUT
    assert tq2.tq2_device_status() == tq2.TQ2_OK  # cleared by the read
    check(run(tq2, kernel, w, p), p, TOL_TC, cos=True, what="after timeout")
    assert tq2.tq2_device_status() == tq2.TQ2_OK


def test_wait_timeout_ws_kernel(tq2):
    p = tq2_synth.make_problem(256, 512, 2048, seed=2)
    w = upload(tq2, p)
    assert tq2.tq2_device_status() == tq2.TQ2_OK
    old = tq2.tq2_set_wait_timeout_ns(0)
    try:
        run_ws(tq2, w, p)
        st = tq2.tq2_device_status()
    finally:
        tq2.tq2_set_wait_timeout_ns(old)
    assert st == tq2.TQ2_ERR_TIMEOUT
    check(run_ws(tq2, w, p), p, TOL_TC, cos=True, what="ws after timeout")
    assert tq2.tq2_device_status() == tq2.TQ2_OK


# ---------------------------------------------------------------------------
# encoder (f32 -> blocks): bit-exact against the oracle


def _encode(tq2, w, n, k):
    wd = torch.from_numpy(np.ascontiguousarray(w, dtype=np.float32)).cuda()
    out = torch.full((tq2.tq2_soa_bytes(n, k),), 0xAB, dtype=torch.uint8, device="cuda")
    tq2.tq2_quantize_f32(wd, out, n, k)
    torch.cuda.synchronize()
    return out.cpu().numpy().reshape(n, k // 128, 34)


@pytest.mark.parametrize("n,k,dist", [(1, 128, "normal"), (7, 384, "normal"), (33, 1024, "uniform"),
                                      (256, 4096, "normal"), (1000, 128, "mixed"),
                                      (64, 2048, "heavy"), (3, 12288, "normal")])
def test_quantize_bit_exact(tq2, n, k, dist):
    rng = np.random.default_rng(7 * n + k)
    if dist == "normal":
        w = rng.standard_normal((n, k)) * 0.02
    elif dist == "uniform":
        w = rng.uniform(-1.0, 1.0, (n, k))
    elif dist == "heavy":
        w = rng.standard_cauchy((n, k))
    else:  # zeros, tiny and large blocks side by side
        w = rng.standard_normal((n, k))
        w[::3] = 0.0
        w[1::7] *= 1e-7
        w[2::11] *= 3e4
    w = w.astype(np.float32)
    assert np.array_equal(_encode(tq2, w, n, k), oracle.quantize(w, n, k))


def test_quantize_special_blocks(tq2):
    blocks = [np.zeros(128), np.full(128, 1e6), np.array([1.5] * 64 + [0.5] * 32 + [-0.5] * 32),
              np.full(128, 3e-8), np.array([-0.0] * 128), np.tile([0.75, -0.75], 64),
              np.r_[np.full(1, 3.0), np.zeros(127)], np.linspace(-2.0, 2.0, 128)]
    w = np.stack(blocks).astype(np.float32).reshape(1, -1)
    n, k = 1, w.size
    assert np.array_equal(_encode(tq2, w, n, k), oracle.quantize(w, n, k))


def test_quantize_exponent_spans(tq2):
    # blocks around the exact-integer route's limit (magnitudes spanning 22
    # binades are summed as integers, 23 and more in double in index order),
    # subnormals next to normals, and block means at the binary16 overflow edge
    rng = np.random.default_rng(3)
    blocks = []
    for span in (0, 1, 21, 22, 23, 24, 40, 100):
        b = rng.uniform(1.0, 2.0, 128) * np.where(rng.random(128) < 0.5, -1.0, 1.0)
        b[rng.integers(0, 128, 3)] *= 2.0 ** -span
        blocks.append(b)
    blocks.append(np.r_[np.full(64, 1e-40), np.full(64, 1e-38)])          # subnormal + normal
    blocks.append(np.r_[np.full(127, 1.4e-45), np.full(1, 1.0)])          # smallest subnormal
    blocks.append(np.full(128, 65504.0))                                  # d = 65504
    blocks.append(np.full(128, 65519.0))                                  # rounds down to 65504
    blocks.append(np.full(128, 65520.0))                                  # rounds up to Inf: codes 1
    blocks.append(np.full(128, 2.0 ** -25))                               # d below the half grid
    blocks.append(np.full(128, 3.0 * 2.0 ** -26))                         # d rounds to the grid
    for _ in range(24):
        blocks.append(rng.standard_normal(128) * np.exp2(rng.uniform(-30, 30, 128)))
    w = np.stack(blocks).astype(np.float32).reshape(1, -1)
    n, k = 1, w.size
    assert np.array_equal(_encode(tq2, w, n, k), oracle.quantize(w, n, k))


def test_quantize_then_matmul(tq2):
    rng = np.random.default_rng(21)
    m, n, k = 64, 300, 1024
    w = (rng.standard_normal((n, k)) * 0.05).astype(np.float32)
    aos = _encode(tq2, w, n, k)
    p = tq2_synth.make_problem(m, n, k, seed=4)
    p.w_aos[:] = aos
    check(run(tq2, tq2.TQ2_KERNEL_AUTO, upload(tq2, p), p), p, TOL_TC, cos=True, what="encode + gemm")


def test_quantize_empty_and_errors(tq2):
    w = torch.zeros((2, 256), device="cuda")
    out = torch.zeros(tq2.tq2_soa_bytes(2, 256), dtype=torch.uint8, device="cuda")
    tq2.tq2_quantize_f32(w, out, 0, 256)  # no-op
    with pytest.raises(tq2.TQ2Error):
        tq2.tq2_quantize_f32(w, out, 2, 100)
    with pytest.raises(tq2.TQ2Error):
        tq2.tq2_quantize_f32(w, out.data_ptr() + 1, 2, 256)


# ---------------------------------------------------------------------------
# fused gate/up + SwiGLU

def run_swiglu(tq2, w, p, f):
    x = torch.from_numpy(p.x).cuda()
    out = torch.full((p.m, f), float("nan"), dtype=torch.float32, device="cuda")
    tq2.tq2_gate_up_swiglu(w, x, out, p.m, f, p.k)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def check_swiglu(got, p, f, rel, *, rows=None, cos=False, what=""):
    """|h - ref| <= 1.1 tg (|u| + tu) + |silu(g)| tu + 2^-22 |h|: the products'
    bound rel * Sigma|xw| (tg, tu) carried through silu (|silu'| <= 1.1) and
    the product, plus f32 rounding of the activation."""
    h, g, u, sg, su = oracle.swiglu(p.w_aos, p.x, f=f, k=p.k, rows=rows)
    got = np.asarray(got, dtype=np.float64).reshape(-1, f)
    got = got if rows is None else got[rows]
    tg, tu = rel * sg, rel * su
    bound = 1.1 * tg * (np.abs(u) + tu) + np.abs(oracle.silu(g)) * tu + 2.0 ** -22 * np.abs(h) + 1e-30
    err = np.abs(got - h)
    worst = float(np.max(err / bound)) if err.size else 0.0
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert np.all(err <= bound), f"{what}: max err/bound {worst:.3g}"
    if cos:
        num = np.sum(got * h, axis=1)
        den = np.linalg.norm(got, axis=1) * np.linalg.norm(h, axis=1)
        c = np.where(den > 0, num / np.where(den > 0, den, 1), 1.0)
        assert np.all(c >= COS_MIN), f"{what}: min row cosine {c.min()}"
    return worst


@pytest.mark.parametrize("f,k", [(6144, 4096), (1, 128), (7, 1152), (100, 3072), (2048, 12288),
                                 (33, 16384),
                                 # 64-weight lanes; odd feature counts put a stage across the
                                 # gate / up boundary of a CTA's rows
                                 (7, 2048), (153, 4096), (1001, 8192)])
def test_swiglu_decode(tq2, f, k):
    # m = 1: fused into the GEMV for k <= 12288 (the 6144 x 4096 case is the
    # decode fused gate/up shape, 2f = 12288 rows); k = 16384 takes the
    # unfused path (exact-f32 product, then the activation)
    p = tq2_synth.make_problem(1, 2 * f, k, seed=f + k, code_probs=(0.3, 0.4, 0.3))
    w = upload(tq2, p)
    check_swiglu(run_swiglu(tq2, w, p, f), p, f, TOL_F32, what=f"swiglu m=1 f={f} k={k}")


@pytest.mark.parametrize("m,f,k", [(1, 6144, 4096), (1, 7, 2048), (1, 153, 4096), (1, 100, 3072),
                                   (1, 33, 16384), (2, 64, 256), (8, 100, 384)])
def test_swiglu_resident_equals_swiglu_bit_for_bit(tq2, m, f, k):
    # resident weights change only when the weight copies are issued (m = 1,
    # 64-weight lanes); every other shape runs the same code as tq2_gate_up_swiglu
    p = tq2_synth.make_problem(m, 2 * f, k, seed=m * 13 + f + k)
    w = upload(tq2, p)
    torch.cuda.synchronize()
    x = torch.from_numpy(p.x).cuda()
    a = torch.full((m, f), float("nan"), device="cuda")
    b = torch.full((m, f), float("nan"), device="cuda")
    tq2.tq2_gate_up_swiglu(w, x, a, m, f, k)
    tq2.tq2_gate_up_swiglu_resident(w, x, b, m, f, k)
    torch.cuda.synchronize()
    assert torch.isfinite(a).all()
    assert torch.equal(a, b)


@pytest.mark.parametrize("m,f,k", [(8, 512, 1024), (2, 64, 256), (129, 48, 640), (300, 1024, 3072),
                                   (64, 6144, 4096), (5, 40, 384), (20, 1000, 1152), (3, 7, 128)])
def test_swiglu_batched(tq2, m, f, k):
    # m >= 2: the tensor-core kernel with the activation in its epilogue when
    # f % 16 == 0 (40, 1000 and 7 take the unfused path)
    p = tq2_synth.make_problem(m, 2 * f, k, seed=m * 31 + f)
    w = upload(tq2, p)
    check_swiglu(run_swiglu(tq2, w, p, f), p, f, TOL_TC, cos=True, what=f"swiglu m={m} f={f} k={k}")


def test_swiglu_dit_shape_sampled(tq2):
    # prefill-sized: m = 1536, 2f = 12288 rows, k = 3072; sampled rows
    m, f, k = 1536, 6144, 3072
    p = tq2_synth.make_problem(m, 2 * f, k, seed=77, d_sigma=0.01, outlier_frac=0.01)
    w = upload(tq2, p)
    got = run_swiglu(tq2, w, p, f)
    check_swiglu(got, p, f, TOL_TC, rows=sample_rows(m), cos=True, what="swiglu dit shape")


def test_swiglu_empty_and_errors(tq2):
    x = torch.zeros(4, 128, device="cuda")
    out = torch.zeros(4, 8, device="cuda")
    w = torch.zeros(int(tq2.tq2_soa_bytes(16, 128)), dtype=torch.uint8, device="cuda")
    assert tq2.lib.tq2_gate_up_swiglu(w.data_ptr(), x.data_ptr(), out.data_ptr(), 0, 8, 128, None) == tq2.TQ2_OK
    assert tq2.lib.tq2_gate_up_swiglu(w.data_ptr(), x.data_ptr(), out.data_ptr(), 4, 0, 128, None) == tq2.TQ2_OK
    assert tq2.lib.tq2_gate_up_swiglu(w.data_ptr(), x.data_ptr(), out.data_ptr(), 4, 8, 100, None) == tq2.TQ2_ERR_BAD_K
    assert tq2.lib.tq2_gate_up_swiglu(w.data_ptr(), x.data_ptr(), out.data_ptr(), -1, 8, 128, None) == tq2.TQ2_ERR_INVALID_ARG
    assert tq2.lib.tq2_gate_up_swiglu(w.data_ptr(), x.data_ptr() + 4, out.data_ptr(), 4, 8, 128, None) == tq2.TQ2_ERR_MISALIGNED
    assert tq2.lib.tq2_gate_up_swiglu(None, x.data_ptr(), out.data_ptr(), 4, 8, 128, None) == tq2.TQ2_ERR_INVALID_ARG
    # out overlapping x
    assert tq2.lib.tq2_gate_up_swiglu(w.data_ptr(), x.data_ptr(), x.data_ptr(), 4, 8, 128, None) == tq2.TQ2_ERR_INVALID_ARG
    torch.cuda.synchronize()


# ---------------------------------------------------------------------------
# binary16 activation layout and the activation-resident GEMM

def act16_perm(k):
    """Storage position of each element: element 16g + i at 16g + (2i if i < 8 else 2(i-8)+1)."""
    i = np.arange(k) % 16
    return (np.arange(k) - i) + np.where(i < 8, 2 * i, 2 * (i - 8) + 1)


def to_act16(x):
    """numpy reference of the layout: float16 (round to nearest even), elements permuted."""
    with np.errstate(over="ignore"):
        x16 = np.asarray(x, dtype=np.float32).astype(np.float16)
    out = np.empty_like(x16)
    out[:, act16_perm(x.shape[1])] = x16
    return out


def from_act16(y):
    return y[:, act16_perm(y.shape[1])]


@pytest.mark.parametrize("m,k", [(1, 16), (3, 48), (129, 1024), (7, 4096)])
def test_act16_converters_bit_exact(tq2, m, k):
    rng = np.random.default_rng(m + k)
    x = (rng.standard_normal((m, k)) * rng.choice([1e-6, 1.0, 300.0], size=(m, k))).astype(np.float32)
    x[0, 0] = 65519.0   # rounds to 65504
    if k > 1:
        x[0, 1] = 65520.0  # rounds to Inf
    xd = torch.from_numpy(x).cuda()
    y = torch.empty((m, k), dtype=torch.float16, device="cuda")
    tq2.tq2_act16_from_f32(xd, y, m, k)
    back = torch.empty((m, k), dtype=torch.float32, device="cuda")
    tq2.tq2_act16_to_f32(y, back, m, k)
    torch.cuda.synchronize()
    ref = to_act16(x)
    assert np.array_equal(y.cpu().numpy().view(np.uint16), ref.view(np.uint16))
    assert np.array_equal(back.cpu().numpy(), from_act16(ref).astype(np.float32))


def run_act16(tq2, w, x16_np, r16_np, m, n, k, *, inplace=False):
    x16 = torch.from_numpy(x16_np).cuda()
    if inplace:
        out = torch.from_numpy(r16_np).cuda()
        r = out
    else:
        out = torch.full((m, n), float("nan"), dtype=torch.float16, device="cuda")
        r = None if r16_np is None else torch.from_numpy(r16_np).cuda()
    tq2.tq2_gemm_act16(w, x16, r, out, m, n, k)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def check_act16(got16, p, x32, r32, *, rows=None, what=""):
    """|out - ref| <= 4e-3 Sigma|xw| + 2^-11 |ref| (the f16 path's product bound and
    the one rounding of the result to binary16; x16 values are inputs, exact)."""
    ref, scale = oracle.matmul(p.w_aos, x32, r32, n=p.n, k=p.k, rows=rows)
    got = from_act16(got16).astype(np.float64)
    got = got if rows is None else got[rows]
    bound = TOL_TC * scale + 2.0 ** -11 * np.abs(ref) + 2.0 ** -24
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got)), what
    assert np.all(err <= bound), f"{what}: max err/bound {float(np.max(err / bound)):.3g}"
    num = np.sum(got * ref, axis=1)
    den = np.linalg.norm(got, axis=1) * np.linalg.norm(ref, axis=1)
    c = np.where(den > 0, num / np.where(den > 0, den, 1), 1.0)
    assert np.all(c >= COS_MIN), f"{what}: min row cosine {c.min()}"


@pytest.mark.parametrize("m,n,k,res", [(8, 1024, 1024, False), (129, 256, 640, True), (300, 48, 128, False),
                                       (64, 4096, 4096, True), (1, 16, 128, False), (1536, 3072, 3072, True)])
def test_gemm_act16_parity(tq2, m, n, k, res):
    # (64, 4096, 4096) splits K; (1536, 3072, 3072) is the DiT shape (sampled rows)
    p = tq2_synth.make_problem(m, n, k, seed=m + n + k, residual=res)
    x16 = to_act16(p.x)
    r16 = to_act16(p.residual) if res else None
    w = upload(tq2, p)
    got = run_act16(tq2, w, x16, r16, m, n, k)
    x32 = from_act16(x16).astype(np.float32)
    r32 = from_act16(r16).astype(np.float32) if res else None
    rows = sample_rows(m) if m > 256 else None
    check_act16(got if rows is None else got, p, x32, r32, rows=rows, what=f"act16 {m}x{n}x{k}")
    if res:  # in place: out16 = residual16 on entry
        got2 = run_act16(tq2, w, x16, r16, m, n, k, inplace=True)
        assert np.array_equal(got2.view(np.uint16), got.view(np.uint16))


def test_gemm_act16_chain_two_layers(tq2):
    # layer 1 (k0 -> k1) feeds layer 2 (k1 -> n2) in the activation layout on the
    # GPU; the oracle runs the same chain with the intermediate rounded to binary16
    # by numpy.  Layer 2's bound adds |W2| times layer 1's bound plus one binary16
    # step of the intermediate (the two sides may round it one step apart).
    m, k0, k1, n2 = 96, 1024, 2048, 512
    p1 = tq2_synth.make_problem(m, k1, k0, seed=5)
    p2 = tq2_synth.make_problem(m, n2, k1, seed=6)
    w1, w2 = upload(tq2, p1), upload(tq2, p2)
    x16 = torch.from_numpy(to_act16(p1.x)).cuda()
    h16 = torch.empty((m, k1), dtype=torch.float16, device="cuda")
    o16 = torch.empty((m, n2), dtype=torch.float16, device="cuda")
    tq2.tq2_gemm_act16(w1, x16, None, h16, m, k1, k0)
    tq2.tq2_gemm_act16(w2, h16, None, o16, m, n2, k1)
    torch.cuda.synchronize()
    x32 = from_act16(to_act16(p1.x)).astype(np.float32)
    ref1, s1 = oracle.matmul(p1.w_aos, x32, n=k1, k=k0)
    h = ref1.astype(np.float16)                       # the oracle's rounded intermediate
    b1 = TOL_TC * s1 + 2.0 ** -11 * np.abs(ref1)      # layer 1's bound
    step = np.abs(np.spacing(h.astype(np.float16))).astype(np.float64)
    ref2, s2 = oracle.matmul(p2.w_aos, h.astype(np.float32), n=n2, k=k1)
    W2 = np.abs(oracle.dequant(p2.w_aos, n2, k1))
    bound = TOL_TC * s2 + 2.0 ** -11 * np.abs(ref2) + (b1 + step) @ W2.T + 2.0 ** -24
    got = from_act16(o16.cpu().numpy()).astype(np.float64)
    assert np.all(np.abs(got - ref2) <= bound)


def test_act16_errors(tq2):
    x = torch.zeros(4, 128, dtype=torch.float16, device="cuda")
    o = torch.zeros(4, 40, dtype=torch.float16, device="cuda")
    w = torch.zeros(int(tq2.tq2_soa_bytes(40, 128)), dtype=torch.uint8, device="cuda")
    L = tq2.lib
    assert L.tq2_gemm_act16(w.data_ptr(), x.data_ptr(), None, o.data_ptr(), 4, 40, 128, None) == tq2.TQ2_ERR_INVALID_ARG
    assert L.tq2_gemm_act16(w.data_ptr(), x.data_ptr(), None, o.data_ptr(), 4, 32, 100, None) == tq2.TQ2_ERR_BAD_K
    assert L.tq2_gemm_act16(w.data_ptr(), x.data_ptr(), None, o.data_ptr(), 0, 32, 128, None) == tq2.TQ2_OK
    assert L.tq2_gemm_act16(w.data_ptr(), x.data_ptr() + 2, None, o.data_ptr(), 4, 32, 128, None) == tq2.TQ2_ERR_MISALIGNED
    f = torch.zeros(4, 24, device="cuda")
    h = torch.zeros(4, 24, dtype=torch.float16, device="cuda")
    assert L.tq2_act16_from_f32(f.data_ptr(), h.data_ptr(), 4, 24, None) == tq2.TQ2_ERR_INVALID_ARG
    assert L.tq2_act16_to_f32(h.data_ptr(), f.data_ptr(), 4, 24, None) == tq2.TQ2_ERR_INVALID_ARG
    torch.cuda.synchronize()


# ---------------------------------------------------------------------------
# DiT joint attention

def run_attention(tq2, q, k, v, h, s, d):
    qd, kd, vd = (torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda() for a in (q, k, v))
    out = torch.full((s, h * d), float("nan"), dtype=torch.float32, device="cuda")
    tq2.tq2_attention_f32(qd, kd, vd, out, h, s, d)
    torch.cuda.synchronize()
    assert tq2.tq2_device_status() == tq2.TQ2_OK
    return out.cpu().numpy()


def check_attention(got, q, k, v, h, s, d, *, rows=None, what=""):
    """Per element: |out - ref| <= (2.1 ds + 4 * 2^-11) * sum_j p_j |v_j|, with
    ds = 2^-10 max_j sum_e |q_e k_je| / sqrt(d) the score error from rounding q
    and k to binary16 (carried through the softmax), and the 2^-11 terms for
    rounding P and v and the normalisation; plus cosine >= 0.9999 per row."""
    ref, absv = oracle.attention(q, k, v, heads=h, seq=s, dim=d, rows=rows)
    t = np.arange(s) if rows is None else np.asarray(rows)
    qa = np.abs(q.reshape(h, s, d).astype(np.float64))[:, t]
    ka = np.abs(k.reshape(h, s, d).astype(np.float64))
    ds = np.stack([(qa[hh] @ ka[hh].T).max(axis=1) for hh in range(h)], axis=1) * 2.0 ** -10 / np.sqrt(d)
    bound = (2.1 * np.repeat(ds, d, axis=1) + 4 * 2.0 ** -11) * absv + 1e-30
    got = got if rows is None else got[t]
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got)), what
    assert np.all(err <= bound), f"{what}: max err/bound {float(np.max(err / bound)):.3g}"
    num = np.sum(got * ref, axis=1)
    den = np.linalg.norm(got, axis=1) * np.linalg.norm(ref, axis=1)
    c = np.where(den > 0, num / np.where(den > 0, den, 1), 1.0)
    assert np.all(c >= COS_MIN), f"{what}: min row cosine {c.min()}"


@pytest.mark.parametrize("h,s,d", [(1, 128, 128), (2, 300, 128), (3, 77, 64), (1, 1, 128), (4, 1024, 128),
                                   (2, 513, 64), (2, 200, 8), (3, 129, 24), (2, 300, 72), (1, 257, 120),
                                   (2, 128, 56), (1, 64, 16), (2, 100, 96)])
def test_attention_parity(tq2, h, s, d):
    rng = np.random.default_rng(h * 1000 + s + d)
    q, k, v = (rng.standard_normal((h, s, d)).astype(np.float32) for _ in range(3))
    check_attention(run_attention(tq2, q, k, v, h, s, d), q, k, v, h, s, d, what=f"attn h={h} s={s} d={d}")


def test_attention_growing_scores_rescale(tq2):
    # scores that grow block after block (keys scaled up with their index) and a
    # wide range (q times 4): the running maximum moves by more than 2^8 several
    # times, so O and the sum are rescaled
    h, s, d = 2, 640, 128
    rng = np.random.default_rng(9)
    q = (rng.standard_normal((h, s, d)) * 4).astype(np.float32)
    k = (rng.standard_normal((h, s, d)) * np.linspace(0.2, 3.0, s)[None, :, None]).astype(np.float32)
    v = rng.standard_normal((h, s, d)).astype(np.float32)
    check_attention(run_attention(tq2, q, k, v, h, s, d), q, k, v, h, s, d, what="attn rescale")


def test_attention_dit_shape_sampled(tq2):
    # FLUX.2-sized: 24 heads of 128 (3072 features), 4096 tokens; sampled rows
    h, s, d = 24, 4096, 128
    rng = np.random.default_rng(24)
    q, k, v = (rng.standard_normal((h, s, d)).astype(np.float32) for _ in range(3))
    got = run_attention(tq2, q, k, v, h, s, d)
    check_attention(got, q, k, v, h, s, d, rows=sample_rows(s), what="attn dit")


@pytest.mark.parametrize("d", [128, 64])
def test_attention_wait_timeout_is_reported_and_context_survives(tq2, d):
    # a zero wait limit makes the kernel's first open wait give up: every role
    # (copies, MMA issue, the paired softmax warps) must leave without hanging,
    # the timeout must reach the status word, and the next call must be exact
    h, s = 2, 300
    rng = np.random.default_rng(31 + d)
    q, k, v = (rng.standard_normal((h, s, d)).astype(np.float32) for _ in range(3))
    qd, kd, vd = (torch.from_numpy(a).cuda() for a in (q, k, v))
    out = torch.zeros((s, h * d), dtype=torch.float32, device="cuda")
    assert tq2.tq2_device_status() == tq2.TQ2_OK
    old = tq2.tq2_set_wait_timeout_ns(0)
    try:
        tq2.tq2_attention_f32(qd, kd, vd, out, h, s, d)
        torch.cuda.synchronize()
        st = tq2.tq2_device_status()
    finally:
        tq2.tq2_set_wait_timeout_ns(old)
    assert st == tq2.TQ2_ERR_TIMEOUT
    check_attention(run_attention(tq2, q, k, v, h, s, d), q, k, v, h, s, d, what="attn after timeout")


def test_attention_errors(tq2):
    a = torch.zeros(2, 128, 128, device="cuda")
    o = torch.zeros(128, 256, device="cuda")
    L = tq2.lib
    # the head dimension must be a multiple of 8 in [8, 128]
    for bad in (0, 4, 12, 100, 136, 256, -8):
        assert L.tq2_attention_f32(a.data_ptr(), a.data_ptr(), a.data_ptr(), o.data_ptr(), 2, 128, bad,
                                   None) == tq2.TQ2_ERR_INVALID_ARG
    assert L.tq2_attention_f32(a.data_ptr(), a.data_ptr(), a.data_ptr(), o.data_ptr(), 0, 128, 128, None) == tq2.TQ2_OK
    assert L.tq2_attention_f32(a.data_ptr(), a.data_ptr(), a.data_ptr(), o.data_ptr(), 2, 0, 128, None) == tq2.TQ2_OK
    assert L.tq2_attention_f32(a.data_ptr() + 4, a.data_ptr(), a.data_ptr(), o.data_ptr(), 2, 128, 128, None) == tq2.TQ2_ERR_MISALIGNED
    assert L.tq2_attention_f32(a.data_ptr(), a.data_ptr(), a.data_ptr(), a.data_ptr(), 2, 128, 128, None) == tq2.TQ2_ERR_INVALID_ARG
    torch.cuda.synchronize()
