"""GPU tests of what each entry point may touch, through the C ABI.

* Guard bands: every output-writing entry point writes into a buffer with
  256 bytes of a sentinel pattern before and after the output; the sentinels
  must be untouched, and the output (filled with NaN beforehand) must be
  written in full.  Ragged shapes (tile tails in M, N and K) and the
  benchmark shapes are covered.
* Residency: an operand that is not device memory of the current device
  (pageable host memory, pinned host memory) is refused with
  TQ2_ERR_INVALID_ARG before anything is launched: the output keeps its
  contents and the stream stays clean.
"""

import ctypes

import numpy as np
import pytest

import tq2_synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

PAD = 256  # guard bytes on each side


@pytest.fixture(scope="module")
def tq2():
    import dit_tq2_g128_gb300 as m
    return m


class Guarded:
    """A device buffer of `numel` elements between two 256-byte sentinel bands."""

    def __init__(self, numel, dtype=torch.float32, fill=float("nan")):
        esz = torch.empty(0, dtype=dtype).element_size()
        self.pad = PAD // esz
        self.buf = torch.empty(self.pad * 2 + numel, dtype=dtype, device="cuda")
        self.buf.view(torch.uint8).fill_(0xA5)
        self.view = self.buf[self.pad:self.pad + numel]
        if fill is not None:
            self.view.fill_(fill)
        self.numel = numel

    def bands_intact(self):
        raw = self.buf.view(torch.uint8).cpu().numpy()
        nb = self.pad * self.buf.element_size()
        return bool(np.all(raw[:nb] == 0xA5) and np.all(raw[-nb:] == 0xA5))

    def written(self):
        v = self.view.float().cpu().numpy()
        return bool(np.all(np.isfinite(v)))


def finish(tq2, g):
    torch.cuda.synchronize()
    assert tq2.tq2_device_status() == tq2.TQ2_OK
    assert g.bands_intact(), "a write landed outside the output"
    assert g.written(), "the output was not written in full"


MATMUL_SHAPES = [(1, 1, 128), (1, 257, 640), (1, 12288, 4096), (1, 4096, 12288), (1, 153, 2048), (2, 300, 384),
                 (3, 7, 128), (8, 1024, 1024), (16, 129, 256), (17, 257, 384), (129, 300, 640),
                 (300, 1028, 256), (1536, 3072, 3072)]


def kernels_for(tq2, m):
    ks = [("AUTO", tq2.TQ2_KERNEL_AUTO), ("TC", tq2.TQ2_KERNEL_TC), ("F32REF", tq2.TQ2_KERNEL_F32REF),
          ("TC_DIRECT", tq2.TQ2_KERNEL_TC_DIRECT)]
    if m == 1:
        ks.append(("GEMV", tq2.TQ2_KERNEL_GEMV))
    if m <= 16:
        ks.append(("SKINNY", tq2.TQ2_KERNEL_SKINNY))
    if 2 <= m <= 32:
        ks.append(("SKINNY_MMA", tq2.TQ2_KERNEL_SKINNY_MMA))
    return ks


@pytest.mark.parametrize("m,n,k", MATMUL_SHAPES)
@pytest.mark.parametrize("res", ["none", "distinct", "inplace"])
def test_matmul_guard_bands(tq2, m, n, k, res):
    p = tq2_synth.make_problem(m, n, k, seed=m + n + k, residual=res != "none")
    w = tq2.upload_weight(p.w_aos, n, k)
    x = torch.from_numpy(p.x).cuda()
    r = None if p.residual is None else torch.from_numpy(p.residual).cuda()
    for name, kern in kernels_for(tq2, m):
        if name == "F32REF" and m * n * k > 2 ** 31:
            continue
        g = Guarded(m * n)
        rr = r
        if res == "inplace":
            g.view.copy_(r.reshape(-1))
            rr = g.view
        tq2.tq2_gemm_with(kern, w, x, rr, g.view, m, n, k)
        finish(tq2, g)
    if tq2.tq2_select_kernel(m, n, k) == tq2.TQ2_KERNEL_TC:
        for entry in ("ws", "noalloc"):
            if entry == "noalloc" and tq2.tq2_gemm_workspace_bytes(m, n, k) > tq2.TQ2_NOALLOC_SCRATCH_BYTES:
                continue
            g = Guarded(m * n)
            rr = r
            if res == "inplace":
                g.view.copy_(r.reshape(-1))
                rr = g.view
            if entry == "ws":
                ws = Guarded(tq2.tq2_gemm_workspace_bytes(m, n, k), torch.uint8, fill=None)
                tq2.tq2_gemm_ws(w, x, rr, g.view, m, n, k, ws.view, ws.numel)
                torch.cuda.synchronize()
                assert ws.bands_intact(), "a write landed outside the workspace"
            else:
                tq2.tq2_gemm_noalloc(w, x, rr, g.view, m, n, k)
            finish(tq2, g)
    if m == 1:
        for fn in (tq2.tq2_gemv, tq2.tq2_gemv_resident):
            g = Guarded(n)
            torch.cuda.synchronize()
            fn(w, x[0], None if r is None else r[0], g.view, n, k)
            finish(tq2, g)


@pytest.mark.parametrize("m,f,k", [(1, 48, 256), (1, 6144, 4096), (2, 64, 256), (8, 100, 384),
                                   (129, 48, 640), (300, 1024, 3072)])
def test_swiglu_guard_bands(tq2, m, f, k):
    p = tq2_synth.make_problem(m, 2 * f, k, seed=f + k)
    w = tq2.upload_weight(p.w_aos, 2 * f, k)
    x = torch.from_numpy(p.x).cuda()
    g = Guarded(m * f)
    tq2.tq2_gate_up_swiglu(w, x, g.view, m, f, k)
    finish(tq2, g)


@pytest.mark.parametrize("m,n,k,res", [(1, 48, 128, False), (7, 1024, 1024, True), (129, 256, 640, True),
                                       (300, 48, 128, False), (1536, 3072, 3072, False)])
def test_act16_guard_bands(tq2, m, n, k, res):
    p = tq2_synth.make_problem(m, n, k, seed=7 * m + n, residual=res)
    w = tq2.upload_weight(p.w_aos, n, k)
    x = torch.from_numpy(p.x).cuda()
    x16 = Guarded(m * k, torch.float16)
    tq2.tq2_act16_from_f32(x, x16.view, m, k)
    finish(tq2, x16)
    r16 = None
    if res:
        r16 = torch.empty(m * n, dtype=torch.float16, device="cuda")
        tq2.tq2_act16_from_f32(torch.from_numpy(p.residual).cuda(), r16, m, n)
    g = Guarded(m * n, torch.float16)
    tq2.tq2_gemm_act16(w, x16.view, r16, g.view, m, n, k)
    finish(tq2, g)
    back = Guarded(m * n)
    tq2.tq2_act16_to_f32(g.view, back.view, m, n)
    finish(tq2, back)


@pytest.mark.parametrize("h,s,d", [(1, 1, 128), (2, 200, 128), (3, 77, 64), (2, 129, 64)])
def test_attention_guard_bands(tq2, h, s, d):
    rng = np.random.default_rng(h * s + d)
    q, k, v = (torch.from_numpy(rng.standard_normal((h, s, d)).astype(np.float32)).cuda() for _ in range(3))
    g = Guarded(s * h * d)
    tq2.tq2_attention_f32(q, k, v, g.view, h, s, d)
    finish(tq2, g)


@pytest.mark.parametrize("n,k", [(1, 128), (7, 384), (300, 1024)])
def test_quantize_and_reformat_guard_bands(tq2, n, k):
    wf = torch.randn((n, k), device="cuda") * 0.02
    nb = tq2.tq2_soa_bytes(n, k)
    aos = Guarded(nb, torch.uint8, fill=None)
    aos.view.fill_(0x5A)
    tq2.tq2_quantize_f32(wf, aos.view, n, k)
    torch.cuda.synchronize()
    assert aos.bands_intact()
    soa = Guarded(nb, torch.uint8, fill=None)
    tq2.tq2_reformat_aos_to_soa(aos.view, soa.view, n, k)
    torch.cuda.synchronize()
    assert soa.bands_intact()


# ---------------------------------------------------------------------------
# residency of the operands


def test_operands_not_on_this_device_are_refused(tq2):
    L = tq2.lib
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    m, n, k = 256, 256, 256
    p = tq2_synth.make_problem(m, n, k, seed=5, residual=True)
    w = tq2.upload_weight(p.w_aos, n, k)
    x = torch.from_numpy(p.x).cuda()
    r = torch.from_numpy(p.residual).cuda()
    out = torch.full((m, n), 3.0, device="cuda")
    x16 = torch.zeros((m, k), dtype=torch.float16, device="cuda")
    o16 = torch.full((m, n), 3.0, dtype=torch.float16, device="cuda")
    # host memory: pageable (numpy) and page-locked (torch pinned)
    host = np.zeros(8 * m * max(n, k), dtype=np.float32)
    pinned = torch.zeros(8 * m * max(n, k), dtype=torch.float32).pin_memory()
    # 256-byte aligned host addresses, so that only residency can be the reason for a refusal
    host_a = (host.ctypes.data + 255) & ~255
    pinned_a = (pinned.data_ptr() + 255) & ~255
    for label, hp in (("pageable", host_a), ("pinned", pinned_a)):
        bad = tq2.TQ2_ERR_INVALID_ARG
        # element-wise converter first (a plain-load kernel), then every other entry point
        assert L.tq2_act16_from_f32(hp, x16.data_ptr(), m, k, stream) == bad, label
        assert L.tq2_act16_to_f32(o16.data_ptr(), hp, m, n, stream) == bad, label
        for gv in (L.tq2_gemv, L.tq2_gemv_resident):
            assert gv(w.data_ptr(), hp, None, out.data_ptr(), n, k, stream) == bad, label
            assert gv(hp, x.data_ptr(), None, out.data_ptr(), n, k, stream) == bad, label
            assert gv(w.data_ptr(), x.data_ptr(), hp, out.data_ptr(), n, k, stream) == bad, label
            assert gv(w.data_ptr(), x.data_ptr(), None, hp, n, k, stream) == bad, label
        for kern in (0, 1, 2, 3, 4, 5, 6):
            mm = 1 if kern == 1 else m
            for args in ((hp, x.data_ptr(), None, out.data_ptr()), (w.data_ptr(), hp, None, out.data_ptr()),
                         (w.data_ptr(), x.data_ptr(), hp, out.data_ptr()),
                         (w.data_ptr(), x.data_ptr(), None, hp)):
                assert L.tq2_gemm_with(kern, *args, mm, n, k, stream) == bad, (label, kern)
        ws = tq2.workspace(m, n, k)
        assert L.tq2_gemm_ws(w.data_ptr(), x.data_ptr(), None, out.data_ptr(), m, n, k, hp,
                             ws.numel(), stream) == bad, label
        assert L.tq2_gemm_ws(w.data_ptr(), hp, None, out.data_ptr(), m, n, k, ws.data_ptr(),
                             ws.numel(), stream) == bad, label
        assert L.tq2_gemm_noalloc(w.data_ptr(), hp, None, out.data_ptr(), m, n, k, stream) == bad, label
        assert L.tq2_gemm_act16(w.data_ptr(), hp, None, o16.data_ptr(), m, n, k, stream) == bad, label
        assert L.tq2_gemm_act16(w.data_ptr(), x16.data_ptr(), hp, o16.data_ptr(), m, n, k, stream) == bad
        assert L.tq2_gemm_act16(w.data_ptr(), x16.data_ptr(), None, hp, m, n, k, stream) == bad, label
        assert L.tq2_gate_up_swiglu(w.data_ptr(), hp, out.data_ptr(), m, n // 2, k, stream) == bad, label
        assert L.tq2_attention_f32(hp, x.data_ptr(), r.data_ptr(), out.data_ptr(), 2, 128, 128,
                                   stream) == bad, label
        assert L.tq2_quantize_f32(hp, out.data_ptr(), n, k, stream) == bad, label
        assert L.tq2_reformat_aos_to_soa(hp, out.data_ptr(), n, k, stream) == bad, label
        assert L.tq2_reformat_aos_to_soa(w.data_ptr(), hp, n, k, stream) == bad, label
    torch.cuda.synchronize()
    assert tq2.tq2_device_status() == tq2.TQ2_OK
    assert torch.all(out == 3.0) and torch.all(o16 == 3.0)  # nothing ran
    # the same calls with every operand on the device succeed
    tq2.tq2_gemm(w, x, r, out, m, n, k)
    tq2.tq2_gemm_act16(w, x16, None, o16, m, n, k)
    torch.cuda.synchronize()
    assert torch.all(torch.isfinite(out))
