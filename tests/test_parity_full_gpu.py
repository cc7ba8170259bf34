"""GPU parity at the full benchmark sizes of the DiT configurations, through
the C ABI, against the CPU oracle.

* The DiT large-M GEMM (M=1536, K=3072, N in {3072, 9216, 12288}) is checked
  on every output element.
* The DiT forward set (100 linears at M=4096) is checked in full on layers 0,
  40, 60 and 80 (one of each (K, N) shape) and on sampled rows (all N columns
  of each) on every one of the 100 layers, residual layers included.

Bars as in the other parity tests: |out - ref| <= 4e-3 * Sigma|xw| +
2^-23 |residual| per element (Sigma|xw| from the oracle in f64) and a per-row
cosine >= 0.9999 for the tensor-core kernel the dispatcher picks here.
"""

import numpy as np
import pytest

import oracle
import tq2_synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL_TC = 4e-3
COS_MIN = 0.9999


@pytest.fixture(scope="module")
def tq2():
    import dit_tq2_g128_gb300 as m
    return m


def run_auto(tq2, p):
    w = tq2.upload_weight(p.w_aos, p.n, p.k)
    x = torch.from_numpy(p.x).cuda()
    r = None if p.residual is None else torch.from_numpy(p.residual).cuda()
    out = torch.full((p.m, p.n), float("nan"), dtype=torch.float32, device="cuda")
    tq2.tq2_gemm(w, x, r, out, p.m, p.n, p.k)
    torch.cuda.synchronize()
    assert tq2.tq2_device_status() == tq2.TQ2_OK
    got = out.cpu().numpy().astype(np.float64)
    del w, x, r, out
    return got


def check(got, p, rows=None, what=""):
    ref, scale = oracle.matmul(p.w_aos, p.x, p.residual, n=p.n, k=p.k, rows=rows)
    g = got if rows is None else got[rows]
    res = 0.0 if p.residual is None else np.abs(
        (p.residual if rows is None else p.residual[rows]).astype(np.float64))
    bound = TOL_TC * scale + 2.0 ** -23 * res + 1e-30
    err = np.abs(g - ref)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    assert np.all(err <= bound), f"{what}: max err/bound {float(np.max(err / bound)):.3g}"
    num = np.sum(g * ref, axis=1)
    den = np.linalg.norm(g, axis=1) * np.linalg.norm(ref, axis=1)
    c = np.where(den > 0, num / np.where(den > 0, den, 1), 1.0)
    assert np.all(c >= COS_MIN), f"{what}: min row cosine {c.min()}"


@pytest.mark.parametrize("n", tq2_synth.DIT_NS)
def test_dit_large_m_every_element(tq2, n):
    p = tq2_synth.dit(n)
    assert tq2.tq2_select_kernel(p.m, p.n, p.k) == tq2.TQ2_KERNEL_TC
    check(run_auto(tq2, p), p, what=f"dit m=1536 n={n}")


@pytest.mark.parametrize("layer", [0, 40, 60, 80])
def test_dit_forward_layer_every_element(tq2, layer):
    p = tq2_synth.dit_forward_layer(layer)
    check(run_auto(tq2, p), p, what=f"dit forward layer {layer}")


def layer_rows(m, layer):
    """First and last row, both sides of the 128- and 256-row tile edges, and
    a few seeded rows: the output tile each lands in varies with the layer."""
    base = {0, 127, 128, 255, 256, m - 257, m - 129, m - 1}
    rng = np.random.default_rng(1000 + layer)
    base.update(rng.integers(0, m, size=6).tolist())
    return np.array(sorted(base), dtype=np.int64)


@pytest.mark.parametrize("layer", range(len(tq2_synth.DIT_FORWARD_SHAPES)))
def test_dit_forward_every_layer_sampled(tq2, layer):
    p = tq2_synth.dit_forward_layer(layer)
    got = run_auto(tq2, p)
    assert np.all(np.isfinite(got)), f"layer {layer}: non-finite output"
    check(got, p, rows=layer_rows(p.m, layer), what=f"dit forward layer {layer}")
