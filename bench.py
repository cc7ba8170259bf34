"""Benchmark of the TQ2_0_g128 ternary matmul library on one GB300.

Default workload (one JSON line): the M=1 decode GEMV, K=4096, N=12288 (the
fused gate/up shape), on seeded synthetic inputs.  One step is one tq2_gemv
call through the C ABI; K steps are captured in a CUDA graph, each step
reading a different copy of the weight so that the copies together exceed
twice the L2 size, and the graph is replayed several times inside the timed
region (median and best reported).  `value` is the weight bytes streamed per
second.  The same JSON line also carries the large-M GEMM numbers (M=1536,
K=3072, N in {3072, 9216, 12288}, TFLOP/s) measured the same way.

The library runs on one GPU only: a request for more GPUs (--gpus N > 1, or a
multi-process launch) is refused before anything touches a GPU.

`--impl reference` times the CPU oracle (test infrastructure, double
precision) on the same workload and metric instead.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import platform
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import tq2_synth  # noqa: E402

METRIC = "TQ2 GEMM TFLOP/s @M=1536 and GEMV weight-GB/s @M=1, as % of GB300 roofline"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-gemm", action="store_true", help="skip the large-M GEMM section")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--gemm-steps", type=int, default=20)
    ap.add_argument("--replays", type=int, default=7, help="timed replays of the GEMV graph (at least 5)")
    ap.add_argument("--gemm-n", type=int, default=0, help="only this N of the large-M set")
    ap.add_argument("--no-clock-window", action="store_true",
                    help="skip the 1 s sustained window that feeds the clock record")
    ap.add_argument("--suite", action="store_true",
                    help="instead of the bench line: every workload configuration (time per call, "
                         "rate, parity on sampled rows against the oracle, oracle time on the sample)")
    ap.add_argument("--cpu-configs", action="store_true",
                    help="instead of the bench line (no GPU): the CPU oracle on configs 1, 2a, 2b and 3, "
                         "one whole call each, at one thread and at all threads")
    ap.add_argument("--cpu-full", action="store_true",
                    help="instead of the bench line (no GPU): the CPU oracle on the DiT configurations in "
                         "full (M=1536 at each N, then the 100-layer forward set at M=4096), all host threads")
    ap.add_argument("--skinny", type=int, default=0,
                    help="instead of the bench line: tq2_gemm at the skinny-sweep shape (M rows, K=N=4096) "
                         "alone, `--steps` calls after `--warmup` on rotating weight copies, one JSON line "
                         "with the time per call (for profiling that path)")
    ap.add_argument("--encoder", action="store_true",
                    help="only tq2_quantize_f32 at 12288 x 3072 (the encoder's ncu workload)")
    ap.add_argument("--attention", action="store_true",
                    help="instead of the bench line: the DiT joint attention alone (24 heads x 4096 "
                         "tokens x 128, seeded N(0,1) inputs), `--steps` calls after `--warmup`, "
                         "one JSON line with the time per call (for profiling that kernel)")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        hbm = float(d.get("hbm_gbs"))
        bf16 = float(d.get("bf16_tflops"))
        bf16s = float(d.get("bf16_tflops_sustained", bf16))
        return hbm, bf16, bf16s, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, FALLBACK_BF16_TFLOPS_SUSTAINED, "fallback"


def world_from_env():
    """(world size, rank) of a torchrun launch, (1, 0) otherwise."""
    return int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0"))


SINGLE_GPU_ONLY = ("bench.py runs on one GPU only: the tensor-core kernels copy shared x tiles "
                   "between the two CTAs of a cluster (cluster multicast), which is offered for "
                   "single-GPU calls only, so no multi-GPU run of this library is provided")


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling while the GPU is busy."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def source_hash(*files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key, src_files):
    """Per-launch DRAM bytes from a committed ncu summary, if taken on the
    current source of the kernel; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[kernel_key]
        if e.get("source_hash") != source_hash(*src_files):
            return None
        return float(e["dram_bytes_per_launch"])
    except Exception:
        return None


# ---------------------------------------------------------------------------
# our arm


def graph_of(fn, steps, torch):
    """Capture `steps` calls fn(i) into one CUDA graph."""
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for i in range(steps):
                fn(i)
    torch.cuda.current_stream().wait_stream(s)
    return g


def time_graph(g, torch, reps=1):
    """Device times (s) of `reps` replays, CUDA events on the replay stream."""
    ts = []
    for _ in range(reps):
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) / 1e3)
    return ts


GEMV_CONFIG = {"workload": "decode_gemv_m1_k4096_n12288", "m": 1, "k": 4096, "n": 12288,
               "weight_bytes": 13369344,
               "l2": "inputs larger than L2: rotating weight copies, together more than twice the L2 size"}


def run_ours(args):
    import torch
    import dit_tq2_g128_gb300 as tq2

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    hbm, bf16, bf16s, peak_src = peaks()
    props = torch.cuda.get_device_properties(device)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))

    # ---- decode GEMV workload
    p = tq2_synth.decode_gate_up(seed=0)
    wbytes = tq2.tq2_soa_bytes(p.n, p.k)
    assert wbytes == GEMV_CONFIG["weight_bytes"]
    copies = max(2, -(-2 * l2 // wbytes) + 1)
    w0 = tq2.upload_weight(p.w_aos, p.n, p.k)
    ws = [w0] + [w0.clone() for _ in range(copies - 1)]
    x = torch.from_numpy(p.x[0]).to(device)
    out = torch.empty(p.n, dtype=torch.float32, device=device)

    def step(i):
        tq2.tq2_gemv(ws[i % copies], x, None, out, p.n, p.k)

    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    assert tq2.tq2_device_status() == tq2.TQ2_OK
    gw = graph_of(step, max(3, args.warmup), torch)
    gt = graph_of(step, args.steps, torch)
    gw.replay()
    torch.cuda.synchronize()
    smi_id = "0"
    try:  # nvidia-smi numbers GPUs physically; the CUDA ordinal may differ
        smi_id = "GPU-" + str(props.uuid)
    except Exception:
        pass
    reps = max(5, args.replays)
    with ClockSampler(smi_id) as clk:
        # sustained window for the clock record (same graph, >= 1 s of load)
        t_end = time.time() + (0.0 if args.no_clock_window else 1.0)
        while time.time() < t_end:
            gt.replay()
            torch.cuda.synchronize()
        t_reps = time_graph(gt, torch, reps=reps)
    clocks = clk.summary()
    t_step = statistics.median(t_reps)
    per_launch = t_step / args.steps
    value = wbytes * args.steps / t_step / 1e9
    achieved = wbytes / per_launch / 1e9

    # ---- the same calls through tq2_gemv_resident (weights uploaded once and
    # synchronised above: its contract holds), reported beside the value
    def step_r(i):
        tq2.tq2_gemv_resident(ws[i % copies], x, None, out, p.n, p.k)

    for i in range(3):
        step_r(i)
    torch.cuda.synchronize()
    gr = graph_of(step_r, args.steps, torch)
    gr.replay()
    torch.cuda.synchronize()
    t_res = time_graph(gr, torch, reps=reps)
    t_res_med = statistics.median(t_res)

    # ---- end to end through the C ABI with host buffers
    x_host = torch.from_numpy(p.x[0].copy()).pin_memory()
    out_host = torch.empty(p.n, dtype=torch.float32).pin_memory()
    xd = torch.empty_like(x)
    stream = torch.cuda.current_stream()

    def e2e_step(i):
        xd.copy_(x_host, non_blocking=True)
        tq2.tq2_gemv(ws[i % copies], xd, None, out, p.n, p.k)
        out_host.copy_(out, non_blocking=True)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    # eager: one Python call per copy and per GEMV (host dispatch paces it)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        e2e_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    t_eager = e0.elapsed_time(e1) / 1e3
    # captured: the same steps (copy up, tq2_gemv, copy down) in one CUDA
    # graph, as a decode loop would run them; value from the median replay
    ge = graph_of(e2e_step, args.steps, torch)
    ge.replay()
    torch.cuda.synchronize()
    t_e2e_reps = time_graph(ge, torch, reps=max(3, min(reps, 5)))
    t_e2e = statistics.median(t_e2e_reps)
    assert np.array_equal(out_host.numpy(), out.cpu().numpy())
    e2e = {"value": wbytes * args.steps / t_e2e / 1e9, "unit": "GB/s",
           "h2d_bytes_per_step": int(x_host.numel() * 4), "d2h_bytes_per_step": int(out_host.numel() * 4),
           "us_per_step": round(t_e2e / args.steps * 1e6, 3),
           "eager_value": round(wbytes * args.steps / t_eager / 1e9, 2),
           "note": "weights resident (uploaded once); every step copies x up from and out down to pinned "
                   "host buffers around tq2_gemv; the steps captured in one CUDA graph and replayed "
                   "(median of the replays); eager_value: the same steps issued one Python call at a time"}

    gemv_src = ["dit_tq2_g128_gb300/csrc/gemv.cu"]
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s (TQ2 weight bytes, M=1 GEMV)",
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_step / args.steps * 1e3, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32 in/out; x as 23-bit fixed point per 128-weight block, int32 (dp4a) ternary dot products, f32 scale and sum",
        "data": "synthetic (seeded numpy: x~N(0,1), codes P(0)=0.4 P(+-1)=0.3, d=f16(|N(0,0.02)|+1e-4))",
        "config": dict(GEMV_CONFIG),
        "timing": {"entry": "tq2_gemv",
                   "method": f"{args.steps} calls captured in one CUDA graph on {copies} rotating weight "
                             f"copies ({copies * wbytes / 2**20:.0f} MiB, L2 {l2 / 2**20:.0f} MiB); "
                             f"{reps} replays timed with CUDA events on the replay stream; value from the median",
                   "us_per_call_median": round(t_step / args.steps * 1e6, 4),
                   "us_per_call_best": round(min(t_reps) / args.steps * 1e6, 4),
                   "us_per_call_replays": [round(t / args.steps * 1e6, 4) for t in t_reps],
                   "sm_mhz_median": clocks.get("sm_mhz"),
                   "note": "consecutive calls overlap through programmatic dependent launch: each call's "
                           "launch and L2 prefetch of its weights run during the previous call",
                   "resident": {"entry": "tq2_gemv_resident",
                                "us_per_call_median": round(t_res_med / args.steps * 1e6, 4),
                                "GB_per_s": round(wbytes * args.steps / t_res_med / 1e9, 2),
                                "note": "same calls, same bits; weights written by no unfinished work, so each "
                                        "call copies its weight rows into shared memory during the previous "
                                        "call (separate timed region, not in value)"}},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "peak_source": f"{peak_src} (copy bandwidth)",
                     "traffic": ncu_traffic("gemv_m1_k4096_n12288", gemv_src),
                     "algorithmic_bytes_per_launch": wbytes,
                     "note": "achieved = weight bytes / (graph time / launches); includes inter-kernel gaps"},
        "clocks": clocks,
        "e2e": e2e,
        "gpu_launches": args.steps * reps,
        "impl": "ours",
    }

    # ---- large-M GEMM (tensor cores)
    if not args.no_gemm:
        gemm = {}
        launches = 0
        for n in tq2_synth.DIT_NS:
            if args.gemm_n and n != args.gemm_n:
                continue
            q = tq2_synth.dit(n, seed=0)
            per = q.m * q.k * 4 + tq2.tq2_soa_bytes(q.n, q.k) + q.m * q.n * 4
            c = max(2, -(-2 * l2 // per) + 1)
            wq = tq2.upload_weight(q.w_aos, q.n, q.k)
            wl = [wq] + [wq.clone() for _ in range(c - 1)]
            xl = [torch.from_numpy(q.x).to(device) for _ in range(c)]
            ol = [torch.empty((q.m, q.n), dtype=torch.float32, device=device) for _ in range(c)]

            wsl = [tq2.workspace(q.m, q.n, q.k, device=device) for _ in range(c)]

            def gstep(i, q=q, wl=wl, xl=xl, ol=ol, c=c):
                tq2.tq2_gemm(wl[i % c], xl[i % c], None, ol[i % c], q.m, q.n, q.k)

            def gstep_ws(i, q=q, wl=wl, xl=xl, ol=ol, c=c, wsl=wsl):
                tq2.tq2_gemm_ws(wl[i % c], xl[i % c], None, ol[i % c], q.m, q.n, q.k, wsl[i % c],
                                wsl[i % c].numel())

            def gstep_direct(i, q=q, wl=wl, xl=xl, ol=ol, c=c):
                tq2.tq2_gemm_with(tq2.TQ2_KERNEL_TC_DIRECT, wl[i % c], xl[i % c], None, ol[i % c],
                                  q.m, q.n, q.k)

            flops = 2.0 * q.m * q.n * q.k
            res = {}
            kernels_per_call = {"tq2_gemm": 2, "tq2_gemm_ws": 2, "tc_direct": 1}
            for name, fn in (("tq2_gemm", gstep), ("tq2_gemm_ws", gstep_ws), ("tc_direct", gstep_direct)):
                for i in range(3):
                    fn(i)
                torch.cuda.synchronize()
                assert tq2.tq2_device_status() == tq2.TQ2_OK
                gg = graph_of(fn, args.gemm_steps, torch)
                gg.replay()
                torch.cuda.synchronize()
                tg = statistics.median(time_graph(gg, torch, reps=3)) / args.gemm_steps
                launches += 3 * args.gemm_steps * kernels_per_call[name]
                res[name] = (tg, flops / tg / 1e12)
            tg, tfl = res["tq2_gemm"]
            gemm[f"n{n}"] = {"m": q.m, "k": q.k, "n": q.n, "entry": "tq2_gemm",
                             "us_per_call": round(tg * 1e6, 2),
                             "tflops": round(tfl, 1), "frac_of_bf16_burst": round(tfl / bf16, 4),
                             "frac_of_bf16_sustained": round(tfl / bf16s, 4),
                             "tq2_gemm_ws": {"us_per_call": round(res["tq2_gemm_ws"][0] * 1e6, 2),
                                             "tflops": round(res["tq2_gemm_ws"][1], 1)},
                             "tc_direct": {"us_per_call": round(res["tc_direct"][0] * 1e6, 2),
                                           "tflops": round(res["tc_direct"][1], 1)},
                             "l2": f"{c} rotating (x, w, out) copies"}
            del wl, xl, ol, wq, wsl
            torch.cuda.empty_cache()
        top = gemm[f"n{max(int(k[1:]) for k in gemm)}"]
        line["gemm_m1536"] = {
            "kernel": "tq2_gemm -> x f16-tile pre-pass into a stream-ordered temporary + clustered "
                      "persistent tcgen05 kind::f16 kernel (f16 operands, f32 accumulation in TMEM); "
                      "tq2_gemm_ws (caller workspace) and tc_direct (in-kernel x conversion) alongside",
            "per_n": gemm,
            "roofline": {"bound": "tensor", "unit": "TFLOP/s",
                         "achieved": top["tflops"], "peak": bf16,
                         "frac": round(top["tflops"] / bf16, 4),
                         "peak_source": f"{peak_src} dense bf16 burst (f16 runs at the bf16 rate)",
                         "traffic": (ncu_traffic("tc_ws_m1536_k3072_n12288",
                                                 ["dit_tq2_g128_gb300/csrc/gemm_tc_ws.cu"])
                                     if top["n"] == 12288 else None),
                         "traffic_note": "DRAM bytes of one tc_ws_kernel launch (the pre-pass is a "
                                         "separate launch); algorithmic: x f16 9.4 MB + weights "
                                         "10.0 MB read, 75.5 MB of output written"},
            "note": "timed separately from `value`; steps per N captured in a CUDA graph"}
    return line


# ---------------------------------------------------------------------------
# --suite: all workload configurations


def run_attention_only(args):
    """The DiT joint attention at the FLUX.2 shape, nothing else (the workload of
    the attention kernel's ncu summary)."""
    import torch
    import dit_tq2_g128_gb300 as tq2

    h, s, d = 24, 4096, 128
    rng = np.random.default_rng(24)
    q, k, v = (torch.from_numpy(rng.standard_normal((h, s, d)).astype(np.float32)).cuda() for _ in range(3))
    out = torch.empty((s, h * d), dtype=torch.float32, device="cuda")
    for _ in range(args.warmup):
        tq2.tq2_attention_f32(q, k, v, out, h, s, d)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        tq2.tq2_attention_f32(q, k, v, out, h, s, d)
    e1.record()
    torch.cuda.synchronize()
    assert tq2.tq2_device_status() == tq2.TQ2_OK
    t = e0.elapsed_time(e1) / 1e3 / max(args.steps, 1)
    return {"workload": "dit_joint_attention_h24_s4096_d128", "steps": args.steps, "warmup": args.warmup,
            "us_per_call": round(t * 1e6, 2), "TFLOPs": round(4.0 * h * s * s * d / t / 1e12, 2)}


def run_encoder_only(args):
    """tq2_quantize_f32 on the largest DiT weight (12288 x 3072, N(0, 0.02)
    weights as in the suite), nothing else: the workload of the encoder's ncu
    summary.  The calls are captured in one CUDA graph."""
    import torch
    import dit_tq2_g128_gb300 as tq2

    n, k = 12288, 3072
    wf = torch.randn((n, k), device="cuda", generator=torch.Generator(device="cuda").manual_seed(12)) * 0.02
    aos = torch.empty(tq2.tq2_soa_bytes(n, k), dtype=torch.uint8, device="cuda")

    def step(i):
        tq2.tq2_quantize_f32(wf, aos, n, k)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    steps = max(args.steps, 1)
    g = graph_of(step, steps, torch)
    g.replay()
    torch.cuda.synchronize()
    t = statistics.median(time_graph(g, torch, reps=3)) / steps
    assert tq2.tq2_device_status() == tq2.TQ2_OK
    return {"workload": "encoder_f32_to_blocks_12288x3072", "steps": args.steps, "warmup": args.warmup,
            "us_per_call": round(t * 1e6, 2), "f32_GBps": round(n * k * 4 / t / 1e9, 1),
            "bytes_GBps": round((n * k * 4 + tq2.tq2_soa_bytes(n, k)) / t / 1e9, 1),
            "method": "steps captured in one CUDA graph, median of 3 replays"}


def run_skinny_only(args):
    """tq2_gemm at M = args.skinny rows, K = N = 4096 (the skinny sweep's shape),
    nothing else: the workload of the skinny kernel's ncu summary."""
    import torch
    import dit_tq2_g128_gb300 as tq2

    m = args.skinny
    p = tq2_synth.skinny(m)
    l2 = int(getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 126 * 2 ** 20))
    wb = tq2.tq2_soa_bytes(p.n, p.k)
    c = max(2, -(-2 * l2 // wb) + 1)
    w0 = tq2.upload_weight(p.w_aos, p.n, p.k)
    ws = [w0] + [w0.clone() for _ in range(c - 1)]
    x = torch.from_numpy(p.x).cuda()
    out = torch.empty((p.m, p.n), dtype=torch.float32, device="cuda")
    def step(i):
        tq2.tq2_gemm(ws[i % c], x, None, out, p.m, p.n, p.k)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    # the calls captured in one CUDA graph (as in the suite): an eager Python
    # loop would time the host's dispatch rate instead of the kernel
    steps = max(args.steps, 1)
    g = graph_of(step, steps, torch)
    g.replay()
    torch.cuda.synchronize()
    t = statistics.median(time_graph(g, torch, reps=3)) / steps
    assert tq2.tq2_device_status() == tq2.TQ2_OK
    return {"workload": f"skinny_m{m}_k4096_n4096", "kernel": tq2.KERNEL_NAMES[tq2.tq2_select_kernel(p.m, p.n, p.k)],
            "steps": args.steps, "warmup": args.warmup, "us_per_call": round(t * 1e6, 2),
            "weight_GBps": round(wb / t / 1e9, 1), "copies": c,
            "method": "steps captured in one CUDA graph, median of 3 replays"}


def run_suite(args):
    import torch
    import oracle
    import dit_tq2_g128_gb300 as tq2

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    l2 = int(getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 126 * 2 ** 20))
    rows_out = []

    def timed(fn, steps):
        for i in range(3):
            fn(i)
        torch.cuda.synchronize()
        g = graph_of(fn, steps, torch)
        g.replay()
        torch.cuda.synchronize()
        ts = []
        for _ in range(3):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) / 1e3 / steps)
        return statistics.median(ts)

    def parity(out, p, rows):
        """max |gpu - oracle| / sum|x w| over the sampled elements; min row cosine; oracle seconds."""
        t0 = time.perf_counter()
        ref, scale = oracle.matmul(p.w_aos, p.x, p.residual, n=p.n, k=p.k, rows=rows)
        t_or = time.perf_counter() - t0
        got = np.asarray(out, dtype=np.float64).reshape(-1, p.n)[rows]
        rel = float(np.max(np.abs(got - ref) / np.maximum(scale, 1e-30)))
        num = np.sum(got * ref, axis=1)
        den = np.linalg.norm(got, axis=1) * np.linalg.norm(ref, axis=1)
        cos = float(np.min(np.where(den > 0, num / np.where(den > 0, den, 1), 1.0)))
        return rel, cos, t_or

    def sample(m, count):
        return np.unique(np.concatenate([[0, m - 1], np.random.default_rng(1).integers(0, m, count)]))

    def one(name, p, kernel_entry, steps, sample_rows):
        wbytes = tq2.tq2_soa_bytes(p.n, p.k)
        per = wbytes + p.m * p.k * 4 + p.m * p.n * 4
        c = max(2, -(-2 * l2 // per) + 1) if per < l2 else 1
        w0 = tq2.upload_weight(p.w_aos, p.n, p.k)
        ws = [w0] + [w0.clone() for _ in range(c - 1)]
        x = torch.from_numpy(p.x).to(device)
        r = None if p.residual is None else torch.from_numpy(p.residual).to(device)
        outs = [torch.empty((p.m, p.n), dtype=torch.float32, device=device) for _ in range(c)]

        def fn(i):
            if kernel_entry == "gemv":
                tq2.tq2_gemv(ws[i % c], x, r, outs[i % c], p.n, p.k)
            else:
                tq2.tq2_gemm(ws[i % c], x, r, outs[i % c], p.m, p.n, p.k)

        t = timed(fn, steps)
        fn(0)
        torch.cuda.synchronize()
        assert tq2.tq2_device_status() == tq2.TQ2_OK
        rows = sample(p.m, sample_rows) if p.m > sample_rows else np.arange(p.m)
        rel, cos, t_or = parity(outs[0].cpu().numpy(), p, rows)
        kern = tq2.KERNEL_NAMES[tq2.tq2_select_kernel(p.m, p.n, p.k)]
        rec = {"config": name, "m": p.m, "n": p.n, "k": p.k, "kernel": kern,
               "us_per_call": round(t * 1e6, 2), "weight_GBps": round(wbytes / t / 1e9, 1),
               "TFLOPs": round(2.0 * p.m * p.n * p.k / t / 1e12, 2),
               "max_err_over_sum_abs_xw": rel, "min_row_cos": cos,
               "parity_rows": int(rows.size),
               "oracle_s_full_extrapolated": round(t_or * p.m / rows.size, 3),
               "l2": f"{c} rotating weight copies" if c > 1 else "inputs larger than L2"}
        del ws, outs, x, r, w0
        torch.cuda.empty_cache()
        return rec, t

    def one_swiglu(name, p, f, steps, sample_rows, resident=False):
        """Fused gate/up + SwiGLU (2f weight rows, out [m, f]); error reported
        relative to the bound's scale 1.1*S_g*|u| + |silu(g)|*S_u (S = sum|xw|).
        resident: through tq2_gate_up_swiglu_resident (weights uploaded and
        synchronised before the timed calls: its contract holds)."""
        fn = tq2.tq2_gate_up_swiglu_resident if resident else tq2.tq2_gate_up_swiglu
        wbytes = tq2.tq2_soa_bytes(p.n, p.k)
        per = wbytes + p.m * p.k * 4 + p.m * f * 4
        c = max(2, -(-2 * l2 // per) + 1) if per < l2 else 1
        w0 = tq2.upload_weight(p.w_aos, p.n, p.k)
        ws = [w0] + [w0.clone() for _ in range(c - 1)]
        x = torch.from_numpy(p.x).to(device)
        outs = [torch.empty((p.m, f), dtype=torch.float32, device=device) for _ in range(c)]
        torch.cuda.synchronize()
        t = timed(lambda i: fn(ws[i % c], x, outs[i % c], p.m, f, p.k), steps)
        fn(ws[0], x, outs[0], p.m, f, p.k)
        torch.cuda.synchronize()
        assert tq2.tq2_device_status() == tq2.TQ2_OK
        rows = sample(p.m, sample_rows) if p.m > sample_rows else np.arange(p.m)
        t0 = time.perf_counter()
        h, g, u, sg, su = oracle.swiglu(p.w_aos, p.x, f=f, k=p.k, rows=rows)
        t_or = time.perf_counter() - t0
        got = outs[0].cpu().numpy().astype(np.float64)[rows]
        scale = 1.1 * sg * np.abs(u) + np.abs(oracle.silu(g)) * su
        rel = float(np.max(np.abs(got - h) / np.maximum(scale, 1e-30)))
        rec = {"config": name, "m": p.m, "f": f, "k": p.k,
               "entry": "tq2_gate_up_swiglu_resident" if resident else "tq2_gate_up_swiglu",
               "us_per_call": round(t * 1e6, 2), "weight_GBps": round(wbytes / t / 1e9, 1),
               "TFLOPs": round(2.0 * p.m * p.n * p.k / t / 1e12, 2),
               "max_err_over_bound_scale": rel, "parity_rows": int(rows.size),
               "oracle_s_full_extrapolated": round(t_or * p.m / rows.size, 3),
               "l2": f"{c} rotating weight copies" if c > 1 else "inputs larger than L2"}
        del ws, outs, x, w0
        torch.cuda.empty_cache()
        return rec

    def host_act16(a):
        """binary16 activation layout made on the host (numpy rounding, then
        element i of each 16-group at 2i or 2(i-8)+1)."""
        a16 = np.asarray(a, dtype=np.float32).astype(np.float16)
        kk = a16.shape[1]
        i = np.arange(kk) % 16
        pos = (np.arange(kk) - i) + np.where(i < 8, 2 * i, 2 * (i - 8) + 1)
        out = np.empty_like(a16)
        out[:, pos] = a16
        return out, a16.astype(np.float32)

    def one_act16(name, p, steps, sample_rows):
        """tq2_gemm_act16: binary16 activations in and out; error against the oracle
        on the binary16 input values, relative to sum|xw| after removing the
        result's own rounding (2^-11 |ref|)."""
        wbytes = tq2.tq2_soa_bytes(p.n, p.k)
        per = wbytes + p.m * p.k * 2 + p.m * p.n * 2
        c = max(2, -(-2 * l2 // per) + 1) if per < l2 else 1
        w0 = tq2.upload_weight(p.w_aos, p.n, p.k)
        ws = [w0] + [w0.clone() for _ in range(c - 1)]
        x16, x32 = host_act16(p.x)
        r16, r32 = host_act16(p.residual) if p.residual is not None else (None, None)
        xd = torch.from_numpy(x16).to(device)
        rd = None if r16 is None else torch.from_numpy(r16).to(device)
        outs = [torch.empty((p.m, p.n), dtype=torch.float16, device=device) for _ in range(c)]
        t = timed(lambda i: tq2.tq2_gemm_act16(ws[i % c], xd, rd, outs[i % c], p.m, p.n, p.k), steps)
        tq2.tq2_gemm_act16(ws[0], xd, rd, outs[0], p.m, p.n, p.k)
        torch.cuda.synchronize()
        assert tq2.tq2_device_status() == tq2.TQ2_OK
        rows = sample(p.m, sample_rows) if p.m > sample_rows else np.arange(p.m)
        t0 = time.perf_counter()
        ref, scale = oracle.matmul(p.w_aos, x32, r32, n=p.n, k=p.k, rows=rows)
        t_or = time.perf_counter() - t0
        got16 = outs[0].cpu().numpy()
        i = np.arange(p.n) % 16
        pos = (np.arange(p.n) - i) + np.where(i < 8, 2 * i, 2 * (i - 8) + 1)
        got = got16[:, pos].astype(np.float64)[rows]
        err = np.maximum(np.abs(got - ref) - 2.0 ** -11 * np.abs(ref), 0.0)
        rel = float(np.max(err / np.maximum(scale, 1e-30)))
        num = np.sum(got * ref, axis=1)
        den = np.linalg.norm(got, axis=1) * np.linalg.norm(ref, axis=1)
        cos = float(np.min(np.where(den > 0, num / np.where(den > 0, den, 1), 1.0)))
        rec = {"config": name, "m": p.m, "n": p.n, "k": p.k, "entry": "tq2_gemm_act16",
               "us_per_call": round(t * 1e6, 2), "TFLOPs": round(2.0 * p.m * p.n * p.k / t / 1e12, 2),
               "max_err_over_sum_abs_xw": rel, "min_row_cos": cos, "parity_rows": int(rows.size),
               "oracle_s_full_extrapolated": round(t_or * p.m / rows.size, 3),
               "l2": f"{c} rotating weight copies" if c > 1 else "inputs larger than L2"}
        del ws, outs, xd, rd, w0
        torch.cuda.empty_cache()
        return rec, t

    rows_out.append(one("1 small", tq2_synth.small(), "gemm", 50, 8)[0])
    rows_out.append(one("2a decode gate/up", tq2_synth.decode_gate_up(), "gemv", 200, 1)[0])
    rows_out.append(one("2b decode down + residual", tq2_synth.decode_down(), "gemv", 200, 1)[0])
    # the same gate/up weight with the activation fused (out: 6144 values)
    rows_out.append(one_swiglu("2a fused gate/up + SwiGLU", tq2_synth.decode_gate_up(), 6144, 200, 1))
    rows_out.append(one_swiglu("2a fused gate/up + SwiGLU, resident weights", tq2_synth.decode_gate_up(), 6144,
                               200, 1, resident=True))
    for m in tq2_synth.SKINNY_MS:
        rows_out.append(one(f"3 skinny m={m}", tq2_synth.skinny(m), "gemv" if m == 1 else "gemm",
                            100, 16)[0])
    for n in tq2_synth.DIT_NS:
        rows_out.append(one(f"4 dit n={n}", tq2_synth.dit(n), "gemm", 10, 16)[0])
    # a DiT-sized fused gate/up: M=1536, 2f = 12288 rows, K=3072 (config 4's x and weights)
    rows_out.append(one_swiglu("4 fused gate/up + SwiGLU m=1536 f=6144", tq2_synth.dit(12288), 6144, 10, 16))
    # config 5: the 100 layers one after another (each timed on its own, summed)
    tot_t, tot_f, worst, cmin, t_or5 = 0.0, 0.0, 0.0, 1.0, 0.0
    for li in range(len(tq2_synth.DIT_FORWARD_SHAPES)):
        p = tq2_synth.dit_forward_layer(li)
        rec, t = one(f"5 layer {li}", p, "gemm", 3, 2)
        tot_t += t
        tot_f += 2.0 * p.m * p.n * p.k
        worst = max(worst, rec["max_err_over_sum_abs_xw"])
        cmin = min(cmin, rec["min_row_cos"])
        t_or5 += rec["oracle_s_full_extrapolated"]
    rows_out.append({"config": "5 dit forward (100 layers, M=4096)", "kernel": "tc",
                     "us_total": round(tot_t * 1e6, 1), "TFLOPs": round(tot_f / tot_t / 1e12, 2),
                     "max_err_over_sum_abs_xw": worst, "min_row_cos": cmin,
                     "parity_rows": "2 sampled rows per layer",
                     "oracle_s_full_extrapolated": round(t_or5, 1)})
    # configs 4 and 5 with binary16 activations in and out (no pre-pass, half the output bytes)
    for n in tq2_synth.DIT_NS:
        rows_out.append(one_act16(f"4 dit n={n} act16", tq2_synth.dit(n), 10, 16)[0])
    tot_t, tot_f, worst, cmin = 0.0, 0.0, 0.0, 1.0
    for li in range(len(tq2_synth.DIT_FORWARD_SHAPES)):
        p = tq2_synth.dit_forward_layer(li)
        rec, t = one_act16(f"5 layer {li} act16", p, 3, 2)
        tot_t += t
        tot_f += 2.0 * p.m * p.n * p.k
        worst = max(worst, rec["max_err_over_sum_abs_xw"])
        cmin = min(cmin, rec["min_row_cos"])
    rows_out.append({"config": "5 dit forward act16 (100 layers, M=4096, binary16 activations)",
                     "entry": "tq2_gemm_act16", "us_total": round(tot_t * 1e6, 1),
                     "TFLOPs": round(tot_f / tot_t / 1e12, 2), "max_err_over_sum_abs_xw": worst,
                     "min_row_cos": cmin, "parity_rows": "2 sampled rows per layer"})
    # DiT joint attention at the FLUX.2 shape: 24 heads x 128, 4096 tokens (4 H S^2 D flops)
    ha, sa, da = 24, 4096, 128
    rng = np.random.default_rng(24)
    qa, ka, va = (rng.standard_normal((ha, sa, da)).astype(np.float32) for _ in range(3))
    qd, kd, vd = (torch.from_numpy(a).to(device) for a in (qa, ka, va))
    oa = torch.empty((sa, ha * da), dtype=torch.float32, device=device)
    t = timed(lambda i: tq2.tq2_attention_f32(qd, kd, vd, oa, ha, sa, da), 5)
    tq2.tq2_attention_f32(qd, kd, vd, oa, ha, sa, da)
    torch.cuda.synchronize()
    assert tq2.tq2_device_status() == tq2.TQ2_OK
    rows = sample(sa, 16)
    t0 = time.perf_counter()
    ref, absv = oracle.attention(qa, ka, va, heads=ha, seq=sa, dim=da, rows=rows)
    t_or = time.perf_counter() - t0
    got = oa.cpu().numpy().astype(np.float64)[rows]
    num = np.sum(got * ref, axis=1)
    den = np.linalg.norm(got, axis=1) * np.linalg.norm(ref, axis=1)
    rows_out.append({"config": "DiT joint attention 24 x 4096 x 128", "entry": "tq2_attention_f32",
                     "us_per_call": round(t * 1e6, 2), "TFLOPs": round(4.0 * ha * sa * sa * da / t / 1e12, 2),
                     "max_err_over_sum_p_abs_v": float(np.max(np.abs(got - ref) / np.maximum(absv, 1e-30))),
                     "min_row_cos": float(np.min(num / den)), "parity_rows": int(rows.size),
                     "oracle_s_full_extrapolated": round(t_or * sa / rows.size, 3)})
    del qd, kd, vd, oa
    torch.cuda.empty_cache()
    # the encoder (f32 -> blocks) on the largest DiT weight: f32 bytes read per second
    n, k = 12288, 3072
    wf = torch.randn((n, k), device=device) * 0.02
    aos = torch.empty(tq2.tq2_soa_bytes(n, k), dtype=torch.uint8, device=device)
    t = timed(lambda i: tq2.tq2_quantize_f32(wf, aos, n, k), 10)
    rows_out.append({"config": "encoder f32 -> blocks (12288 x 3072)", "us_per_call": round(t * 1e6, 2),
                     "f32_GBps": round(n * k * 4 / t / 1e9, 1),
                     "bytes_GBps": round((n * k * 4 + tq2.tq2_soa_bytes(n, k)) / t / 1e9, 1)})
    return {"suite": rows_out, "oracle_threads": oracle.threads()}


# ---------------------------------------------------------------------------
# CPU oracle (cpu_baseline leg, and the --impl reference arm)


def oracle_gemv_rate(p, seconds):
    """Weight GB/s of the oracle on the decode GEMV; runs whole calls for about `seconds`."""
    import oracle
    wbytes = p.w_aos.size
    oracle.matmul(p.w_aos[:64], p.x, n=64, k=p.k)  # build + warm
    t0 = time.perf_counter()
    calls = 0
    while True:
        oracle.matmul(p.w_aos, p.x, n=p.n, k=p.k)
        calls += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return calls * wbytes / el / 1e9, calls, el, oracle.threads()


def run_cpu_configs():
    """The CPU oracle (f64 naive loop, OpenMP over output rows) on the small and
    skinny configurations, one whole call each, at one thread and at all of the
    host's threads: the reported CPU baseline of those rows."""
    import oracle
    probs = [("1 small", tq2_synth.small()), ("2a decode gate/up", tq2_synth.decode_gate_up()),
             ("2b decode down + residual", tq2_synth.decode_down())]
    probs += [(f"3 skinny m={m}", tq2_synth.skinny(m)) for m in tq2_synth.SKINNY_MS]
    full = oracle.threads()
    oracle.matmul(probs[0][1].w_aos, probs[0][1].x, n=probs[0][1].n, k=probs[0][1].k)  # build + warm
    rows = []
    for name, p in probs:
        rec = {"config": name, "m": p.m, "n": p.n, "k": p.k}
        for t in (1, full):
            oracle.set_threads(t)
            t0 = time.perf_counter()
            oracle.matmul(p.w_aos, p.x, p.residual, n=p.n, k=p.k)
            rec[f"seconds_{t}_threads"] = round(time.perf_counter() - t0, 4)
        rows.append(rec)
    oracle.set_threads(full)
    return {"cpu_oracle": rows, "host_threads": full, "cpu": platform.machine()}


def run_cpu_full():
    """The CPU oracle (f64 naive loop, OpenMP over output rows) on the DiT
    configurations in full, every output element: M=1536 at each N, then the
    100 layers of the forward set at M=4096 one after another.  Input
    generation is outside the timed calls."""
    import oracle
    full = oracle.threads()
    p0 = tq2_synth.small()
    oracle.matmul(p0.w_aos, p0.x, n=p0.n, k=p0.k)  # build + warm
    rows = []
    for n in tq2_synth.DIT_NS:
        p = tq2_synth.dit(n)
        t0 = time.perf_counter()
        oracle.matmul(p.w_aos, p.x, p.residual, n=p.n, k=p.k)
        el = time.perf_counter() - t0
        rows.append({"config": f"4 dit m=1536 n={n}", "seconds": round(el, 3),
                     "GFLOP": round(2.0 * p.m * p.n * p.k / 1e9, 1), "GFLOPs": round(2.0 * p.m * p.n * p.k / el / 1e9, 2)})
        print(json.dumps(rows[-1]), flush=True)
    tot, flops, per = 0.0, 0.0, []
    for li in range(len(tq2_synth.DIT_FORWARD_SHAPES)):
        p = tq2_synth.dit_forward_layer(li)
        t0 = time.perf_counter()
        oracle.matmul(p.w_aos, p.x, p.residual, n=p.n, k=p.k)
        el = time.perf_counter() - t0
        tot += el
        flops += 2.0 * p.m * p.n * p.k
        per.append(round(el, 2))
    rows.append({"config": "5 dit forward, 100 layers at M=4096 (every element)", "seconds": round(tot, 1),
                 "TFLOP": round(flops / 1e12, 2), "GFLOPs": round(flops / tot / 1e9, 2), "per_layer_s": per})
    return {"cpu_oracle_full": rows, "host_threads": full, "cpu": platform.machine()}


def run_reference(args):
    """The reference arm: the CPU oracle on the decode GEMV workload, whole calls."""
    import oracle
    p = tq2_synth.decode_gate_up()
    wbytes = p.w_aos.size
    for _ in range(args.warmup):
        oracle.matmul(p.w_aos, p.x, n=p.n, k=p.k)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.matmul(p.w_aos, p.x, n=p.n, k=p.k)
    el = time.perf_counter() - t0
    v = args.steps * wbytes / el / 1e9
    cores = oracle.threads()
    return {
        "metric": METRIC, "value": round(v, 4), "unit": "GB/s (TQ2 weight bytes, M=1 GEMV)",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (same seeded workload)",
        "config": dict(GEMV_CONFIG),
        "impl": "reference",
        "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} full GEMV calls (12288x4096), double precision"},
        "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    world, rank = world_from_env()
    if args.impl == "reference":
        # the oracle runs on the host: under a multi-process launch rank 0
        # alone runs and prints it, the other ranks leave without work
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1 or args.gpus != 1:
        # refused before anything touches a GPU
        sys.stderr.write(SINGLE_GPU_ONLY + f" (asked for --gpus {args.gpus}, WORLD_SIZE {world})\n")
        sys.exit(2)
    if args.suite:
        print(json.dumps(run_suite(args)), flush=True)
        return
    if args.attention:
        print(json.dumps(run_attention_only(args)), flush=True)
        return
    if args.skinny:
        print(json.dumps(run_skinny_only(args)), flush=True)
        return
    if args.encoder:
        print(json.dumps(run_encoder_only(args)), flush=True)
        return
    if args.cpu_configs:
        print(json.dumps(run_cpu_configs()), flush=True)
        return
    if args.cpu_full:
        print(json.dumps(run_cpu_full()), flush=True)
        return
    line = run_ours(args)
    if not args.no_cpu:
        p = tq2_synth.decode_gate_up()
        v, calls, el, cores = oracle_gemv_rate(p, 10.0)
        line["cpu_baseline"] = {"value": round(v, 4), "unit": "GB/s", "cores": cores,
                                "kind": "oracle",
                                "sample": f"{calls} full decode GEMV calls in {el:.1f} s "
                                          "(double precision, OpenMP over output rows)"}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
