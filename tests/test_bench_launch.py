"""How bench.py treats requests for more than one GPU (no GPU needed).

The library runs on one GPU only (its tensor-core kernels copy shared x tiles
between the two CTAs of a cluster, which is offered for single-GPU calls
only), so the benchmark refuses `--gpus N > 1` and multi-process launches
before anything touches a GPU.  The reference arm (the CPU oracle) runs on
rank 0 of a multi-process launch and the other ranks leave without work."""

import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(args, env_extra=None, timeout=300):
    env = dict(os.environ)
    env["CUDA_VISIBLE_DEVICES"] = ""  # nothing here may reach a GPU
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        env.pop(k, None)
    env.update(env_extra or {})
    t0 = time.time()
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=timeout)
    return r, time.time() - t0


def test_more_than_one_gpu_is_refused():
    r, _ = _bench(["--gpus", "2", "--steps", "1", "--warmup", "0"])
    assert r.returncode == 2
    assert "one GPU only" in r.stderr
    assert r.stdout == ""


def test_multi_process_launch_is_refused_on_every_rank():
    for rank in ("0", "1"):
        r, _ = _bench(["--gpus", "1"], {"WORLD_SIZE": "2", "RANK": rank, "LOCAL_RANK": rank})
        assert r.returncode == 2, r.stderr
        assert "one GPU only" in r.stderr and r.stdout == ""


def test_reference_arm_rank0_only():
    # rank 1 of a two-process launch: no work, no output, success
    r, el = _bench(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"],
                   {"WORLD_SIZE": "2", "RANK": "1", "LOCAL_RANK": "1"})
    assert r.returncode == 0 and r.stdout.strip() == ""
    # rank 0 runs the oracle once and prints the reference line
    r, _ = _bench(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"],
                  {"WORLD_SIZE": "2", "RANK": "0", "LOCAL_RANK": "0"})
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["config"]["workload"] == "decode_gemv_m1_k4096_n12288"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_both_arms_name_the_same_config():
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    import tq2_synth
    p = tq2_synth.decode_gate_up()
    cfg = bench.GEMV_CONFIG
    assert (cfg["m"], cfg["k"], cfg["n"]) == (p.m, p.k, p.n)
    assert cfg["weight_bytes"] == p.w_aos.size
