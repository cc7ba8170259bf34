"""The benchmark's multi-rank host logic as two gloo ranks on CPU (no GPU).

`bench.py --gpus N` runs one independent problem per rank (weak scaling): a
barrier and a max over ranks bracket the timing, the whole-job rate counts
every rank's units over the slowest rank's time, and the reference arm runs on
rank 0 only.  These are exactly the pieces exercised here, with the process
group forced onto gloo."""

import json
import os
import socket

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _load_bench():
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _worker(rank, world, port, outdir):
    # CPU only: hide any GPU before torch looks for one, so the group is gloo
    os.environ["CUDA_VISIBLE_DEVICES"] = ""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    bench = _load_bench()
    w, r, local, pg = bench.dist_setup(world)
    backend = pg.get_backend()
    t = bench.max_over_ranks(0.25 * (rank + 1), pg, "cpu")  # rank 1 is the slow one
    bench.barrier(pg)
    rate = bench.whole_job_rate(w, 1000.0, t)

    class Args:
        steps = 1
        warmup = 0

    ref = bench.run_reference(Args, w, r) if r != 0 else "rank 0 not run here"
    with open(os.path.join(outdir, f"r{rank}.json"), "w") as f:
        json.dump({"world": w, "rank": r, "local": local, "backend": backend, "t": t,
                   "rate": rate, "ref": ref}, f)
    pg.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks(tmp_path):
    mp.spawn(_worker, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(2)]
    for r, d in enumerate(res):
        assert d["world"] == 2 and d["rank"] == r and d["local"] == r
        assert d["backend"] == "gloo"
        assert d["t"] == 0.5                      # max over ranks, seen by both
        assert d["rate"] == 2 * 1000.0 / 0.5      # all ranks' units over the slowest time
    assert res[1]["ref"] is None                  # the reference arm prints on rank 0 only


def test_single_rank_has_no_group():
    bench = _load_bench()
    old = {k: os.environ.pop(k, None) for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    try:
        world, rank, local, pg = bench.dist_setup(1)
    finally:
        for k, v in old.items():
            if v is not None:
                os.environ[k] = v
    assert (world, rank, local, pg) == (1, 0, 0, None)
    assert bench.max_over_ranks(1.5, None, "cpu") == 1.5
    assert bench.whole_job_rate(1, 10.0, 2.0) == 5.0
