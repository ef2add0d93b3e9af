"""The benchmark's multi-process path on CPU (gloo, world size 2): every rank
runs an independent replica, the timed region is bracketed by barriers, and
the job time is the maximum over ranks -- the same helpers bench.py uses
under torchrun with NCCL on GPUs."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q):
    sys.path.insert(0, ROOT)
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import bench
    w, r, lr = bench.dist_env()
    dist = bench.init_dist(w, "gloo")
    bench.barrier(dist)
    got = bench.max_over_ranks(dist, 10.0 * (rank + 1))
    bench.barrier(dist)
    q.put((rank, w, r, got))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [x[0] for x in res] == [0, 1]
    assert all(x[1] == 2 for x in res)
    assert all(x[3] == 20.0 for x in res)  # every rank sees the slowest rank's time


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.init_dist(1, "gloo") is None
    assert bench.max_over_ranks(None, 3.5) == 3.5


def test_reference_arm_other_ranks_do_no_work(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    args = bench.argparse.Namespace(workload="tiny", steps=1, warmup=3, gpus=2)
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""


@pytest.mark.parametrize("steps,budget", [(3, 30.0), (400, 0.5)], ids=["row-mode", "key-mode"])
def test_reference_arm_line_and_bounded_time(monkeypatch, capsys, steps, budget):
    """Rank 0 prints one contract line with impl reference; every step is
    sized from the run's budget (whole rows when a step can afford a wave of
    them, else one row over a bounded number of keys), so K x ms_per_step is
    the measured time of the timed steps and the run stays near the budget."""
    import json
    import time
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "1")
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setattr(bench, "REFERENCE_BUDGET_S", budget)
    args = bench.argparse.Namespace(workload="tiny", steps=steps, warmup=3, gpus=1)
    t0 = time.perf_counter()
    assert bench.run_reference(args) == 0
    wall = time.perf_counter() - t0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["steps"] == steps and line["warmup"] == 3
    assert line["value"] > 0 and line["unit"] == "steps/s" and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert steps * line["ms_per_step"] / 1e3 <= wall
    if steps == 3:
        assert "attention rows per timed step" in line["step_unit"]
    else:
        assert "bounded number of its keys" in line["step_unit"] and line["cpu_baseline"]["cores"] == 1


def test_verify_algorithmic_bytes_counts_the_cache_layout():
    """The roofline's bytes, counted from the oracle's cache arrays: every
    visible key's K and V codes and the scales that cover it, Q in, O out,
    the page-table entries used and the lengths."""
    sys.path.insert(0, ROOT)
    import numpy as np

    import bench
    import oracle
    import synth
    for name in ("multi_lane", "int4_12slot", "long_context", "plain_decode", "tiny"):
        spec = synth.WORKLOADS[name]
        lens = synth.context_lengths(spec)
        c = oracle.Cache(spec.kv_dtype, 1, spec.num_kv_heads)  # one page: its arrays give the sizes
        want = 0
        for L in lens:
            n_tok = int(L) + spec.window
            n_pages = (n_tok + 63) // 64
            per_token = (c.k_codes.nbytes + c.v_codes.nbytes) // 64
            if spec.kv_dtype == synth.KV_FP8:  # one scale per page and head
                want += n_tok * per_token + n_pages * (c.k_scales.nbytes + c.v_scales.nbytes)
            else:  # scales per token
                want += n_tok * (per_token + (c.k_scales.nbytes + c.v_scales.nbytes) // 64)
            want += n_pages * 4 + 4
        want += 2 * len(lens) * spec.window * spec.num_q_heads * 128 * 2
        assert bench.verify_algorithmic_bytes(spec, lens) == want, name
