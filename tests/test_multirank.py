"""The multi-rank path of bench.py on CPU: two gloo ranks, as `torchrun
--nproc-per-node 2 bench.py` would start them (one rank per GPU there).  The
matrices are independent, so ranks exchange nothing on the data path: each
draws and preconditions its own stack (weak scaling) and the job's time is the
slowest rank's.  This covers that host logic: the max over ranks, the
whole-job rate, disjoint draws per rank and rank-0-only output of the
reference arm."""
import os
import socket

import numpy as np
import pytest


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q):
    import torch
    import torch.distributed as dist
    import bench
    from workloads import synth
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank's elapsed time differs; every rank must see the slowest
        elapsed = bench.max_over_ranks(1.5 + rank, dist, torch.device("cpu"))
        rate = bench.job_rate(world, 3, elapsed)
        # each rank draws its own gradient batch (small stand-in of the stack recipe)
        w = synth.workload(1)
        rng = synth.rng_for(w.index, bench.rank_step_seed(rank, 0), 0)
        g = synth.gradient(64, 32, w.alpha, rng, synth.F32)
        digest = torch.tensor(g[:4, :4].astype(np.float64).ravel())
        gathered = [torch.zeros_like(digest) for _ in range(world)]
        dist.all_gather(gathered, digest)
        q.put((rank, elapsed, rate, [x.tolist() for x in gathered]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_like_the_bench():
    import torch.multiprocessing as mp
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    for rank, elapsed, rate, gathered in res:
        assert elapsed == 2.5                       # the slowest rank's time, on every rank
        assert rate == pytest.approx(world * 3 / 2.5)
        assert gathered[0] != gathered[1]           # disjoint draws: ranks process different units
    assert res[0][3] == res[1][3]                   # and all ranks agree on what was drawn


def test_reference_arm_prints_on_rank_zero_only(capsys, monkeypatch):
    import argparse
    import bench
    monkeypatch.setenv("RANK", "1")
    args = argparse.Namespace(workload=0, power=None, warmup=0, steps=1, gpus=2)
    bench.run_reference(args)
    assert capsys.readouterr().out == ""


def test_rank_seeds_are_disjoint():
    import bench
    seeds = {bench.rank_step_seed(r, s) for r in range(8) for s in range(10)}
    assert len(seeds) == 80


def test_reference_arm_json_line(capsys, monkeypatch):
    """The reference arm (the float64 oracle) prints one JSON line with the
    fields the benchmark contract names."""
    import argparse
    import json
    import bench
    monkeypatch.setenv("RANK", "0")
    args = argparse.Namespace(workload=0, power=None, warmup=1, steps=2, gpus=1, opt=[])
    bench.run_reference(args)
    lines = [l for l in capsys.readouterr().out.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["value"] > 0 and d["unit"] == "preconditioner steps/s" and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 1 and d["n_gpus"] == 1
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == "single-256x128"
    # the same config object as the main arm's line for the same arguments
    assert d["config"] == bench.workload_config(bench.synth_workload(0), -0.25, {})


def test_reference_arm_reports_the_steps_it_ran(capsys, monkeypatch):
    """When whole oracle steps do not fit the arm's time budget, the line says
    how many steps it actually ran (at least one, no warm-up) next to the
    requested counts, and ms_per_step is the measured whole-step time."""
    import argparse
    import json
    import bench
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setattr(bench, "REFERENCE_BUDGET_S", 0.0)
    args = argparse.Namespace(workload=0, power=None, warmup=3, steps=5, gpus=1, opt=[])
    bench.run_reference(args)
    d = json.loads([l for l in capsys.readouterr().out.splitlines() if l.strip()][0])
    assert d["steps"] == 1 and d["warmup"] == 0
    assert d["requested"] == {"steps": 5, "warmup": 3}
    assert d["extrapolated"] is False
    assert abs(d["ms_per_step"] * d["value"] - 1e3) < 1e-6 * 1e3
