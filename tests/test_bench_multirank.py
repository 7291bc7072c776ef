"""Host logic of bench.py with more than one rank, on CPU over gloo (world size 2).

With N ranks each GPU forwards its own batch (replicas, no collective on the
data path); the only cross-rank steps are the barrier, the max over ranks of
the timed region and the whole-job rate.  These run here on two CPU
processes.
"""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402
import workloads  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        my_ms = 100.0 + 50.0 * rank            # rank 1 is the slower one
        slowest = bench.max_over_ranks(my_ms, dist, "cpu")
        cfg = workloads.get_config("small")
        rate = bench.job_rate(world, cfg.batch * cfg.seq, 10, slowest)
        toks = bench.rank_tokens(cfg, rank)
        out[rank] = (slowest, rate, int(toks.sum()), toks.shape)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_takes_the_slowest_rank_and_sums_the_work():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
        codes = [p.exitcode for p in procs]
        res = dict(out)
    assert codes == [0, 0], codes
    cfg = workloads.get_config("small")
    for r in range(world):
        slowest, rate, _, shape = res[r]
        assert slowest == 150.0                    # max over ranks, identical on both
        assert shape == (cfg.batch, cfg.seq)
        assert rate == pytest.approx(world * cfg.batch * cfg.seq * 10 / 0.150)
    assert res[0][2] != res[1][2]                  # independent batches per replica


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    assert bench.job_rate(1, 1000, 4, 2000.0) == pytest.approx(2000.0)
    t0 = bench.rank_tokens(workloads.get_config("tiny"), 0)
    assert np.array_equal(t0, workloads.make_tokens(workloads.get_config("tiny")))


def test_reference_arm_runs_on_rank_zero_only(capsys):
    """bench.py --impl reference: rank 0 times the oracle and prints one JSON line
    with the reference fields; any other rank returns without work or output."""
    import argparse
    import json
    args = argparse.Namespace(config="tiny", steps=1, warmup=0, gpus=2)
    bench.run_reference(args, world=2, rank=1)
    assert capsys.readouterr().out == ""
    bench.run_reference(args, world=2, rank=0)
    lines = [l for l in capsys.readouterr().out.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0 and line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"],
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
