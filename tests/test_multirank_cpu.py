"""The multi-process path of the benchmark on CPU (gloo, world size 2): the
attention shards by (batch, head) with no exchange, so N processes run N
independent streams; the job's time is the slowest rank's (a MAX all-reduce)
and its rate counts every rank's chunks.  The reference arm runs on rank 0
only."""

import json
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out_dir):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        # rank r was slower on the first timing and faster on the second
        ms = bench.max_over_ranks(dist, [100.0 + 10 * rank, 50.0 - 5 * rank], "cpu")
        rate = bench.whole_job_rate(20, world, ms[0])
        dist.barrier()
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"ms": ms, "rate": rate}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    import tempfile

    with tempfile.TemporaryDirectory() as d:
        mp.start_processes(_rank, args=(2, _free_port(), d), nprocs=2, join=True, start_method="spawn")
        res = [json.load(open(os.path.join(d, f"r{r}.json"))) for r in range(2)]
    for r in res:
        assert r["ms"] == [110.0, 50.0]  # every rank sees the max over ranks
        assert r["rate"] == pytest.approx(20 * 2 / 0.110)


def test_single_process_is_identity():
    assert bench.max_over_ranks(None, [3.0, 4.5], "cpu") == [3.0, 4.5]
    assert bench.whole_job_rate(10, 1, 500.0) == pytest.approx(20.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = bench.argparse.Namespace(steps=1, warmup=0)
    assert bench.run_reference(args) is None  # returns at once, no oracle work
    assert capsys.readouterr().out == ""
    assert bench._dist() == (2, 1, 0)
