"""The replica path of bench.py on CPU: two gloo ranks, no GPU.

Every rank runs its own batch (the path shards by sequence with no exchange
step), the job's time is the slowest rank's, and the whole-job throughput counts
the tokens of every rank.
"""
import argparse
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    mine = 100.0 + 50.0 * rank  # rank 1 is the slower one
    got = bench.max_over_ranks(mine, world)
    value = bench.job_value(256, world, 10, got)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, got, value))


def test_replicas_take_the_slowest_rank_and_count_every_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    assert [r for r, _, _ in res] == [0, 1]
    for _, got, value in res:
        assert got == 150.0
        assert value == pytest.approx(256 * 2 * 10 / 0.150)


def test_single_rank_is_a_no_op():
    import bench
    assert bench.max_over_ranks(42.0, 1) == 42.0
    assert bench.job_value(64, 1, 5, 2.0) == pytest.approx(64 * 5 / 0.002)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    args = argparse.Namespace(workload=0, steps=1, warmup=3, cpu_budget=1.0)
    assert bench.run_reference(args) is None
    assert capsys.readouterr().out == ""


def test_reference_arm_prints_one_contract_line(monkeypatch, capsys):
    # --impl reference on the tiny workload: the oracle on the host's cores, one JSON
    # line with the metric, a cpu_baseline naming the threads it used, and an e2e
    # entry without transfers.
    import json
    import bench
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.delenv("RANK", raising=False)
    args = argparse.Namespace(workload=0, steps=4, warmup=3, cpu_budget=1.0)
    bench.run_reference(args)
    out = capsys.readouterr().out.strip().splitlines()
    assert len(out) == 1
    line = json.loads(out[0])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == bench.UNIT and line["value"] > 0 and line["steps"] == 4
    assert line["cpu_baseline"]["cores"] == bench.host_cores()
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["config"]["workload"] == "tiny-b1-ctx512"
