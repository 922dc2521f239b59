"""N > 1 host path of bench.py on CPU: two gloo ranks on 127.0.0.1.

Ranks are independent replicas of the workload (no data-path collective); the
only cross-rank step is the max of the timed region, which these tests check,
together with the whole-job throughput formula and the reference arm's
rank-0-only behaviour."""

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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
        m = bench.reduce_max_over_ranks(local_ms, world)
        out[rank] = (m, bench.job_throughput(1e12, world, 4, m))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0
    # 2 ranks x 4 steps x 1 TFLOP in 15 ms
    assert res[0][1] == pytest.approx(2 * 4 * 1.0 / 15e-3)


def test_single_rank_is_identity():
    assert bench.reduce_max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(2e12, 1, 10, 20.0) == pytest.approx(1000.0)


def test_reference_arm_runs_on_rank0_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    args = type("A", (), dict(workload="single1k_d64", steps=1, warmup=3, gpus=2,
                              ref_step_seconds=0.01))()
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""


def test_visible_pairs_closed_form():
    # per request: n * prefix + n(n+1)/2
    assert bench.visible_pairs([32768], [0]) == 32768 * 32769 // 2
    assert bench.visible_pairs([517, 1000, 33, 2048, 3, 1500], [0, 256, 0, 1024, 17, 0]) == \
        6212099
