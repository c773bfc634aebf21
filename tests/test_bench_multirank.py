"""The bench's multi-rank host logic on CPU, with the gloo backend and two
ranks: the replicas share no data, the job's time is the slowest rank's (one
all-reduce MAX of one number), throughput is weak-scaling (every rank decodes
its own batch), and under the reference arm only rank 0 works."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        assert (r, w, local) == (rank, world, rank)
        mine = 10.0 + 5.0 * rank  # rank 1 is the slow one
        slowest = bench.max_over_ranks(mine, w)
        out[rank] = (slowest, bench.job_throughput(w, 8, slowest / 100))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_add_their_batches():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0
    # 2 ranks x batch 8 tokens per 0.15 ms step
    assert res[0][1] == pytest.approx(2 * 8 / 0.15e-3)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(1, 8, 0.05) == pytest.approx(160000.0)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        steps, warmup, gpus = 3, 3, 2

    bench.reference_arm(A())
    assert capsys.readouterr().out == ""
