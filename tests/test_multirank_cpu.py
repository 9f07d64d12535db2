"""The N > 1 bench path on CPU ranks (gloo, world size 2): replicas time their own steps, the
slowest rank defines the job time, and rank 0 alone reports."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = [10.0 + 5.0 * rank, 20.0 - 7.0 * rank]
    got = bench.max_over_ranks(mine, dist, "cpu")
    q.put((rank, got, bench.job_tokens_per_s(world, 4096, 10, got[0])))
    dist.barrier()
    dist.destroy_process_group()


def test_two_cpu_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, val in res:
        assert got == [15.0, 20.0]
        assert val == pytest.approx(2 * 4096 * 10 / 0.015)


def test_reference_arm_only_rank0_reports(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    args = type("A", (), dict(workload="tiny_fp32", tokens=128, steps=1, warmup=0, seed=0,
                              gpus=2))()
    assert bench.run_reference(args) is None
    assert capsys.readouterr().out == ""
