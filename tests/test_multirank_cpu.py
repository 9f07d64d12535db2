"""Multi-rank host logic on CPU ranks (gloo).

The N > 1 bench path (world size 2): replicas time their own steps, the slowest rank defines
the job time, and rank 0 alone reports.  The token-sharded routing exchange (world size 3):
each rank's expert counts reach every rank, and the oracle's shard dispatch with the
resulting bases reproduces the whole batch's routing."""
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


def _shard_rank_main(rank, world, port, q):
    import numpy as np
    import torch
    import torch.distributed as dist

    import oracle
    from sparse_expert_ffn_layer_gb300 import sharded
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    rng = np.random.default_rng(11)
    T, E, k = 301, 8, 2
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[:, 5] += 1.0                                        # a hot expert
    _, idx, _ = oracle.softmax_topk(logits, k)
    cuts = [0, 77, 77, T]                                     # rank 1 holds no tokens
    lo, hi = cuts[rank], cuts[rank + 1]
    mine = idx[lo:hi]
    counts = torch.from_numpy(np.bincount(mine.reshape(-1), minlength=E).astype(np.int32))
    counts_all, T_global = sharded.exchange_counts(counts, hi - lo)
    C = oracle.capacity(T_global, E, 1.0)
    base = oracle.shard_bases(counts_all.numpy())[rank]
    got = oracle.dispatch_shard(mine, E, C, base)
    q.put((rank, T_global, counts_all.numpy().tolist(), got.slot_of.tolist(),
           got.perm.tolist(), got.offsets.tolist()))
    dist.barrier()
    dist.destroy_process_group()


def test_sharded_routing_exchange_on_three_cpu_ranks():
    import numpy as np

    import oracle
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    world = 3
    procs = [ctx.Process(target=_shard_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    rng = np.random.default_rng(11)
    T, E, k = 301, 8, 2
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[:, 5] += 1.0
    _, idx, _ = oracle.softmax_topk(logits, k)
    whole = oracle.dispatch(idx, E, oracle.capacity(T, E, 1.0))
    cuts = [0, 77, 77, T]
    assert whole.kept.max() == oracle.capacity(T, E, 1.0)      # the cut binds somewhere
    for rank, T_global, counts_all, slot_of, perm, offsets in res:
        assert T_global == T
        assert np.array_equal(np.array(counts_all).sum(0), whole.counts_raw)
        lo, hi = cuts[rank], cuts[rank + 1]
        slot_of = np.array(slot_of).reshape(hi - lo, k)
        assert np.array_equal(slot_of >= 0, whole.slot_of[lo:hi] >= 0)
        for e in range(E):
            seg = np.array(perm[offsets[e]:offsets[e + 1]], dtype=np.int64) + lo
            w = whole.perm[whole.offsets[e]:whole.offsets[e + 1]]
            assert np.array_equal(seg, w[(w >= lo) & (w < hi)])
