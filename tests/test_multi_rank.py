"""Host logic of the N>1 benchmark path, on CPU with gloo (world size 2).

Ranks run independent batches (weak scaling, no collective on the data path);
the only collectives are the timing reductions, which these tests exercise.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, local, w = bench.dist_env()
        assert (r, local, w) == (rank, rank, world)
        # max over ranks of a per-rank time, and the whole-job sum of work
        t = bench.max_over_ranks(10.0 + rank, world)
        s = bench.sum_over_ranks(1.0 + rank, world)
        bench.barrier(world)
        # every rank draws its own batch: different seeds give different data
        wl = bench.WORKLOAD.with_(B=1, Sq=64, Sk=64, seed=bench.WORKLOAD.seed + 1000 * rank)
        q = synth.make_inputs(wl)[0]
        gathered = [torch.zeros_like(q) for _ in range(world)]
        dist.all_gather(gathered, q.float().to(torch.bfloat16))
        distinct = not torch.equal(gathered[0], gathered[1])
        out[rank] = (t, s, distinct)
    finally:
        dist.destroy_process_group()


def test_two_rank_reductions():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0, "rank process failed"
    for r in range(world):
        t, s, distinct = out[r]
        assert t == 11.0, "max over ranks"
        assert s == 3.0, "sum over ranks"
        assert distinct, "ranks must process different batches"


@pytest.mark.parametrize("n,world", [(64, 2), (65, 2), (7, 4), (3, 8), (1024, 8)])
def test_shard_units_partition(n, world):
    spans = [synth.shard_units(n, r, world) for r in range(world)]
    assert spans[0][0] == 0 and spans[-1][1] == n
    for (a, b), (c, d) in zip(spans, spans[1:]):
        assert b == c
    sizes = [b - a for a, b in spans]
    assert max(sizes) - min(sizes) <= 1


def test_weak_scaling_value_arithmetic():
    """value = FLOPs of all ranks / max-over-ranks time."""
    w = bench.WORKLOAD
    f = bench.step_flops(w)
    assert f == pytest.approx(3.5 * 4 * 2 * 16 * 8192 * 8192 * 128 * 0.5)
    steps, world, total_ms = 10, 4, 5.0
    value = f * world * steps / (total_ms * 1e-3) / 1e12
    assert value == pytest.approx(4 * 10 * f / 5e-3 / 1e12)
