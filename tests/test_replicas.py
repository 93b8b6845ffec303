"""Replica launch logic on CPU with two gloo ranks (no GPU needed)."""

import os
import socket

import pytest
import torch.multiprocessing as mp

from tiled_attention_fa_gb300 import replicas


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    assert replicas.init("gloo")
    replicas.barrier()
    m = replicas.max_over_ranks(rank + 1.5)
    lo, hi = replicas.shard_units(10, rank, world)
    q.put((rank, m, replicas.replica_seed(7, rank), lo, hi, replicas.dist_env()))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=60) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[1] for o in out] == [2.5, 2.5]          # max over ranks
    assert out[0][2] != out[1][2]                       # independent batches
    assert (out[0][3], out[0][4], out[1][3], out[1][4]) == (0, 5, 5, 10)
    assert out[1][5] == (2, 1, 1)


@pytest.mark.parametrize("n,world", [(10, 3), (7, 7), (3, 5), (256, 8)])
def test_shards_are_disjoint_and_cover(n, world):
    seen = []
    for r in range(world):
        lo, hi = replicas.shard_units(n, r, world)
        seen.extend(range(lo, hi))
    assert seen == list(range(n))


def test_single_process_defaults(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert replicas.dist_env() == (1, 0, 0)
    assert replicas.max_over_ranks(3.0) == 3.0
    assert replicas.aggregate_rate(10.0, 4, 2.0) == 20.0
