"""The multi-process host logic (sharding over (b, h), max-over-ranks timing) with
world_size 2 on the gloo backend, on CPU."""
import os

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from gated_delta_rule_26_gb300 import dist as kdist


@pytest.mark.parametrize("n,world", [(256, 2), (255, 2), (7, 3), (1, 4), (0, 2), (8192, 8)])
def test_shard_range_partitions_exactly(n, world):
    seen = []
    sizes = []
    for r in range(world):
        b, e = kdist.shard_range(n, r, world)
        seen.extend(range(b, e))
        sizes.append(e - b)
    assert seen == list(range(n))
    assert max(sizes) - min(sizes) <= 1


def test_shard_range_rejects_bad_rank():
    with pytest.raises(ValueError):
        kdist.shard_range(10, 2, 2)


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, _ = kdist.env()
        b, e = kdist.shard_range(16, r, ws)
        kdist.barrier()
        m = kdist.max_over_ranks(1.5 + r)  # each rank's "elapsed time"
        q.put((r, ws, b, e, m))
    finally:
        dist.destroy_process_group()


def test_gloo_two_ranks_shard_and_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1]
    assert all(r[1] == 2 for r in res)
    assert (res[0][2], res[0][3], res[1][2], res[1][3]) == (0, 8, 8, 16)
    assert all(r[4] == 2.5 for r in res)  # max over ranks
