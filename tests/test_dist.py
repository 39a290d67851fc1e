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


def _bwd_worker(rank, world, port, q, shard):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        p, d_o, dhT = shard  # this rank's sequences (all heads): inputs and output adjoints
        ref = oracle.backward(p["q"], p["k"], p["v"], p["z"], p["beta"], p["A_log"],
                              p["dt_bias"], p["scale"], p["h0"], d_o, dhT)
        g = {"dA_log": torch.from_numpy(ref["dA_log"]),
             "ddt_bias": torch.from_numpy(ref["ddt_bias"]),
             "dq": torch.from_numpy(ref["dq"])}
        kdist.sum_param_grads(g)
        q.put((rank, g["dA_log"].numpy(), g["ddt_bias"].numpy(), g["dq"].numpy()))
    finally:
        dist.destroy_process_group()


def test_gloo_two_ranks_backward_parameter_gradients():
    """The batch split over two ranks (each computing its sequences' gradients; the f64
    oracle stands in for the kernel on the CPU), then sum_param_grads: dA_log and ddt_bias
    equal the whole batch's, on both ranks; per-token gradients stay each rank's own."""
    import numpy as np
    import oracle
    rng = np.random.default_rng(3)
    B, H, T, K, V = 3, 2, 20, 4, 3
    nrm = lambda x: x / np.linalg.norm(x, axis=-1, keepdims=True)
    p = dict(q=nrm(rng.normal(size=(B, H, T, K))), k=nrm(rng.normal(size=(B, H, T, K))),
             v=rng.normal(size=(B, H, T, V)), z=rng.normal(size=(B, H, T, K)),
             beta=1.0 / (1.0 + np.exp(-rng.normal(size=(B, H, T)))),
             A_log=rng.uniform(-1, 1, size=H), dt_bias=0.3 * rng.normal(size=(H, K)),
             scale=K ** -0.5, h0=0.2 * rng.normal(size=(B, H, K, V)))
    d_o = rng.normal(size=(B, H, T, V))
    dhT = rng.normal(size=(B, H, K, V))
    whole = oracle.backward(p["q"], p["k"], p["v"], p["z"], p["beta"], p["A_log"], p["dt_bias"],
                            p["scale"], p["h0"], d_o, dhT)
    shards = []
    for r in range(2):
        b, e = kdist.shard_range(B, r, 2)
        sub = {n: (x[b:e] if n in ("q", "k", "v", "z", "beta", "h0") else x) for n, x in p.items()}
        shards.append((sub, d_o[b:e], dhT[b:e]))
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29700 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_bwd_worker, args=(r, 2, port, q, shards[r])) for r in range(2)]
    for pr in procs:
        pr.start()
    res = sorted((q.get(timeout=120) for _ in procs), key=lambda x: x[0])
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    for r, dA, ddt, dq in res:
        np.testing.assert_allclose(dA, whole["dA_log"], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(ddt, whole["ddt_bias"], rtol=1e-12, atol=1e-14)
        b, e = kdist.shard_range(B, r, 2)
        np.testing.assert_array_equal(dq, whole["dq"][b:e])
