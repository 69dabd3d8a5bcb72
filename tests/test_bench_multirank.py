"""The N > 1 host logic of bench.py on CPU with gloo, world size 2: each rank
is an independent replica, the timing is the max over ranks and the work is
the sum over ranks (value = total work / max time, weak scaling)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, lr = bench.dist_env()
    ms = 10.0 + 5.0 * rank                  # rank 1 is the slower replica
    flops = 1e12 * (rank + 1)
    t = bench.max_over_ranks(ms, w)
    f = bench.sum_over_ranks(flops, w)
    q.put((r, w, lr, t, f))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, world, local, t, f) in enumerate(out):
        assert (rank, world, local) == (r, 2, r)
        assert t == 15.0           # max over ranks
        assert f == 3e12           # sum over ranks
    value = out[0][4] / (out[0][3] * 1e-3) / 1e12
    assert value == pytest.approx(200.0)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.sum_over_ranks(7.0, 1) == 7.0
