"""The FP8 weight all-gather protocol (float8_mixed_precision_gb300.fsdp) on
CPU gloo ranks, world size 2 and 4, without a GPU: every rank holds a row
shard of W, the device steps are the oracle's (amax, cast with a given
amax's scale, transpose) passed in as the protocol's ops, and the collectives
are gloo's all-reduce(MAX) and all-gather.  On every rank the gathered q(W),
q(W)^T, amax and scale must equal the oracle's quantisation of the whole W:
one scale over all shards, not one per shard.  Also checked: the shards'
own amaxes differ (so a protocol that skipped the all-reduce would fail),
and the bytes on the wire are 1 per element."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _weight(N, K):
    from float8_mixed_precision_gb300 import workloads as wl
    w = wl.normal((N, K), 0.02, 4242)
    # one large entry in the last shard: the global amax comes from there
    w[N - 3, 5] = 1.5
    return w


def _oracle_ops():
    import oracle
    from float8_mixed_precision_gb300 import fsdp
    from float8_mixed_precision_gb300 import workloads as wl

    def amax(shard):
        a, _ = oracle.amax(wl.bits(shard))
        return torch.tensor(float(a), dtype=torch.float32)

    def cast(shard, a):
        s = oracle.scale(float(a))
        q, _ = oracle.cast_transpose(wl.bits(shard.contiguous()), s)
        return torch.from_numpy(q), torch.tensor(float(s), dtype=torch.float32)

    def transpose(q):
        return q.t().contiguous()

    return fsdp.GatherOps(amax=amax, cast=cast, transpose=transpose)


def _worker(rank, world, port, N, K, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from float8_mixed_precision_gb300 import fsdp
    w = _weight(N, K)
    n = N // world
    shard = w[rank * n:(rank + 1) * n].contiguous()
    ops = _oracle_ops()
    local = float(ops.amax(shard))
    q_w, q_w_t, amax, scale = fsdp.fp8_all_gather_weight(shard, ops=ops)
    q.put((rank, local, q_w.numpy().copy(), q_w_t.numpy().copy(), float(amax), float(scale),
           q_w.element_size()))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_fp8_all_gather_equals_whole_weight_quantisation(world, oracle_mod):
    from float8_mixed_precision_gb300 import workloads as wl
    N, K = 256, 96
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, N, K, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted((q.get(timeout=180) for _ in procs), key=lambda t: t[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    ref = oracle_mod.quantize(wl.bits(_weight(N, K)))
    locals_ = [o[1] for o in out]
    assert len(set(locals_)) > 1 and max(locals_) == float(ref["amax"])
    for rank, _, q_w, q_w_t, amax, scale, esize in out:
        assert amax == float(ref["amax"]) and scale == float(ref["scale"]), rank
        assert np.array_equal(q_w, ref["q"]), rank
        assert np.array_equal(q_w_t, ref["qt"]), rank
        assert esize == 1
