"""The FP8 weight all-gather on the GPU: the protocol of
float8_mixed_precision_gb300.fsdp with libf8's kernels (f8_amax,
f8_cast_transpose, f8_transpose_u8) and NCCL collectives, on a process group
of one rank (the one GPU a box has here: the all-reduce and the all-gather
are then copies, but every call of the path runs).  The gathered q(W),
q(W)^T and scalars equal the oracle's quantisation of W; f8_linear_fwd_qw on
them, then f8_linear_bwd, give outputs bit-identical to f8_linear_fwd /
f8_linear_bwd on the bf16 W.  f8_transpose_u8 is checked against torch's
transpose on ragged shapes."""
import os
import socket

import numpy as np
import pytest
import torch

import oracle
from float8_mixed_precision_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def f8():
    import float8_mixed_precision_gb300 as m
    from float8_mixed_precision_gb300 import build
    build.build()
    oracle.build()
    m.lib()
    return m


# full 128 x 128 tiles take the 16-byte tiled kernel; ragged shapes and
# buffers off 16-byte alignment the byte kernel
@pytest.mark.parametrize("rows,cols", [(1, 1), (7, 300), (64, 64), (130, 257), (128, 200),
                                       (256, 384), (1024, 4096), (1792, 4096)])
def test_transpose_u8(f8, rows, cols):
    x = torch.randint(0, 256, (rows, cols), dtype=torch.uint8, device=DEV)
    t = f8.f8_transpose_u8(x)
    assert f8.f8_last_device_status() == 0
    assert torch.equal(t, x.t().contiguous())


def test_transpose_u8_unaligned_buffers(f8):
    rows, cols = 256, 384
    raw = torch.randint(0, 256, (rows * cols + 8,), dtype=torch.uint8, device=DEV)
    x = raw[8:].view(rows, cols)              # 8 bytes past a 16-byte boundary
    out = torch.empty(rows * cols + 8, dtype=torch.uint8, device=DEV)[8:].view(cols, rows)
    f8.f8_transpose_u8(x, out=out)
    assert f8.f8_last_device_status() == 0
    assert torch.equal(out, x.t().contiguous())


@pytest.fixture(scope="module")
def nccl_one_rank():
    import torch.distributed as dist
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    os.environ.setdefault("NCCL_NVLS_ENABLE", "0")
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    yield dist.group.WORLD
    dist.destroy_process_group()


def test_fp8_all_gather_and_linear_on_the_gathered_weight(f8, nccl_one_rank):
    from float8_mixed_precision_gb300 import fsdp
    M, N, K = 512, 768, 1024
    d = wl.custom_linear(M, K, N, seed=77, dy_std=0.01)
    x, w, dy = d["x"].to(DEV), d["w"].to(DEV), d["dy"].to(DEV)
    q_w, q_w_t, amax, scale = fsdp.fp8_all_gather_weight(w, group=nccl_one_rank)
    torch.cuda.synchronize()
    ref = oracle.quantize(wl.bits(d["w"]))
    assert amax.item() == float(ref["amax"]) and scale.item() == float(ref["scale"])
    assert np.array_equal(q_w.cpu().numpy(), ref["q"])
    assert np.array_equal(q_w_t.cpu().numpy(), ref["qt"])
    saved = fsdp.gathered_saved(q_w_t, amax, scale, M)
    y = f8.f8_linear_fwd_qw(x, q_w, saved)
    dx, dw = f8.f8_linear_bwd(dy, saved)
    y1, s1 = f8.f8_linear_fwd(x, w)
    dx1, dw1 = f8.f8_linear_bwd(dy, s1)
    assert f8.f8_last_device_status() == 0
    for a, b in ((y, y1), (dx, dx1), (dw, dw1)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(saved.x_t, s1.x_t) and torch.equal(saved.scalars, s1.scalars)
