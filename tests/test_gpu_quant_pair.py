"""f8_linear_fwd quantises X and W of a linear that fits in L2 with two
launches (one amax over both, one TMA cast over both) instead of four.  The
result must not depend on that: every output of the forward pass (Y, the
saved E4M3 transposes, the four scalars) is compared bit for bit with the
four-launch path (F8_QUANT_PAIR=0), on shapes from equal sizes to a W 64x
smaller than X, and against the oracle on one of them."""
import os

import numpy as np
import pytest
import torch

import oracle
from float8_mixed_precision_gb300 import workloads as wl
from tolerance import check_close

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


def _fwd(f8, x, w, pair):
    old = os.environ.get("F8_QUANT_PAIR")
    os.environ["F8_QUANT_PAIR"] = "1" if pair else "0"
    try:
        y, saved = f8.f8_linear_fwd(x, w)
        assert f8.f8_last_device_status() == 0
    finally:
        if old is None:
            del os.environ["F8_QUANT_PAIR"]
        else:
            os.environ["F8_QUANT_PAIR"] = old
    return y, saved


@pytest.mark.parametrize("M,N,K", [(256, 512, 256), (128, 128, 128), (8192, 1024, 4096),
                                   (8192, 4096, 4096), (1024, 128, 8192), (8192, 128, 4096)])
def test_pair_path_equals_four_launches(f8, M, N, K):
    d = wl.custom_linear(M, K, N, seed=M + N + K, w_std=0.02)
    x, w = d["x"].to(DEV), d["w"].to(DEV)
    y1, s1 = _fwd(f8, x, w, True)
    y0, s0 = _fwd(f8, x, w, False)
    assert torch.equal(y1.view(torch.int16), y0.view(torch.int16))
    assert torch.equal(s1.x_t, s0.x_t) and torch.equal(s1.w_t, s0.w_t)
    assert torch.equal(s1.scalars, s0.scalars)


def test_pair_path_against_oracle(f8):
    M, N, K = 512, 384, 640
    d = wl.custom_linear(M, K, N, seed=77)
    y, saved = _fwd(f8, d["x"].to(DEV), d["w"].to(DEV), True)
    ref = oracle.linear_fwd(wl.bits(d["x"]), wl.bits(d["w"]))
    assert np.array_equal(saved.x_t.cpu().numpy(), ref["x"]["qt"])
    assert np.array_equal(saved.w_t.cpu().numpy(), ref["w"]["qt"])
    assert saved.scalars.cpu().tolist() == [float(ref["x"]["amax"]), float(ref["x"]["scale"]),
                                            float(ref["w"]["amax"]), float(ref["w"]["scale"])]
    check_close(y, ref["y"], what="Y")


@pytest.mark.parametrize("which", ["x", "w"])
def test_pair_path_flags_nonfinite(f8, which):
    M, N, K = 256, 256, 256
    d = wl.custom_linear(M, K, N, seed=5)
    t = d[which].clone()
    t[3, 7] = float("inf")
    d[which] = t
    os.environ["F8_QUANT_PAIR"] = "1"
    try:
        f8.f8_linear_fwd(d["x"].to(DEV), d["w"].to(DEV))
        assert f8.f8_last_device_status() == f8.binding.F8_ERR_NONFINITE
    finally:
        del os.environ["F8_QUANT_PAIR"]


def test_kernel_launch_counts(f8, monkeypatch):
    """libf8's own launch counter: the forward of a linear that fits in L2
    is 3 kernels (paired amax, paired cast, GEMM), 5 on the four-launch path
    or for a shape the TMA cast does not take; the backward is 3 (amax and
    cast of dY, dgrad and wgrad in one GEMM launch), 4 with F8_GEMM_GROUP=0."""
    def count(fn):
        torch.cuda.synchronize()
        n0 = f8.f8_kernel_launches()
        out = fn()
        return f8.f8_kernel_launches() - n0, out
    d = wl.custom_linear(256, 256, 512, seed=3)
    x, w, dy = d["x"].to(DEV), d["w"].to(DEV), d["dy"].to(DEV)
    n, (y, saved) = count(lambda: _fwd(f8, x, w, True))
    assert n == 3
    n, _ = count(lambda: _fwd(f8, x, w, False))
    assert n == 5
    n, _ = count(lambda: f8.f8_linear_bwd(dy, saved))
    assert n == 3
    monkeypatch.setenv("F8_GEMM_GROUP", "0")
    n, _ = count(lambda: f8.f8_linear_bwd(dy, saved))
    assert n == 4
    monkeypatch.delenv("F8_GEMM_GROUP")
    d = wl.custom_linear(272, 528, 400, seed=4)      # not multiples of 128
    n, _ = count(lambda: _fwd(f8, d["x"].to(DEV), d["w"].to(DEV), True))
    assert n == 5
    assert f8.f8_last_device_status() == 0
