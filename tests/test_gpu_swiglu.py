"""GPU parity of the SwiGLU quantisation (h = bf16(silu(a) b) produced with its
amax in one pass, then cast):
- h within one bf16 ulp of the oracle's fp64 definition, with the fraction of
  differing elements asserted (tolerance.check_swiglu_ulp);
- amax, the scale and every E4M3 byte of q(h), q(h)^T bit-exact against the
  oracle's quantize of the GPU's h;
- the w2 linear fed by it (forward and backward) within the GEMM bar against
  the oracle's linear of the GPU's h, small in full and at the Llama-3.1-8B
  FFN size on sampled rows."""
import numpy as np
import pytest
import torch

import oracle
from float8_mixed_precision_gb300 import workloads as wl
from tolerance import (SWIGLU_MISMATCH_ORDINARY, SWIGLU_MISMATCH_SWEEP, check_close,
                       check_swiglu_ulp)

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


def _ab(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    a = (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)
    b = torch.randn(shape, generator=g).to(torch.bfloat16)
    return a, b


@pytest.mark.parametrize("shape,scale", [((1, 1), 1.0), ((7, 33), 1.0), ((130, 260), 3.0),
                                         ((320, 528), 1.0), ((1024, 4096), 1.0), ((256, 512), 40.0)])
def test_quantize_swiglu_bytes(f8, shape, scale):
    a, b = _ab(shape, shape[0] + shape[1], scale)
    q, qt, s, amax, hg = f8.f8_quantize_swiglu(a.to(DEV), b.to(DEV))
    check_swiglu_ulp(hg, oracle.swiglu_h(wl.bits(a), wl.bits(b)),
                     SWIGLU_MISMATCH_ORDINARY if scale == 1.0 else SWIGLU_MISMATCH_SWEEP, what="h")
    ref = oracle.quantize(wl.bits(hg.cpu()))
    assert amax.item() == float(ref["amax"]) and s.item() == float(ref["scale"])
    assert np.array_equal(q.cpu().numpy(), ref["q"]) and np.array_equal(qt.cpu().numpy(), ref["qt"])
    assert f8.f8_last_device_status() == 0


def test_quantize_swiglu_special_values(f8):
    """Zeros, the fast path's edge (|a| = 87.5, 88.5) and the negative tail
    (a = -88.5, -92, -100, where silu(a) b is still a bf16 normal or
    subnormal), huge and tiny a: within one ulp of the oracle."""
    vals = [0.0, -0.0, 1.0, -1.0, 20.0, -20.0, 87.5, -87.5, 88.5, -88.5, 100.0, -100.0, 1e-30, 1e30,
            -92.0, -95.0]
    a = torch.tensor(vals * 16, dtype=torch.bfloat16).reshape(16, 16)
    b = torch.tensor([1.0, -2.0, 0.5, 0.0] * 64, dtype=torch.bfloat16).reshape(16, 16)
    q, qt, s, amax, hg = f8.f8_quantize_swiglu(a.to(DEV), b.to(DEV))
    check_swiglu_ulp(hg, oracle.swiglu_h(wl.bits(a), wl.bits(b)), SWIGLU_MISMATCH_SWEEP * 10, what="h")
    ref = oracle.quantize(wl.bits(hg.cpu()))
    assert amax.item() == float(ref["amax"]) and s.item() == float(ref["scale"])
    assert np.array_equal(q.cpu().numpy(), ref["q"])


@pytest.mark.parametrize("order", ["sorted", "shuffled"])
def test_swiglu_h_every_bf16_a(f8, order):
    """Every one of the 65536 bf16 values of a (inf and NaN included) against
    random b: h within one ulp of the oracle (NaN where it has NaN).
    Sorted, the groups of 8 consecutive elements fall wholly inside or
    outside |a| <= 87; shuffled, most groups mix the two."""
    codes = np.arange(65536, dtype=np.uint16)
    if order == "shuffled":
        codes = codes[np.random.default_rng(7).permutation(65536)]
    a = torch.from_numpy(codes.view(np.int16).copy()).view(torch.bfloat16).reshape(256, 256)
    b = torch.randn((256, 256), generator=torch.Generator().manual_seed(8)).to(torch.bfloat16)
    _, _, _, _, hg = f8.f8_quantize_swiglu(a.to(DEV), b.to(DEV))
    f8.f8_last_device_status()   # NaN inputs flag the amax non-finite; clear it
    check_swiglu_ulp(hg, oracle.swiglu_h(wl.bits(a), wl.bits(b)), SWIGLU_MISMATCH_SWEEP, what="h")


@pytest.mark.parametrize("M,N,K", [(256, 384, 512), (272, 400, 528)])
def test_linear_fwd_swiglu_full_compare(f8, M, N, K):
    a, b = _ab((M, K), M + K)
    w = (torch.randn(N, K, generator=torch.Generator().manual_seed(N)) * 0.02).to(torch.bfloat16)
    dy = torch.randn(M, N, generator=torch.Generator().manual_seed(M)).to(torch.bfloat16)
    hg = torch.empty((M, K), dtype=torch.bfloat16, device=DEV)
    y, saved = f8.f8_linear_fwd_swiglu(a.to(DEV), b.to(DEV), w.to(DEV), h=hg)
    dx, dw = f8.f8_linear_bwd(dy.to(DEV), saved)
    assert f8.f8_last_device_status() == 0
    h = wl.bits(hg.cpu())
    check_swiglu_ulp(h, oracle.swiglu_h(wl.bits(a), wl.bits(b)), SWIGLU_MISMATCH_ORDINARY, what="h")
    fwd = oracle.linear_fwd(h, wl.bits(w))
    bwd = oracle.linear_bwd(wl.bits(dy), fwd)
    assert np.array_equal(saved.x_t.cpu().numpy(), fwd["x"]["qt"])
    assert saved.scalars[1].item() == float(fwd["x"]["scale"])
    check_close(y, fwd["y"], what="Y")
    check_close(dx, bwd["dx"], what="dX")
    check_close(dw, bwd["dw"], what="dW")


def test_linear_fwd_swiglu_llama8b_w2(f8):
    """The w2 linear of the Llama-3.1-8B FFN workload (M=8192, K=14336 ->
    N=4096) with its input given as the a, b of the SwiGLU."""
    c, l = 3, 2
    lin = wl.workload(c)[1][l]
    shape = (lin.M, lin.K)
    g_a = torch.Generator().manual_seed(wl.seed_of(c, l, 3))
    g_b = torch.Generator().manual_seed(wl.seed_of(c, l, 4))
    a = torch.randn(shape, generator=g_a).to(torch.bfloat16)
    b = torch.randn(shape, generator=g_b).to(torch.bfloat16)
    w = wl.normal((lin.N, lin.K), lin.w_std, wl.seed_of(c, l, 1))
    hg = torch.empty(shape, dtype=torch.bfloat16, device=DEV)
    y, saved = f8.f8_linear_fwd_swiglu(a.to(DEV), b.to(DEV), w.to(DEV), h=hg)
    assert f8.f8_last_device_status() == 0
    h = wl.bits(hg.cpu())
    check_swiglu_ulp(h, oracle.swiglu_h(wl.bits(a), wl.bits(b)), SWIGLU_MISMATCH_ORDINARY, what="h")
    qh = oracle.quantize(h)
    qw = oracle.quantize(wl.bits(w))
    assert saved.scalars[1].item() == float(qh["scale"])
    assert np.array_equal(saved.x_t.cpu().numpy(), qh["qt"])
    rng = np.random.default_rng(4)
    rows = np.array([r * 128 + rng.integers(0, 128) for r in range(lin.M // 128)], np.int64)
    check_close(y[torch.from_numpy(rows).to(DEV)],
                oracle.gemm_rows(qh["q"], qw["q"], qh["scale"], qw["scale"], rows), what="Y rows")
