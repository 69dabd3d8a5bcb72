"""GPU parity of f8_linear_fwd_w13_swiglu: the group {w1, w3} of a SwiGLU FFN
as one Float8 linear whose GEMM epilogue also forms h = bf16(silu(a) b) and
takes its amax.

- AB (a and b, interleaved by 128 columns) meets the GEMM bar against the
  oracle's linear_fwd of X and W13.
- h is within one bf16 ulp of the oracle's swiglu_h (the fp64 definition) of
  the GPU's own a and b, with the fraction of differing elements asserted
  (the GEMM's fp32 accumulation order decides a and b to within the GEMM
  bar; h is defined from the bf16 a, b).
- amax(h), the scale and every E4M3 byte of q(h), q(h)^T are bit-exact
  against the oracle's quantize of the GPU's h, and the saved q(X)^T, q(W13)^T
  and scalars against the oracle's quantize of X and W13.
- The CTA-pair kernel (M >= 256) and the single-CTA kernel (M < 256), M and K
  tails, several waves of tiles, the Llama-3.1-8B FFN size (sampled rows),
  and the chain into the w2 GEMM and the group's backward.
"""
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


def _interleave(w1, w3):
    """W13 per the entry point's definition, written out here: rows [256j,
    256j + 128) from W1 rows [128j, 128j + 128), the next 128 from W3."""
    F = w1.shape[0]
    parts = []
    for j in range(F // 128):
        parts += [w1[128 * j:128 * (j + 1)], w3[128 * j:128 * (j + 1)]]
    return torch.cat(parts)


def _inputs(M, F, K, seed, x_std=1.0):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn((M, K), generator=g) * x_std).to(torch.bfloat16)
    w1 = (torch.randn((F, K), generator=g) * 0.02).to(torch.bfloat16)
    w3 = (torch.randn((F, K), generator=g) * 0.02).to(torch.bfloat16)
    return x, w1, w3


def _check_h_and_quant(f8, ab, h, h_q, h_t, scale_h, amax_h, max_frac=SWIGLU_MISMATCH_ORDINARY):
    a_g, b_g = oracle.split_ab(wl.bits(ab.cpu()))
    h_g = wl.bits(h.cpu())
    check_swiglu_ulp(h_g, oracle.swiglu_h(a_g, b_g), max_frac, what="h")
    qh = oracle.quantize(h_g)
    assert amax_h.item() == float(qh["amax"]) and scale_h.item() == float(qh["scale"])
    assert np.array_equal(h_q.cpu().numpy(), qh["q"])
    assert np.array_equal(h_t.cpu().numpy(), qh["qt"])
    return h_g, qh


def test_interleave_helper_matches_definition(f8):
    x, w1, w3 = _inputs(16, 384, 32, 3)
    assert torch.equal(f8.interleave_w13(w1, w3), _interleave(w1, w3))
    ab = torch.arange(5 * 768, dtype=torch.int16).view(5, 768).view(torch.bfloat16)
    a, b = f8.split_ab(ab)
    ao, bo = oracle.split_ab(wl.bits(ab))
    assert np.array_equal(wl.bits(a.contiguous()), ao) and np.array_equal(wl.bits(b.contiguous()), bo)


@pytest.mark.parametrize("M,F,K", [(256, 128, 256), (272, 256, 528), (128, 384, 512),
                                   (48, 128, 64), (1040, 640, 1024)])
def test_w13_swiglu_full_compare(f8, M, F, K):
    x, w1, w3 = _inputs(M, F, K, M + F + K)
    w13 = _interleave(w1, w3)
    ab, h, saved, h_q, h_t, scale_h, amax_h = f8.f8_linear_fwd_w13_swiglu(x.to(DEV), w13.to(DEV))
    assert f8.f8_last_device_status() == 0
    ref = oracle.linear_fwd(wl.bits(x), wl.bits(w13))
    assert np.array_equal(saved.x_t.cpu().numpy(), ref["x"]["qt"])
    assert np.array_equal(saved.w_t.cpu().numpy(), ref["w"]["qt"])
    assert saved.scalars.cpu().tolist() == [float(ref["x"]["amax"]), float(ref["x"]["scale"]),
                                            float(ref["w"]["amax"]), float(ref["w"]["scale"])]
    check_close(ab, ref["y"], what="AB")
    _check_h_and_quant(f8, ab, h, h_q, h_t, scale_h, amax_h)


def test_w13_swiglu_large_activations(f8):
    """X scaled so that |a| reaches the tens: silu's negative tail and exp's
    reduction over a wide range, h still within one ulp."""
    M, F, K = 256, 256, 256
    x, w1, w3 = _inputs(M, F, K, 99, x_std=300.0)
    w13 = _interleave(w1, w3)
    ab, h, saved, h_q, h_t, scale_h, amax_h = f8.f8_linear_fwd_w13_swiglu(x.to(DEV), w13.to(DEV))
    assert f8.f8_last_device_status() == 0
    assert float(ab.float().abs().max()) > 20.0
    check_close(ab, oracle.linear_fwd(wl.bits(x), wl.bits(w13))["y"], what="AB")
    _check_h_and_quant(f8, ab, h, h_q, h_t, scale_h, amax_h, SWIGLU_MISMATCH_SWEEP)


def test_w13_chain_into_w2_and_group_backward(f8):
    """q(h) from the epilogue feeds the w2 GEMM (f8_quantize of W2, then
    f8_gemm), and the group's backward is f8_linear_bwd with N = 2F."""
    M, F, K, D = 256, 256, 256, 384
    x, w1, w3 = _inputs(M, F, K, 5)
    w13 = _interleave(w1, w3)
    g = torch.Generator().manual_seed(6)
    w2 = (torch.randn((D, F), generator=g) * 0.02).to(torch.bfloat16)
    dy13 = (torch.randn((M, 2 * F), generator=g) * 0.01).to(torch.bfloat16)
    ab, h, saved, h_q, h_t, scale_h, amax_h = f8.f8_linear_fwd_w13_swiglu(x.to(DEV), w13.to(DEV))
    w2_q, w2_t, scale_w2, amax_w2 = f8.f8_quantize(w2.to(DEV))
    y = f8.f8_gemm(h_q, w2_q, scale_h, scale_w2)
    dx, dw = f8.f8_linear_bwd(dy13.to(DEV), saved)
    assert f8.f8_last_device_status() == 0
    h_g = wl.bits(h.cpu())
    ref2 = oracle.linear_fwd(h_g, wl.bits(w2))
    check_close(y, ref2["y"], what="Y of w2")
    fwd = oracle.linear_fwd(wl.bits(x), wl.bits(w13))
    bwd = oracle.linear_bwd(wl.bits(dy13), fwd)
    check_close(dx, bwd["dx"], what="dX of the group")
    check_close(dw, bwd["dw"], what="dW13")


def test_w13_swiglu_llama8b(f8):
    """The Llama-3.1-8B FFN input side at full size: M=8192, K=4096, F=14336.
    AB on one sampled row per 128-row block against the oracle; h within one
    ulp and q(h) bit-exact, in full."""
    M, F, K = 8192, 14336, 4096
    x = wl.normal((M, K), 1.0, wl.seed_of(3, 0, 0))
    w1 = wl.normal((F, K), 0.02, wl.seed_of(3, 0, 1))
    w3 = wl.normal((F, K), 0.02, wl.seed_of(3, 1, 1))
    w13 = _interleave(w1, w3)
    ab, h, saved, h_q, h_t, scale_h, amax_h = f8.f8_linear_fwd_w13_swiglu(x.to(DEV), w13.to(DEV))
    assert f8.f8_last_device_status() == 0
    qx = oracle.quantize(wl.bits(x))
    qw = oracle.quantize(wl.bits(w13))
    assert saved.scalars.cpu().tolist() == [float(qx["amax"]), float(qx["scale"]),
                                            float(qw["amax"]), float(qw["scale"])]
    rng = np.random.default_rng(13)
    rows = np.array([r * 128 + rng.integers(0, 128) for r in range(M // 128)], np.int64)
    check_close(ab[torch.from_numpy(rows).to(DEV)],
                oracle.gemm_rows(qx["q"], qw["q"], qx["scale"], qw["scale"], rows), what="AB rows")
    _check_h_and_quant(f8, ab, h, h_q, h_t, scale_h, amax_h)


@pytest.mark.parametrize("M,F,K", [(272, 256, 528), (128, 128, 256)])
def test_gemm_w13_swiglu_alone_equals_fused_call(f8, M, F, K):
    """The standalone GEMM entry point on q(X), q(W13) gives the same AB and
    h bits as the fused call, and amax_h = max |h| of the oracle."""
    x, w1, w3 = _inputs(M, F, K, 17)
    w13 = _interleave(w1, w3).to(DEV)
    xd = x.to(DEV)
    ab, h, saved, h_q, h_t, scale_h, amax_h = f8.f8_linear_fwd_w13_swiglu(xd, w13)
    x_q, _, sx, _ = f8.f8_quantize(xd)
    w_q, _, sw, _ = f8.f8_quantize(w13)
    ab2, h2, amax2 = f8.f8_gemm_w13_swiglu(x_q, w_q, sx, sw)
    assert f8.f8_last_device_status() == 0
    assert torch.equal(ab.view(torch.int16), ab2.view(torch.int16))
    assert torch.equal(h.view(torch.int16), h2.view(torch.int16))
    assert amax2.item() == amax_h.item() == float(oracle.quantize(wl.bits(h.cpu()))["amax"])


def _split(ab):
    return oracle.split_ab(wl.bits(ab.cpu()))


@pytest.mark.parametrize("M,F,K", [(256, 256, 256), (272, 384, 528), (128, 128, 64)])
def test_w13_swiglu_bwd_full_compare(f8, M, F, K):
    """Forward, then the backward for a random dh: d(AB) within one ulp of
    the oracle's swiglu_bwd of dh and the GPU's own a, b (merged in AB's
    order); dX and dW13 within the GEMM bar against the oracle's linear_bwd
    of the GPU's d(AB)."""
    x, w1, w3 = _inputs(M, F, K, 3 * M + F)
    w13 = _interleave(w1, w3)
    dh = (torch.randn((M, F), generator=torch.Generator().manual_seed(M + 7)) * 0.01).to(torch.bfloat16)
    ab, h, saved, h_q, h_t, scale_h, amax_h = f8.f8_linear_fwd_w13_swiglu(x.to(DEV), w13.to(DEV))
    dx, dw, dab = f8.f8_linear_bwd_w13_swiglu(dh.to(DEV), ab, saved)
    assert f8.f8_last_device_status() == 0
    a_g, b_g = _split(ab)
    da, db = oracle.swiglu_bwd(wl.bits(dh), a_g, b_g)
    dab_g = wl.bits(dab.cpu())
    check_swiglu_ulp(dab_g, oracle.merge_ab(da, db), SWIGLU_MISMATCH_ORDINARY, what="d(AB)")
    fwd = oracle.linear_fwd(wl.bits(x), wl.bits(w13))
    bwd = oracle.linear_bwd(dab_g, fwd)
    check_close(dx, bwd["dx"], what="dX of the group")
    check_close(dw, bwd["dw"], what="dW13")


@pytest.mark.parametrize("order", ["sorted", "shuffled"])
def test_w13_swiglu_bwd_every_bf16_a(f8, order):
    """d(AB) for every one of the 65536 bf16 values of a (inf and NaN
    included) with random b and dh: within one ulp of the oracle (NaN where
    it has NaN)."""
    M, F, K = 256, 256, 64
    codes = np.arange(65536, dtype=np.uint16)
    if order == "shuffled":
        codes = codes[np.random.default_rng(9).permutation(65536)]
    a = codes.reshape(M, F)
    rng = torch.Generator().manual_seed(10)
    b = wl.bits(torch.randn((M, F), generator=rng).to(torch.bfloat16))
    dh = torch.randn((M, F), generator=rng).to(torch.bfloat16)
    ab = torch.from_numpy(oracle.merge_ab(a, b).view(np.int16).copy()).view(torch.bfloat16)
    x, w1, w3 = _inputs(M, F, K, 11)
    _, _, saved, _, _, _, _ = f8.f8_linear_fwd_w13_swiglu(x.to(DEV), _interleave(w1, w3).to(DEV))
    _, _, dab = f8.f8_linear_bwd_w13_swiglu(dh.to(DEV), ab.to(DEV), saved)
    f8.f8_last_device_status()   # NaN inputs flag the amax non-finite; clear it
    da, db = oracle.swiglu_bwd(wl.bits(dh), a, b)
    check_swiglu_ulp(dab, oracle.merge_ab(da, db), SWIGLU_MISMATCH_SWEEP, what="d(AB)")


def test_w13_swiglu_bwd_llama8b(f8):
    """The Llama-3.1-8B FFN backward through the group at full size
    (M=8192, K=4096, F=14336): d(AB) within one ulp in full; dX and dW13 on
    one sampled row per 128-row block, against the oracle's GEMMs of the
    GPU's d(AB)."""
    M, F, K = 8192, 14336, 4096
    x = wl.normal((M, K), 1.0, wl.seed_of(3, 0, 0))
    w13 = _interleave(wl.normal((F, K), 0.02, wl.seed_of(3, 0, 1)),
                      wl.normal((F, K), 0.02, wl.seed_of(3, 1, 1)))
    dh = wl.normal((M, F), 0.01, wl.seed_of(3, 2, 5))
    ab, h, saved, h_q, h_t, scale_h, amax_h = f8.f8_linear_fwd_w13_swiglu(x.to(DEV), w13.to(DEV))
    dx, dw, dab = f8.f8_linear_bwd_w13_swiglu(dh.to(DEV), ab, saved)
    assert f8.f8_last_device_status() == 0
    a_g, b_g = _split(ab)
    da, db = oracle.swiglu_bwd(wl.bits(dh), a_g, b_g)
    dab_g = wl.bits(dab.cpu())
    check_swiglu_ulp(dab_g, oracle.merge_ab(da, db), SWIGLU_MISMATCH_ORDINARY, what="d(AB)")
    q = oracle.quantize(dab_g)
    qx = oracle.quantize(wl.bits(x))
    qw = oracle.quantize(wl.bits(w13))
    rng = np.random.default_rng(14)
    rows = np.array([r * 128 + rng.integers(0, 128) for r in range(M // 128)], np.int64)
    check_close(dx[torch.from_numpy(rows).to(DEV)],
                oracle.gemm_rows(q["q"], qw["qt"], q["scale"], qw["scale"], rows), what="dX rows")
    rows_n = np.array([r * 128 + rng.integers(0, 128) for r in range(2 * F // 128)], np.int64)
    check_close(dw[torch.from_numpy(rows_n).to(DEV)],
                oracle.gemm_rows(q["qt"], qx["qt"], q["scale"], qx["scale"], rows_n), what="dW13 rows")


def test_quantize_swiglu_bwd_alone(f8):
    """f8_quantize_swiglu_bwd: d(AB) within one ulp of the oracle's, and
    amax, scale, q and q^T bit-exact against the oracle's quantize of the
    GPU's d(AB)."""
    M, F = 272, 384
    g = torch.Generator().manual_seed(23)
    ab = torch.randn((M, 2 * F), generator=g).to(torch.bfloat16)
    dh = (torch.randn((M, F), generator=g) * 0.01).to(torch.bfloat16)
    q, qt, s, amax, dab = f8.f8_quantize_swiglu_bwd(dh.to(DEV), ab.to(DEV))
    assert f8.f8_last_device_status() == 0
    a, b = oracle.split_ab(wl.bits(ab))
    dab_g = wl.bits(dab.cpu())
    check_swiglu_ulp(dab_g, oracle.merge_ab(*oracle.swiglu_bwd(wl.bits(dh), a, b)),
                     SWIGLU_MISMATCH_ORDINARY, what="d(AB)")
    ref = oracle.quantize(dab_g)
    assert amax.item() == float(ref["amax"]) and s.item() == float(ref["scale"])
    assert np.array_equal(q.cpu().numpy(), ref["q"]) and np.array_equal(qt.cpu().numpy(), ref["qt"])


def test_w13_swiglu_bwd_e5m2(f8):
    """The group's backward with d(AB) in E5M2 (scale 57344/amax, E5M2 x E4M3
    GEMMs): d(AB) within one ulp of the oracle and equal between the two
    entry points; q(d(AB)) and its scale bit-exact against the oracle's E5M2
    quantize of the GPU's d(AB); dX and dW13 within the GEMM bar against the
    oracle's linear_bwd of it with dy_fmt = E5M2."""
    M, F, K = 272, 256, 528
    x, w1, w3 = _inputs(M, F, K, 41)
    w13 = _interleave(w1, w3)
    dh = (torch.randn((M, F), generator=torch.Generator().manual_seed(42)) * 0.01).to(torch.bfloat16)
    ab, h, saved, h_q, h_t, scale_h, amax_h = f8.f8_linear_fwd_w13_swiglu(x.to(DEV), w13.to(DEV))
    dx, dw, dab = f8.f8_linear_bwd_w13_swiglu(dh.to(DEV), ab, saved, dy_fmt=f8.F8_E5M2)
    q, qt, s, amax, dab2 = f8.f8_quantize_swiglu_bwd(dh.to(DEV), ab, fmt=f8.F8_E5M2)
    assert f8.f8_last_device_status() == 0
    a_g, b_g = _split(ab)
    dab_g = wl.bits(dab.cpu())
    check_swiglu_ulp(dab_g, oracle.merge_ab(*oracle.swiglu_bwd(wl.bits(dh), a_g, b_g)),
                     SWIGLU_MISMATCH_ORDINARY, what="d(AB)")
    assert np.array_equal(wl.bits(dab2.cpu()), dab_g)
    qref = oracle.quantize(dab_g, oracle.E5M2)
    assert s.item() == float(qref["scale"])
    assert np.array_equal(q.cpu().numpy(), qref["q"]) and np.array_equal(qt.cpu().numpy(), qref["qt"])
    fwd = oracle.linear_fwd(wl.bits(x), wl.bits(w13))
    bwd = oracle.linear_bwd(dab_g, fwd, dy_fmt=oracle.E5M2)
    check_close(dx, bwd["dx"], what="dX (E5M2 d(AB))")
    check_close(dw, bwd["dw"], what="dW13 (E5M2 d(AB))")


def test_w13_swiglu_smallest_shape(f8):
    """M = 16 rows (single-CTA kernel, one partial tile), F = 128, K = 16."""
    M, F, K = 16, 128, 16
    x, w1, w3 = _inputs(M, F, K, 51)
    w13 = _interleave(w1, w3)
    ab, h, saved, h_q, h_t, scale_h, amax_h = f8.f8_linear_fwd_w13_swiglu(x.to(DEV), w13.to(DEV))
    dh = (torch.randn((M, F), generator=torch.Generator().manual_seed(52)) * 0.01).to(torch.bfloat16)
    dx, dw, dab = f8.f8_linear_bwd_w13_swiglu(dh.to(DEV), ab, saved)
    assert f8.f8_last_device_status() == 0
    check_close(ab, oracle.linear_fwd(wl.bits(x), wl.bits(w13))["y"], what="AB")
    _check_h_and_quant(f8, ab, h, h_q, h_t, scale_h, amax_h)
    a_g, b_g = _split(ab)
    check_swiglu_ulp(dab, oracle.merge_ab(*oracle.swiglu_bwd(wl.bits(dh), a_g, b_g)),
                     SWIGLU_MISMATCH_SWEEP * 10, what="d(AB)")


def test_w13_swiglu_bwd_flags_nonfinite_dh(f8):
    """An infinite dh makes d(AB) non-finite: the pass still writes every
    finite element within one ulp of the oracle, the non-finite ones where
    the oracle has them, and the status reads F8_ERR_NONFINITE."""
    M, F, K = 256, 128, 64
    x, w1, w3 = _inputs(M, F, K, 61)
    ab, h, saved, *_ = f8.f8_linear_fwd_w13_swiglu(x.to(DEV), _interleave(w1, w3).to(DEV))
    assert f8.f8_last_device_status() == 0
    dh = (torch.randn((M, F), generator=torch.Generator().manual_seed(62)) * 0.01).to(torch.bfloat16)
    dh[5, 17] = float("inf")
    _, _, dab = f8.f8_linear_bwd_w13_swiglu(dh.to(DEV), ab, saved)
    assert f8.f8_last_device_status() == f8.binding.F8_ERR_NONFINITE
    a_g, b_g = _split(ab)
    ref = oracle.merge_ab(*oracle.swiglu_bwd(wl.bits(dh), a_g, b_g)).ravel()
    got = wl.bits(dab.cpu()).ravel()
    finite = (ref & 0x7FFF) < 0x7F80
    assert np.array_equal((got & 0x7FFF) >= 0x7F80, ~finite)
    check_swiglu_ulp(got[finite], ref[finite], SWIGLU_MISMATCH_ORDINARY, what="finite d(AB)")


@pytest.mark.parametrize("want", ["dx", "dw"])
def test_w13_swiglu_bwd_one_output(f8, want):
    """dX only or dW13 only: the one asked for equals the full backward's."""
    M, F, K = 256, 256, 128
    x, w1, w3 = _inputs(M, F, K, 71)
    ab, h, saved, *_ = f8.f8_linear_fwd_w13_swiglu(x.to(DEV), _interleave(w1, w3).to(DEV))
    dh = (torch.randn((M, F), generator=torch.Generator().manual_seed(72)) * 0.01).to(torch.bfloat16)
    dx, dw, _ = f8.f8_linear_bwd_w13_swiglu(dh.to(DEV), ab, saved)
    dx1, dw1, _ = f8.f8_linear_bwd_w13_swiglu(dh.to(DEV), ab, saved, want_dx=(want == "dx"),
                                              want_dw=(want == "dw"))
    assert f8.f8_last_device_status() == 0
    if want == "dx":
        assert dw1 is None and torch.equal(dx1.view(torch.int16), dx.view(torch.int16))
    else:
        assert dx1 is None and torch.equal(dw1.view(torch.int16), dw.view(torch.int16))
