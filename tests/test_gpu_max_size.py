"""Sizes past 2^31 elements, where a 32-bit element index would wrap: the
largest linear of the workloads (the 70B w1 input, 235M elements) stays
below it, so these cases are built for the purpose.

- f8_amax over 2^31 + 1000 elements (a ragged tail of 8-element vectors),
  with the maximum planted past element 2^31;
- f8_quantize of a [65536, 32896] bf16 tensor (2.16e9 elements, 4.3 GB):
  the scale and 4,000 sampled codes of both layouts, plus the corners,
  against the oracle's cast of those elements under the oracle's scale of
  the planted amax (the cast is elementwise, so a sample is exact);
- f8_gemm of C [65536, 32896] (2.16e9 outputs) with K = 32: five full
  rows of C against the oracle, the last row included.

tests/test_zz_checked_build.py also runs these cases against the checked
build, whose kernels test every manually indexed access against its
buffer; the TMA copies are clipped by their tensor maps in both builds.
"""
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


def test_amax_past_2_31_elements(f8):
    n = 2 ** 31 + 1000
    x = torch.full((n,), 0.5, dtype=torch.bfloat16, device=DEV)
    x[2 ** 31 + 5] = -7.25
    x[n - 3] = 3.0
    a = f8.f8_amax(x)
    assert f8.f8_last_device_status() == 0
    assert a.item() == 7.25
    del x
    torch.cuda.empty_cache()


def test_quantize_past_2_31_elements(f8):
    rows, cols = 65536, 32896
    assert rows * cols > 2 ** 31
    g = torch.Generator(device=DEV).manual_seed(7)
    x = torch.randn((rows, cols), generator=g, device=DEV, dtype=torch.bfloat16)
    x[rows - 7, cols - 3] = -300.0          # the amax, past element 2^31
    q, qt, s, a = f8.f8_quantize(x)
    assert f8.f8_last_device_status() == 0
    assert a.item() == 300.0
    s_or = oracle.scale(300.0)
    assert s.item() == float(s_or)
    rng = np.random.default_rng(11)
    r = np.concatenate([rng.integers(0, rows, 4000), [0, 0, rows - 1, rows - 1, rows - 7]])
    c = np.concatenate([rng.integers(0, cols, 4000), [0, cols - 1, 0, cols - 1, cols - 3]])
    ri, ci = torch.from_numpy(r).to(DEV), torch.from_numpy(c).to(DEV)
    xs = x[ri, ci].cpu()
    want, _ = oracle.cast_transpose(wl.bits(xs.reshape(1, -1)), s_or)
    assert np.array_equal(q[ri, ci].cpu().numpy(), want[0])
    assert np.array_equal(qt[ci, ri].cpu().numpy(), want[0])
    del x, q, qt
    torch.cuda.empty_cache()


def test_gemm_past_2_31_outputs(f8):
    M, N, K = 65536, 32896, 32
    assert M * N > 2 ** 31
    a = wl.normal((M, K), 1.0, 71).to(DEV)
    b = wl.normal((N, K), 0.05, 72).to(DEV)
    qa, _, sa, _ = f8.f8_quantize(a, want_t=False)
    qb, _, sb, _ = f8.f8_quantize(b, want_t=False)
    c = f8.f8_gemm(qa, qb, sa, sb)
    assert f8.f8_last_device_status() == 0
    qa_h, qb_h = qa.cpu().numpy(), qb.cpu().numpy()
    for row in (0, 255, 40000, M - 256, M - 1):
        ref = oracle.gemm_rows_fmt(qa_h[row:row + 1], 0, qb_h, 0, sa.item(), sb.item())
        check_close(c[row:row + 1], ref, what=f"C row {row}")
    del c
    torch.cuda.empty_cache()
