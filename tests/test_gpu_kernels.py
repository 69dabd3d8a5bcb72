"""GPU parity of each kernel against the CPU oracle, through the C ABI.

amax, scales and every E4M3 byte must be bit-exact; GEMM outputs must meet
the bf16 bar of tests/tolerance.py.  Sizes span several tiles with ragged
tails, plus the degenerate cases (empty, one element, all-zero, K == 0).
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
    assert m.f8_last_device_status() == 0
    return m


def _u16(t):
    return wl.bits(t.cpu())


def _u8(t):
    return t.cpu().numpy()


# ------------------------------------------------------------------ amax
@pytest.mark.parametrize("n", [1, 7, 8, 9, 4095, 4097, 65536 + 5, 3_000_001])
def test_amax_sizes(f8, n):
    x = wl.normal((n,), 1.0, 500 + n)
    got = f8.f8_amax(x.to(DEV))
    want, nf = oracle.amax(_u16(x))
    assert not nf
    assert got.item() == float(want)
    assert f8.f8_last_device_status() == 0


def test_amax_special_values(f8):
    z = torch.zeros(10_000, dtype=torch.bfloat16)
    assert f8.f8_amax(z.to(DEV)).item() == 0.0
    for idx, v in [(0, -3.5), (9_999, 2.0 ** -130), (4_444, -448.0), (7, 1e30)]:
        t = z.clone()
        t[idx] = v
        want, _ = oracle.amax(_u16(t))
        assert f8.f8_amax(t.to(DEV)).item() == float(want)
    assert f8.f8_amax(torch.empty(0, dtype=torch.bfloat16, device=DEV)).item() == 0.0
    assert f8.f8_last_device_status() == 0


def test_amax_nonfinite_sets_status(f8):
    t = torch.ones(5000, dtype=torch.bfloat16)
    t[1234] = float("nan")
    f8.f8_amax(t.to(DEV))
    assert f8.f8_last_device_status() == f8.binding.F8_ERR_NONFINITE
    t[1234] = float("-inf")
    f8.f8_amax(t.to(DEV))
    assert f8.f8_last_device_status() == f8.binding.F8_ERR_NONFINITE
    assert f8.f8_last_device_status() == 0     # read-and-clear


# ------------------------------------------------------------------ cast
def _cast_both(f8, x):
    xd = x.to(DEV)
    amax = f8.f8_amax(xd)
    q, qt, s = f8.f8_cast_transpose(xd, amax)
    ref = oracle.quantize(_u16(x))
    return q, qt, s, ref


@pytest.mark.parametrize("shape", [(1, 1), (7, 33), (16, 16), (128, 128), (256, 384), (130, 260),
                                   (320, 528), (96, 100), (100, 96), (1024, 4096)])
def test_cast_transpose_bytes(f8, shape):
    x = wl.normal(shape, 1.0, shape[0] * 7 + shape[1])
    q, qt, s, ref = _cast_both(f8, x)
    assert s.item() == float(ref["scale"])
    assert np.array_equal(_u8(q), ref["q"])
    assert np.array_equal(_u8(qt), ref["qt"])


def test_cast_every_rounding_boundary(f8):
    """amax = 448 gives s = 1, so x * s = x: the bf16 inputs are every E4M3
    midpoint, their bf16 neighbours, every code value, and both signs."""
    dec = np.array([oracle.e4m3_decode(c) for c in range(0x7F)])
    vals = [448.0]
    for lo, hi in zip(dec[:-1], dec[1:]):
        mid = np.float32((lo + hi) / 2)
        b = torch.tensor([mid], dtype=torch.float32).to(torch.bfloat16)
        assert b.float().item() == mid       # midpoints are exact in bf16
        bits = int(b.view(torch.int16).item()) & 0xFFFF
        for nb in (bits - 1, bits, bits + 1):
            vals.append(torch.tensor([nb], dtype=torch.int32).to(torch.int16).view(torch.bfloat16).item())
        vals.append(float(lo))
    vals += [0.0, 2.0 ** -12, 2.0 ** -133, 447.0, 446.0]
    v = torch.tensor(vals + [-a for a in vals], dtype=torch.bfloat16)
    n = v.numel()
    pad = (-n) % 16
    x = torch.cat([v, torch.zeros(pad, dtype=torch.bfloat16)]).reshape(-1, 16)
    q, qt, s, ref = _cast_both(f8, x)
    assert ref["scale"] == 1.0 and s.item() == 1.0
    got, want = _u8(q), ref["q"]
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)[:8]
        detail = [(x[tuple(i)].item(), hex(got[tuple(i)]), hex(want[tuple(i)])) for i in bad]
        raise AssertionError(f"cast differs from the oracle at {detail}")
    assert np.array_equal(_u8(qt), ref["qt"])


def test_cast_saturation_and_outliers(f8):
    x = wl.student_t_outliers((512, 640), 3, 1e-3, 100.0, 77)
    q, qt, s, ref = _cast_both(f8, x)
    assert s.item() == float(ref["scale"])
    assert np.array_equal(_u8(q), ref["q"]) and np.array_equal(_u8(qt), ref["qt"])
    # explicit scale far above 448/amax: everything saturates to +-448
    xd = x.to(DEV)
    big = torch.tensor(1e-30, device=DEV)          # amax 1e-30 -> clamp 1e-12 -> s = 4.48e14
    q2, _, s2 = f8.f8_cast_transpose(xd, big, want_t=False)
    ref2, _ = oracle.cast_transpose(_u16(x), oracle.scale(1e-30))
    assert s2.item() == float(oracle.scale(1e-30))
    assert np.array_equal(_u8(q2), ref2)


def test_cast_all_zero(f8):
    x = torch.zeros((64, 48), dtype=torch.bfloat16)
    q, qt, s, ref = _cast_both(f8, x)
    assert s.item() == float(ref["scale"])
    assert np.array_equal(_u8(q), ref["q"]) and np.array_equal(_u8(qt), ref["qt"])


def test_cast_only_one_layout(f8):
    x = wl.normal((256, 256), 1.0, 3)
    xd = x.to(DEV)
    amax = f8.f8_amax(xd)
    ref = oracle.quantize(_u16(x))
    q, qt, _ = f8.f8_cast_transpose(xd, amax, want_t=False)
    assert qt is None and np.array_equal(_u8(q), ref["q"])
    q, qt, _ = f8.f8_cast_transpose(xd, amax, want_q=False)
    assert q is None and np.array_equal(_u8(qt), ref["qt"])


# ------------------------------------------------------------------ GEMM
def _codes(shape, seed):
    g = torch.Generator().manual_seed(seed)
    t = torch.randint(0, 256, shape, generator=g, dtype=torch.uint8)
    t[(t & 0x7F) == 0x7F] = 0x38   # no NaN codes
    return t


@pytest.mark.parametrize("M,N,K", [(1, 1, 16), (37, 50, 48), (128, 256, 128), (128, 256, 4096),
                                   (300, 520, 400), (129, 257, 1040), (640, 384, 2048),
                                   (1000, 1000, 16), (2048, 2304, 1024)])
def test_gemm_shapes(f8, M, N, K):
    a, b = _codes((M, K), M + K), _codes((N, K), N + 3 * K)
    sa, sb = np.float32(3.5), np.float32(0.25)
    sad = torch.tensor(sa, device=DEV)
    sbd = torch.tensor(sb, device=DEV)
    c = f8.f8_gemm(a.to(DEV), b.to(DEV), sad, sbd)
    ref = oracle.gemm(a.numpy(), b.numpy(), sa, sb)
    check_close(c, ref, what=f"gemm {M}x{N}x{K}")
    assert f8.f8_last_device_status() == 0


def test_gemm_quantised_normal_data(f8):
    """Operands produced by the cast from N(0,1) data (the realistic code mix)."""
    x = wl.normal((384, 1536), 1.0, 8)
    w = wl.normal((512, 1536), 0.02, 9)
    qx = oracle.quantize(_u16(x))
    qw = oracle.quantize(_u16(w))
    c = f8.f8_gemm(torch.from_numpy(qx["q"]).to(DEV), torch.from_numpy(qw["q"]).to(DEV),
                   torch.tensor(qx["scale"], device=DEV), torch.tensor(qw["scale"], device=DEV))
    check_close(c, oracle.gemm(qx["q"], qw["q"], qx["scale"], qw["scale"]), what="gemm N(0,1)")


@pytest.mark.parametrize("sa,sb", [(4.48e14, 4.48e14), (1.3e-30, 2.0), (448.0, 1e-20), (1e-8, 1e-8)])
def test_gemm_extreme_scales(f8, sa, sb):
    a, b = _codes((256, 512), 1), _codes((256, 512), 2)
    sa, sb = np.float32(sa), np.float32(sb)
    c = f8.f8_gemm(a.to(DEV), b.to(DEV), torch.tensor(sa, device=DEV), torch.tensor(sb, device=DEV))
    ref = oracle.gemm(a.numpy(), b.numpy(), sa, sb)
    rb = ref.view(np.int16) & 0x7FFF
    if (rb >= 0x7F80).any():
        pytest.skip("result overflows bf16 at these scales")
    check_close(c, ref, what=f"gemm scales {sa} {sb}")


def test_gemm_degenerate(f8):
    one = torch.tensor(1.0, device=DEV)
    c = torch.full((5, 7), 3.0, dtype=torch.bfloat16, device=DEV)
    f8.f8_gemm(torch.empty((5, 0), dtype=torch.uint8, device=DEV),
               torch.empty((7, 0), dtype=torch.uint8, device=DEV), one, one, out=c)
    assert (c == 0).all()
    c0 = f8.f8_gemm(torch.empty((0, 32), dtype=torch.uint8, device=DEV),
                    torch.zeros((7, 32), dtype=torch.uint8, device=DEV), one, one)
    assert c0.shape == (0, 7)
    with pytest.raises(f8.F8Error):
        f8.f8_gemm(torch.zeros((4, 24), dtype=torch.uint8, device=DEV),
                   torch.zeros((4, 24), dtype=torch.uint8, device=DEV), one, one)


def test_gemm_repeat_is_deterministic(f8):
    a, b = _codes((512, 2048), 5), _codes((768, 2048), 6)
    s = torch.tensor(1.0, device=DEV)
    ad, bd = a.to(DEV), b.to(DEV)
    c1 = f8.f8_gemm(ad, bd, s, s)
    c2 = f8.f8_gemm(ad, bd, s, s)
    assert torch.equal(c1, c2)


# ------------------------------------------------------------------ failure path
def test_wait_timeout_is_reported_and_context_survives(f8):
    f8.f8_selftest_wait_timeout(2_000_000)   # 2 ms limit on a barrier nobody signals
    assert f8.f8_last_device_status() == f8.binding.F8_ERR_TIMEOUT
    assert f8.f8_last_device_status() == 0
    x = torch.ones(100, dtype=torch.bfloat16, device=DEV)
    assert f8.f8_amax(x).item() == 1.0


@pytest.mark.parametrize("M,N,K", [(256, 256, 128), (300, 520, 400), (513, 264, 1040), (640, 1000, 2048),
                                   (1024, 4096, 1024)])
def test_gemm_single_and_pair_kernels(f8, M, N, K, monkeypatch):
    """Both kernel shapes (one CTA per 128-row tile, CTA pairs per 256-row
    tile), each with TMA-store (N % 8 == 0) and direct-store epilogues, match
    the oracle and each other bit for bit (same K order of accumulation)."""
    a, b = _codes((M, K), 3 * M + K), _codes((N, K), N + 7 * K)
    sa, sb = np.float32(1.75), np.float32(0.5)
    sad, sbd = torch.tensor(sa, device=DEV), torch.tensor(sb, device=DEV)
    ref = oracle.gemm(a.numpy(), b.numpy(), sa, sb)
    outs = []
    for v in ("1", "2"):
        monkeypatch.setenv("F8_GEMM_VARIANT", v)
        c = f8.f8_gemm(a.to(DEV), b.to(DEV), sad, sbd)
        check_close(c, ref, what=f"gemm {M}x{N}x{K} variant {v}")
        outs.append(c)
    assert f8.f8_last_device_status() == 0
    assert torch.equal(outs[0], outs[1])


# ------------------------------------------------------------------ quantize (amax partials + cast)
@pytest.mark.parametrize("shape", [(1, 1), (7, 33), (16, 16), (320, 528), (130, 260), (1024, 4096),
                                   (4096, 8192), (8192, 1024)])
def test_quantize_matches_oracle(f8, shape):
    x = wl.normal(shape, 0.3, shape[0] + 11 * shape[1])
    q, qt, s, a = f8.f8_quantize(x.to(DEV))
    ref = oracle.quantize(_u16(x))
    assert a.item() == float(ref["amax"]) and s.item() == float(ref["scale"])
    assert np.array_equal(_u8(q), ref["q"]) and np.array_equal(_u8(qt), ref["qt"])
    assert f8.f8_last_device_status() == 0


def test_quantize_workspace_reuse_and_garbage(f8):
    """The partial maxima need no clean workspace: back-to-back calls on one
    workspace, and a workspace full of random bytes, both give the oracle's
    bytes."""
    ws = torch.randint(0, 256, (f8.f8_quantize_workspace_bytes(),), dtype=torch.uint8, device=DEV)
    for i, (shape, std) in enumerate([((2048, 2048), 1.0), ((512, 4096), 1e-3), ((2048, 2048), 50.0)]):
        x = wl.student_t_outliers(shape, 3, 1e-3, 100.0, 40 + i) if i == 2 else wl.normal(shape, std, 40 + i)
        q, qt, s, a = f8.f8_quantize(x.to(DEV), ws=ws)
        ref = oracle.quantize(_u16(x))
        assert a.item() == float(ref["amax"]) and s.item() == float(ref["scale"])
        assert np.array_equal(_u8(q), ref["q"]) and np.array_equal(_u8(qt), ref["qt"])
    assert f8.f8_last_device_status() == 0


def test_quantize_nonfinite_and_empty(f8):
    t = torch.ones((64, 64), dtype=torch.bfloat16)
    t[5, 6] = float("inf")
    f8.f8_quantize(t.to(DEV))
    assert f8.f8_last_device_status() == f8.binding.F8_ERR_NONFINITE
    q, qt, s, a = f8.f8_quantize(torch.empty((0, 32), dtype=torch.bfloat16, device=DEV))
    assert a.item() == 0.0 and s.item() == float(oracle.scale(0.0))
    assert f8.f8_last_device_status() == 0
