"""GPU parity of the E5M2 path against the oracle: E5M2 quantisation (every
byte and the scale bit-exact, including every rounding boundary), mixed
E5M2 x E4M3 GEMMs on both kernel shapes, and the E5M2-gradient backward of
the linear, small in full and one Llama shape at full size (sampled rows)."""
import numpy as np
import pytest
import torch

import oracle
from float8_mixed_precision_gb300 import workloads as wl
from tolerance import check_close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
E4, E5 = 0, 1


@pytest.fixture(scope="module")
def f8():
    import float8_mixed_precision_gb300 as m
    from float8_mixed_precision_gb300 import build
    build.build()
    oracle.build()
    m.lib()
    return m


def _u8(t):
    return t.cpu().numpy()


@pytest.mark.parametrize("shape,std", [((1, 1), 1.0), ((7, 33), 0.01), ((320, 528), 0.01),
                                       ((1024, 4096), 1e-3), ((130, 260), 3.0)])
def test_quantize_e5m2(f8, shape, std):
    x = wl.normal(shape, std, shape[0] * 3 + shape[1])
    q, qt, s, a = f8.f8_quantize(x.to(DEV), fmt=E5)
    ref = oracle.quantize(wl.bits(x), oracle.E5M2)
    assert a.item() == float(ref["amax"]) and s.item() == float(ref["scale"])
    assert np.array_equal(_u8(q), ref["q"]) and np.array_equal(_u8(qt), ref["qt"])


def test_e5m2_every_rounding_boundary(f8):
    """amax = 57344 gives s = 1: the inputs are every E5M2 midpoint, their
    bf16 neighbours and every code value, with both signs."""
    dec = np.array([oracle.e5m2_decode(c) for c in range(0x7C)])
    vals = [57344.0]
    for lo, hi in zip(dec[:-1], dec[1:]):
        b = torch.tensor([(lo + hi) / 2], dtype=torch.float32).to(torch.bfloat16)
        assert b.double().item() == (lo + hi) / 2
        bits = int(b.view(torch.int16).item()) & 0xFFFF
        for nb in (bits - 1, bits, bits + 1):
            vals.append(torch.tensor([nb], dtype=torch.int32).to(torch.int16).view(torch.bfloat16).item())
        vals.append(float(lo))
    vals += [0.0, 2.0 ** -18, 57000.0]
    v = torch.tensor(vals + [-a for a in vals], dtype=torch.bfloat16)
    x = torch.cat([v, torch.zeros((-v.numel()) % 16, dtype=torch.bfloat16)]).reshape(-1, 16)
    q, qt, s, a = f8.f8_quantize(x.to(DEV), fmt=E5)
    ref = oracle.quantize(wl.bits(x), oracle.E5M2)
    assert s.item() == 1.0 and ref["scale"] == 1.0
    assert np.array_equal(_u8(q), ref["q"]) and np.array_equal(_u8(qt), ref["qt"])


def _codes(shape, seed, fmt):
    g = torch.Generator().manual_seed(seed)
    t = torch.randint(0, 256, shape, generator=g, dtype=torch.uint8)
    if fmt == E5:
        t[(t & 0x7F) >= 0x7C] = 0x3C
    else:
        t[(t & 0x7F) == 0x7F] = 0x38
    return t


@pytest.mark.parametrize("M,N,K,fa,fb", [(37, 50, 48, E5, E4), (300, 520, 400, E5, E4),
                                         (640, 1024, 2048, E5, E4), (256, 256, 512, E5, E5),
                                         (512, 384, 1024, E4, E5)])
def test_gemm_mixed_formats(f8, M, N, K, fa, fb, monkeypatch):
    a, b = _codes((M, K), M * 5 + K, fa), _codes((N, K), N * 3 + K, fb)
    sa, sb = np.float32(3.0 if fa == E4 else 1e-3), np.float32(0.5 if fb == E4 else 2e-3)
    ref = oracle.gemm_rows_fmt(a.numpy(), fa, b.numpy(), fb, sa, sb)
    outs = []
    for v in ("1", "2"):
        monkeypatch.setenv("F8_GEMM_VARIANT", v)
        c = f8.f8_gemm(a.to(DEV), b.to(DEV), torch.tensor(sa, device=DEV), torch.tensor(sb, device=DEV),
                       fmt_a=fa, fmt_b=fb)
        check_close(c, ref, what=f"gemm {fa}x{fb} {M}x{N}x{K} variant {v}")
        outs.append(c)
    assert torch.equal(outs[0], outs[1])
    assert f8.f8_last_device_status() == 0


@pytest.mark.parametrize("M,N,K", [(256, 512, 256), (272, 400, 528)])
def test_linear_backward_e5m2_full_compare(f8, M, N, K):
    d = wl.custom_linear(M, K, N, seed=M * 7 + N, dy_std=0.01)
    y, saved = f8.f8_linear_fwd(d["x"].to(DEV), d["w"].to(DEV))
    dx, dw = f8.f8_linear_bwd(d["dy"].to(DEV), saved, dy_fmt=E5)
    assert f8.f8_last_device_status() == 0
    fwd = oracle.linear_fwd(wl.bits(d["x"]), wl.bits(d["w"]))
    bwd = oracle.linear_bwd(wl.bits(d["dy"]), fwd, dy_fmt=oracle.E5M2)
    check_close(dx, bwd["dx"], what="dX (E5M2 dY)")
    check_close(dw, bwd["dw"], what="dW (E5M2 dY)")


def test_linear_backward_e5m2_llama_wq_full_size(f8):
    c, l = 2, 0
    lin = wl.workload(c)[1][l]
    d = wl.linear_inputs(c, l)
    y, saved = f8.f8_linear_fwd(d["x"].to(DEV), d["w"].to(DEV))
    dx, dw = f8.f8_linear_bwd(d["dy"].to(DEV), saved, dy_fmt=E5)
    assert f8.f8_last_device_status() == 0
    qx = oracle.quantize(wl.bits(d["x"]))
    qw = oracle.quantize(wl.bits(d["w"]))
    qdy = oracle.quantize(wl.bits(d["dy"]), oracle.E5M2)
    rng = np.random.default_rng(9)
    rows = np.array([b * 128 + rng.integers(0, 128) for b in range(lin.M // 128)], np.int64)
    ref = oracle.gemm_rows_fmt(qdy["q"], oracle.E5M2, qw["qt"], oracle.E4M3, qdy["scale"], qw["scale"], rows)
    check_close(dx[torch.from_numpy(rows).to(DEV)], ref, what="dX rows (E5M2 dY)")
    rows = np.array([b * 128 + rng.integers(0, 128) for b in range(lin.N // 128)], np.int64)
    ref = oracle.gemm_rows_fmt(qdy["qt"], oracle.E5M2, qx["qt"], oracle.E4M3, qdy["scale"], qx["scale"], rows)
    check_close(dw[torch.from_numpy(rows).to(DEV)], ref, what="dW rows (E5M2 dY)")


@pytest.mark.parametrize("shapes", [
    ((300, 520, 400, E5, E4), (640, 1024, 2048, E4, E4)),   # ragged + costlier second problem
    ((1024, 256, 4096, E4, E5), (256, 1536, 512, E5, E5)),  # costlier first problem
    ((37, 50, 48, E5, E4), (100, 60, 32, E4, E4)),          # both on the single-CTA kernel
    ((512, 384, 1024, E4, E4), (0, 64, 64, E4, E4)),        # an empty problem: separate launches
])
def test_gemm_grouped_matches_single_launches(f8, shapes, monkeypatch):
    """f8_gemm_grouped on two problems of different shapes and formats (the
    grouping forced on) writes the bits f8_gemm writes for each alone, and
    both match the oracle."""
    monkeypatch.setenv("F8_GEMM_GROUP", "2")
    probs, refs, singles = [], [], []
    for i, (M, N, K, fa, fb) in enumerate(shapes):
        a, b = _codes((M, K), 11 * i + M + K, fa), _codes((N, K), 13 * i + N + K, fb)
        sa, sb = np.float32(2.0 if fa == E4 else 1e-3), np.float32(0.25 if fb == E4 else 4e-3)
        ad, bd = a.to(DEV), b.to(DEV)
        sad, sbd = torch.tensor(sa, device=DEV), torch.tensor(sb, device=DEV)
        probs.append((ad, bd, sad, sbd, None, fa, fb))
        refs.append(oracle.gemm_rows_fmt(a.numpy(), fa, b.numpy(), fb, sa, sb) if M else None)
        singles.append(f8.f8_gemm(ad, bd, sad, sbd, fmt_a=fa, fmt_b=fb))
    outs = f8.f8_gemm_grouped(probs)
    assert f8.f8_last_device_status() == 0
    for out, single, ref, (M, N, K, fa, fb) in zip(outs, singles, refs, shapes):
        assert torch.equal(out.view(torch.int16), single.view(torch.int16))
        if ref is not None:
            check_close(out, ref, what=f"grouped gemm {M}x{N}x{K}")


def test_gemm_grouped_one_problem_is_f8_gemm(f8):
    a, b = _codes((512, 1024), 1, E4), _codes((768, 1024), 2, E4)
    s = torch.tensor(1.5, device=DEV)
    one = f8.f8_gemm_grouped([(a.to(DEV), b.to(DEV), s, s)])[0]
    assert torch.equal(one, f8.f8_gemm(a.to(DEV), b.to(DEV), s, s))
    assert f8.f8_last_device_status() == 0
