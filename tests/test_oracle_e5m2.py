"""Pins of the oracle's E5M2 codec and mixed-format GEMM.

- landmarks of the format (tests/golden/e5m2_landmarks.txt, from the FP8
  formats paper cited by the torchtitan walkthrough, Part XI item 9);
- torch's float8_e5m2 decode of all 256 codes and RNE encode in range;
- brute-force nearest-code search in exact rationals at every boundary;
- saturation and signed zero;
- the __int128 mixed-format GEMM against exact Python integer arithmetic
  and, where every sum is below 2^53, against numpy's float64 matmul;
- E4M3 x E4M3 through the mixed route equals the int64 route;
- the E5M2-gradient backward against the unquantised product (SQNR).
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from float8_mixed_precision_gb300 import workloads as wl
from test_oracle_gemm import _bf16_bits_of_f64, _bits_to_f64, _dec, _sqnr_db

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e5m2_landmarks.txt")


def _torch_decode_all():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e5m2).to(torch.float64).numpy()


def _dec5(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e5m2).to(torch.float64).numpy()


def test_landmarks(oracle_mod):
    n = 0
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        code_s, val_s = line.split()
        got = oracle_mod.e5m2_decode(int(code_s, 16))
        if val_s == "nan":
            assert math.isnan(got)
        else:
            want = float(val_s)
            assert got == want and math.copysign(1, got) == math.copysign(1, want), code_s
        n += 1
    assert n >= 12


def test_decode_all_codes_matches_torch(oracle_mod):
    ref = _torch_decode_all()
    for c in range(256):
        got = oracle_mod.e5m2_decode(c)
        if math.isnan(ref[c]):
            assert math.isnan(got), c
        else:
            assert got == ref[c] and math.copysign(1, got) == math.copysign(1, ref[c]), c


def test_roundtrip_finite_codes(oracle_mod):
    for c in range(256):
        v = oracle_mod.e5m2_decode(c)
        if math.isnan(v) or math.isinf(v):
            continue
        assert oracle_mod.e5m2_encode(v) == c, hex(c)


def _brute(v, grid):
    sign = 0x80 if math.copysign(1.0, v) < 0 else 0
    a = abs(v)
    if math.isinf(a) or a >= 57344:
        return sign | 0x7B
    fa = Fraction(a)
    return sign | min(grid, key=lambda gc: (abs(gc[0] - fa), gc[1] & 1))[1]


def test_every_boundary_brute_force(oracle_mod):
    ref = _torch_decode_all()
    grid = [(Fraction(float(ref[c])), c) for c in range(0x7C)]
    vals = sorted(g[0] for g in grid)
    probes = []
    for lo, hi in zip(vals[:-1], vals[1:]):
        mid = float((lo + hi) / 2)
        f = np.float32(mid)
        probes += [float(np.nextafter(f, np.float32(-np.inf))), float(f),
                   float(np.nextafter(f, np.float32(np.inf))), float(lo)]
    probes += [57344.0, 61439.0, 61440.0, 1e30, float("inf"), 2.0 ** -17, 2.0 ** -30]
    for p in probes:
        for v in (p, -p):
            assert oracle_mod.e5m2_encode(v) == _brute(v, grid), v


def test_encode_matches_torch_in_range(oracle_mod):
    g = torch.Generator().manual_seed(5)
    v = torch.cat([torch.randn(3000, generator=g) * s for s in (1e-4, 1.0, 300.0, 2e4)]).float()
    v = v[v.abs() < 57344]
    ref = v.to(torch.float8_e5m2).view(torch.uint8).tolist()
    assert [oracle_mod.e5m2_encode(float(x)) for x in v.tolist()] == ref


def test_scale_and_cast(oracle_mod):
    assert oracle_mod.scale_fmt(1.0, oracle_mod.E5M2) == 57344.0
    assert oracle_mod.scale_fmt(1.0, oracle_mod.E4M3) == oracle_mod.scale(1.0)
    x = wl.normal((64, 96), 0.01, 3)
    q = oracle_mod.quantize(wl.bits(x), oracle_mod.E5M2)
    assert np.abs(_dec5(q["q"])).max() == 57344.0
    v = torch.clamp(x.float() * torch.tensor(q["scale"]), -57344, 57344)
    assert np.array_equal(q["q"], v.to(torch.float8_e5m2).view(torch.uint8).numpy())
    assert np.array_equal(q["qt"], q["q"].T)


def _codes(shape, seed, fmt):
    g = torch.Generator().manual_seed(seed)
    t = torch.randint(0, 256, shape, generator=g, dtype=torch.uint8)
    if fmt == 1:
        t[(t & 0x7F) >= 0x7C] = 0x3C     # no inf / NaN codes
    else:
        t[(t & 0x7F) == 0x7F] = 0x38
    return t.numpy()


def test_mixed_gemm_exact_integers(oracle_mod):
    a, b = _codes((6, 40), 1, 1), _codes((5, 40), 2, 0)
    a[0, :] = 0x7B                        # all +57344: the largest sums
    b[0, :] = 0x7E                        # all +448
    sa, sb = 2.0, 0.5
    got = oracle_mod.gemm_rows_fmt(a, 1, b, 0, sa, sb)
    ea = [Fraction(x) for x in _dec5(a).reshape(-1)]
    eb = [Fraction(x) for x in _dec(b).reshape(-1)]
    for m in range(6):
        for n in range(5):
            exact = sum(ea[m * 40 + k] * eb[n * 40 + k] for k in range(40)) / Fraction(sa * sb)
            assert got[m, n] == _bf16_bits_of_f64(np.float64(float(exact))), (m, n)


def test_mixed_gemm_matches_numpy(oracle_mod):
    a, b = _codes((33, 256), 3, 1), _codes((17, 256), 4, 0)
    sa, sb = np.float32(7.0), np.float32(0.125)
    ref = (_dec5(a) @ _dec(b).T) / (np.float64(sa) * np.float64(sb))
    assert np.array_equal(oracle_mod.gemm_rows_fmt(a, 1, b, 0, sa, sb), _bf16_bits_of_f64(ref))


def test_mixed_route_equals_e4m3_route(oracle_mod):
    a, b = _codes((20, 64), 5, 0), _codes((12, 64), 6, 0)
    assert np.array_equal(oracle_mod.gemm_rows_fmt(a, 0, b, 0, 3.0, 5.0), oracle_mod.gemm(a, b, 3.0, 5.0))


def test_e5m2_backward_quality(oracle_mod):
    d = wl.custom_linear(96, 128, 80, seed=77, dy_std=0.01)
    f = oracle_mod.linear_fwd(wl.bits(d["x"]), wl.bits(d["w"]))
    b = oracle_mod.linear_bwd(wl.bits(d["dy"]), f, dy_fmt=oracle_mod.E5M2)
    x, w, dy = (d[k].to(torch.float64).numpy() for k in ("x", "w", "dy"))
    for ref, got in [(dy @ w, b["dx"]), (dy.T @ x, b["dw"])]:
        s = _sqnr_db(ref, _bits_to_f64(got))
        assert 17.0 <= s < 30.0, s
