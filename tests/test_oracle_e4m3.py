"""Pins of the oracle's E4M3 codec against facts fixed outside it.

- the format's landmark codes (tests/golden/e4m3_landmarks.txt, from the
  FP8 formats paper cited by the torchtitan walkthrough, Part XI item 9);
- torch's own float8_e4m3fn decode of all 256 codes and its RNE encode of
  in-range fp32 values (an independent library implementation);
- brute-force nearest-code search in exact rational arithmetic at every
  rounding boundary (midpoints and their fp32 neighbours), written here
  without the oracle's binade arithmetic;
- saturation and the sign of zero.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_landmarks.txt")


def _torch_decode_all():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_landmarks(oracle_mod):
    n = 0
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        code_s, val_s = line.split()
        code = int(code_s, 16)
        got = oracle_mod.e4m3_decode(code)
        if val_s == "nan":
            assert math.isnan(got)
        else:
            want = float(val_s)
            assert got == want and math.copysign(1, got) == math.copysign(1, want), (code_s, got)
        n += 1
    assert n >= 10


def test_decode_all_codes_matches_torch(oracle_mod):
    ref = _torch_decode_all()
    for c in range(256):
        got = oracle_mod.e4m3_decode(c)
        if math.isnan(ref[c]):
            assert math.isnan(got), c
        else:
            assert got == ref[c] and math.copysign(1, got) == math.copysign(1, ref[c]), c


def test_encode_decode_roundtrip_all_finite_codes(oracle_mod):
    for c in range(256):
        v = oracle_mod.e4m3_decode(c)
        if math.isnan(v):
            continue
        assert oracle_mod.e4m3_encode(v) == c, hex(c)


def _grid():
    """All non-negative finite E4M3 values with their codes, from torch's decode."""
    ref = _torch_decode_all()
    return [(Fraction(float(ref[c])), c) for c in range(0x7F)]


def _brute_force(v: float, grid) -> int:
    """Nearest code by exhaustive search, ties to the even code, >= 448 saturates."""
    sign = 0x80 if math.copysign(1.0, v) < 0 else 0
    a = abs(v)
    if math.isinf(a) or a >= 448:
        return sign | 0x7E
    fa = Fraction(a)
    best = min(grid, key=lambda gc: (abs(gc[0] - fa), gc[1] & 1))
    return sign | best[1]


def _f32_neighbours(x: float):
    f = np.float32(x)
    return [float(np.nextafter(f, np.float32(-np.inf))), float(f), float(np.nextafter(f, np.float32(np.inf)))]


def test_every_rounding_boundary_brute_force(oracle_mod):
    grid = _grid()
    vals = sorted(g[0] for g in grid)
    probes = []
    for lo, hi in zip(vals[:-1], vals[1:]):
        mid = (lo + hi) / 2
        assert float(mid) == mid  # every midpoint is exact in fp32
        probes += _f32_neighbours(float(mid))
        probes.append(float(lo))
    probes += _f32_neighbours(448.0) + _f32_neighbours(464.0) + [480.0, 1e30, float(np.finfo(np.float32).max)]
    probes += [2.0 ** -10, 2.0 ** -11, 2.0 ** -30, 1e-45]
    n = 0
    for p in probes:
        for v in (p, -p):
            assert oracle_mod.e4m3_encode(v) == _brute_force(v, grid), v
            n += 1
    assert n > 1000


def test_encode_matches_torch_in_range(oracle_mod):
    g = torch.Generator().manual_seed(7)
    v = torch.cat([torch.randn(4000, generator=g) * s for s in (1e-3, 0.05, 1.0, 30.0, 120.0)])
    v = v[v.abs() < 448].to(torch.float32)
    ref = v.to(torch.float8_e4m3fn).view(torch.uint8).tolist()
    got = [oracle_mod.e4m3_encode(float(x)) for x in v.tolist()]
    assert got == ref


def test_saturation_and_signed_zero(oracle_mod):
    for v, want in [(448.0, 0x7E), (449.0, 0x7E), (463.99, 0x7E), (464.0, 0x7E), (465.0, 0x7E),
                    (1e38, 0x7E), (float("inf"), 0x7E), (-float("inf"), 0xFE), (-500.0, 0xFE),
                    (0.0, 0x00), (-0.0, 0x80), (2.0 ** -11, 0x00), (-(2.0 ** -11), 0x80),
                    (2.0 ** -10, 0x00), (1.5 * 2.0 ** -9, 0x02), (2.5 * 2.0 ** -9, 0x02)]:
        assert oracle_mod.e4m3_encode(v) == want, v


def test_grid_spacing_closed_form(oracle_mod):
    # within the binade [2^E, 2^(E+1)) the 8 codes are 2^(E-3) apart (E >= -6);
    # below 2^-6 the spacing is 2^-9.
    for c in range(1, 0x7E):
        d = oracle_mod.e4m3_decode(c + 1) - oracle_mod.e4m3_decode(c)
        v = oracle_mod.e4m3_decode(c)
        E = max(math.floor(math.log2(v)), -6)
        assert d == 2.0 ** (E - 3), hex(c)
