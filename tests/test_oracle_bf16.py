"""Pins of the oracle's round-to-nearest-even fp64 -> bf16 step.

- torch's fp32 -> bf16 conversion (RNE) on values that are exact in fp32,
  where a single rounding is all there is;
- exact rational rounding (Fractions) on fp64 values just off a bf16
  midpoint, where rounding through fp32 first would give the wrong answer;
- the format's landmarks: 1.0 = 0x3F80, largest finite (2 - 2^-7) * 2^127 =
  0x7F7F, overflow to 0x7F80, smallest subnormal 2^-133 = 0x0001.
"""
from fractions import Fraction

import numpy as np
import torch


def _exact_round(y: float) -> int:
    """Nearest bf16 by exact search over the two fp32-truncated neighbours."""
    fy = Fraction(y)
    sign = 0x8000 if y < 0 else 0
    a = abs(fy)
    # candidates: the bf16 below (truncate) and the next one up
    lo_bits = int(np.array([abs(y)], np.float32).view(np.uint32)[0] >> 16)
    cands = []
    for b in (lo_bits - 1, lo_bits, lo_bits + 1, lo_bits + 2):
        if 0 <= b <= 0x7F80:
            v = Fraction(0) if b == 0 else Fraction(float(np.array([b << 16], np.uint32).view(np.float32)[0]))
            cands.append((abs(v - a), b & 1, b))
    best = min(cands)
    return sign | best[2]


def test_landmarks(oracle_mod):
    assert oracle_mod.f64_to_bf16(1.0) == 0x3F80
    assert oracle_mod.f64_to_bf16(-2.0) == 0xC000
    assert oracle_mod.f64_to_bf16((2 - 2 ** -7) * 2.0 ** 127) == 0x7F7F
    assert oracle_mod.f64_to_bf16(2.0 ** 128) == 0x7F80
    assert oracle_mod.f64_to_bf16((2 - 2 ** -8) * 2.0 ** 127) == 0x7F80   # midpoint to 2^128: ties to even -> inf
    assert oracle_mod.f64_to_bf16(2.0 ** -133) == 0x0001
    assert oracle_mod.f64_to_bf16(2.0 ** -134) == 0x0000                  # tie -> even (0)
    assert oracle_mod.f64_to_bf16(1.5 * 2.0 ** -134) == 0x0001
    assert oracle_mod.f64_to_bf16(0.0) == 0x0000
    assert oracle_mod.f64_to_bf16(-0.0) == 0x8000
    assert oracle_mod.f64_to_bf16(float("inf")) == 0x7F80


def test_matches_torch_on_fp32_values(oracle_mod):
    g = torch.Generator().manual_seed(3)
    v = torch.cat([torch.randn(3000, generator=g) * s for s in (1e-39, 1e-20, 1.0, 1e10, 1e37)])
    v = v.to(torch.float32)
    ref = v.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).tolist()
    got = [oracle_mod.f64_to_bf16(x) for x in v.tolist()]
    assert got == ref


def test_no_double_rounding(oracle_mod):
    rng = np.random.default_rng(11)
    n = 0
    for _ in range(400):
        e = int(rng.integers(-120, 120))
        m = int(rng.integers(128, 256))
        mid = (m + 0.5) * 2.0 ** (e - 7)          # a bf16 midpoint, exact in fp64
        for off in (2.0 ** (e - 40), -(2.0 ** (e - 40)), 0.0):
            y = mid + off
            assert oracle_mod.f64_to_bf16(y) == _exact_round(y), (y, off)
            assert oracle_mod.f64_to_bf16(-y) == (_exact_round(y) | 0x8000)
            n += 1
    assert n == 1200
