"""Pins of the oracle's SwiGLU step (the input of the w2 linear).

exp is Cody-Waite range reduction plus the degree-7 Taylor polynomial in
fp32; it is checked against the exact exponential (math.exp) over the finite
range, silu against its float64 definition, and h = bf16(silu(a) * b)
against the same product formed in float64 and rounded once to bf16: the two
agree except where the fp32 route lands within an fp32 ulp or two of a bf16
rounding boundary, and then by one bf16 ulp.
"""
import math

import numpy as np
import torch

from float8_mixed_precision_gb300 import workloads as wl


def _ulp32(v):
    return np.spacing(np.float32(abs(v)))


def test_exp_error_bound(oracle_mod):
    xs = np.concatenate([np.linspace(-87.0, 88.0, 20001), np.linspace(-1, 1, 2001)]).astype(np.float32)
    worst = 0.0
    for x in xs:
        got = oracle_mod.exp_cw(float(x))
        ref = math.exp(float(x))
        worst = max(worst, abs(got - ref) / _ulp32(ref))
    assert worst <= 2.0, worst
    assert oracle_mod.exp_cw(0.0) == 1.0
    assert oracle_mod.exp_cw(100.0) == math.inf and oracle_mod.exp_cw(-100.0) == 0.0


def test_silu_error_bound(oracle_mod):
    xs = np.concatenate([np.linspace(-30, 30, 6001), np.linspace(-1e-3, 1e-3, 101)]).astype(np.float32)
    worst = 0.0
    for x in xs:
        xd = float(x)
        ref = xd / (1.0 + math.exp(-xd))
        got = oracle_mod.silu(xd)
        if ref != 0.0:
            worst = max(worst, abs(got - ref) / _ulp32(ref))
    assert worst <= 4.0, worst
    assert oracle_mod.silu(0.0) == 0.0
    assert math.copysign(1.0, oracle_mod.silu(-200.0)) == -1.0 and oracle_mod.silu(-200.0) == 0.0
    assert oracle_mod.silu(200.0) == 200.0


def test_swiglu_h_against_float64(oracle_mod):
    shape = (300, 700)
    g = torch.Generator().manual_seed(12)
    a = torch.randn(shape, generator=g).to(torch.bfloat16)
    b = torch.randn(shape, generator=g).to(torch.bfloat16)
    h = oracle_mod.swiglu_h(wl.bits(a), wl.bits(b))
    ad, bd = a.double(), b.double()
    ref = (ad / (1 + torch.exp(-ad)) * bd).to(torch.bfloat16)   # one rounding from float64... via fp32
    got = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16)
    diff = (got.double() - ref.double()).abs()
    ulp = torch.from_numpy(np.spacing(np.abs(ref.float().numpy())).astype(np.float64)) * 2 ** 16
    mismatch = diff > 0
    assert mismatch.float().mean() < 1e-3
    assert bool((diff[mismatch] <= ulp[mismatch] + 1e-30).all())


def test_linear_fwd_swiglu_is_the_linear_of_h(oracle_mod):
    g = torch.Generator().manual_seed(5)
    a = torch.randn(64, 96, generator=g).to(torch.bfloat16)
    b = torch.randn(64, 96, generator=g).to(torch.bfloat16)
    w = (torch.randn(48, 96, generator=g) * 0.02).to(torch.bfloat16)
    f = oracle_mod.linear_fwd_swiglu(wl.bits(a), wl.bits(b), wl.bits(w))
    f2 = oracle_mod.linear_fwd(f["h"], wl.bits(w))
    assert np.array_equal(f["y"], f2["y"]) and np.array_equal(f["x"]["q"], f2["x"]["q"])
