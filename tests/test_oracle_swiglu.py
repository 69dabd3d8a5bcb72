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


def test_split_ab_index_map_brute_force(oracle_mod):
    """Every column of a and b against the interleaving rule, one element at
    a time: column c of a is AB column 256 (c // 128) + c % 128, column c of
    b the one 128 further."""
    M, F = 3, 384
    ab = np.arange(M * 2 * F, dtype=np.uint16).reshape(M, 2 * F)
    a, b = oracle_mod.split_ab(ab)
    for r in range(M):
        for c in range(F):
            src = 256 * (c // 128) + c % 128
            assert a[r, c] == ab[r, src] and b[r, c] == ab[r, src + 128]


def test_w13_group_rows_are_w1_and_w3(oracle_mod):
    """AB of the interleaved group, split, gives the products with W1 and W3
    under the group's one scale: each sampled element of a (b) is the bf16
    nearest to the exact dot product of a row of X with the W1 (W3) row it
    names, computed here one output at a time from torch's decode of the
    codes."""
    g = torch.Generator().manual_seed(21)
    M, F, K = 4, 256, 32
    x = torch.randn((M, K), generator=g).to(torch.bfloat16)
    w1 = (torch.randn((F, K), generator=g) * 0.02).to(torch.bfloat16)
    w3 = (torch.randn((F, K), generator=g) * 0.05).to(torch.bfloat16)
    rows = []
    for j in range(F // 128):
        rows += [w1[128 * j:128 * (j + 1)], w3[128 * j:128 * (j + 1)]]
    w13 = torch.cat(rows)
    out = oracle_mod.linear_fwd_w13_swiglu(wl.bits(x), wl.bits(w13))
    a, b = oracle_mod.split_ab(out["y"])
    xd = torch.from_numpy(out["x"]["q"]).view(torch.float8_e4m3fn).double().numpy()
    wd = torch.from_numpy(out["w"]["q"]).view(torch.float8_e4m3fn).double().numpy()
    inv = 1.0 / (float(out["x"]["scale"]) * float(out["w"]["scale"]))

    def as_f(bits):
        return float(np.array([bits], np.uint16).astype(np.uint32).__lshift__(16).view(np.float32)[0])

    for r in range(M):
        for c in range(0, F, 37):
            src = 256 * (c // 128) + c % 128
            for got, wrow in ((a[r, c], src), (b[r, c], src + 128)):
                exact = sum(xd[r, k] * wd[wrow, k] for k in range(K)) * inv
                v = as_f(got)
                assert abs(v - exact) <= 0.5 * np.spacing(np.float32(abs(v))) * 2 ** 16 * (1 + 1e-9)
    # the rows W13 names are W1's and W3's
    assert np.array_equal(wl.bits(w13)[256:384], wl.bits(w1)[128:256])
    assert np.array_equal(wl.bits(w13)[384:512], wl.bits(w3)[128:256])
    assert np.array_equal(out["h"], oracle_mod.swiglu_h(a, b))
