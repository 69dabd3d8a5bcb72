"""Pins of the oracle's SwiGLU step (the input of the w2 linear and its
gradient).

The oracle takes the definition: h = silu(a) b with silu(a) = a / (1 +
exp(-a)), formed in fp64 from the bf16 inputs and rounded once to bf16, and
the gradient db = dh silu(a), da = dh b silu'(a), likewise.  These tests tie
it to things other than itself:
- the same quantities in 60-digit arithmetic (mpmath), rounded to bf16 by a
  brute-force nearest-value search over neighbouring bf16 codes (exact
  comparisons), for random, large, tiny and boundary inputs;
- silu'(a) from mpmath's numerical differentiation of silu, not from the
  closed form sigma (1 + a (1 - sigma)) the oracle uses;
- torch's float64 autograd of silu(a) * b;
- a central finite difference of the float64 silu;
- exact special cases (a = 0, large |a|, dh = 0, non-finite a).
"""
import math

import numpy as np
import pytest
import torch

from float8_mixed_precision_gb300 import workloads as wl


def _bits_f(bits):
    """float64 values of bf16 bit patterns."""
    b = np.ascontiguousarray(np.asarray(bits, np.uint16))
    return torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).double().numpy()


def _bf16_value(code):
    return float(np.array([code << 16], np.uint32).view(np.float32)[0])


def _nearest_bf16(mp, x):
    """bf16 bits nearest to the mpmath value x (ties to the even code): a
    binary search over the finite non-negative codes (their values increase
    with the code) finds the two that bracket |x|, compared exactly; past the
    midpoint between the largest finite value and 2^128 the result is inf."""
    if mp.isnan(x):
        return 0x7FC0
    sign = 0x8000 if x < 0 else 0
    a = abs(x)
    if mp.isinf(a):
        return sign | 0x7F80
    top = mp.mpf(_bf16_value(0x7F7F))
    if a >= top + (mp.mpf(2) ** 128 - top) / 2:
        return sign | 0x7F80   # at or past the midpoint to 2^128 (a tie goes to the even code, inf)
    lo, hi = 0, 0x7F7F          # invariant: value(lo) <= a
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if mp.mpf(_bf16_value(mid)) <= a:
            lo = mid
        else:
            hi = mid - 1
    if lo == 0x7F7F:
        return sign | lo
    d_lo = a - mp.mpf(_bf16_value(lo))
    d_hi = mp.mpf(_bf16_value(lo + 1)) - a
    if d_lo < d_hi or (d_lo == d_hi and lo % 2 == 0):
        return sign | lo
    return sign | (lo + 1)


def _mp():
    mp = pytest.importorskip("mpmath").mp
    mp.dps = 60
    return mp


def _near_boundary(mp, x, rel=2.0 ** -45):
    """Whether x lies within `rel` (relative) of a bf16 rounding boundary,
    where an fp64 evaluation may round either way."""
    a = abs(x)
    if a == 0 or mp.isinf(a) or mp.isnan(a):
        return False
    c = _nearest_bf16(mp, a) & 0x7FFF
    if c >= 0x7F80:
        return False
    v = mp.mpf(_bf16_value(c))
    for n in (c - 1, c + 1):
        if 0 <= n <= 0x7F7F:
            mid = (v + mp.mpf(_bf16_value(n))) / 2
            if abs(a - mid) <= rel * a:
                return True
    return False


def _mp_silu(mp, a):
    return a / (1 + mp.exp(-a))


def _inputs_h():
    g = torch.Generator().manual_seed(12)
    a = torch.randn(3000, generator=g)
    b = torch.randn(3000, generator=g)
    special_a = [0.0, -0.0, 1.0, -1.0, 2.5, -1.28125, -20.0, 20.0, 36.0, -36.0, 87.0, -87.0, 88.5,
                 -88.5, -89.0, -92.0, -95.0, -100.0, -104.0, -110.0, 100.0, 1e10, -1e10, 3e38, -3e38,
                 1e-30, -1e-30, 1e-38, 5e-40]
    special_b = [1.0, -2.0, 0.5, 3.0, -1.5, 7.0, 1e30, -1e-20, 1.0, 1.125]
    sa = torch.tensor([v for v in special_a for _ in special_b])
    sb = torch.tensor([v for _ in special_a for v in special_b])
    a = torch.cat([a, a * 8, sa]).to(torch.bfloat16)
    b = torch.cat([b, b, sb]).to(torch.bfloat16)
    return a, b


def test_swiglu_h_is_the_correctly_rounded_definition(oracle_mod):
    """h equals the 60-digit silu(a) b rounded to the nearest bf16, except
    where that exact value lies within 2^-45 (relative) of a bf16 rounding
    boundary: there the fp64 evaluation may land on either side and h may be
    either neighbour (e.g. a subnormal a, b = 1: silu(a) = a / (2 - a) is a
    hair above the midpoint a / 2, which fp64 rounds to exactly)."""
    mp = _mp()
    a, b = _inputs_h()
    h = oracle_mod.swiglu_h(wl.bits(a), wl.bits(b))
    av, bv = a.double().numpy(), b.double().numpy()
    near = 0
    for i in range(av.size):
        ea, eb = mp.mpf(av[i]), mp.mpf(bv[i])
        exact = _mp_silu(mp, ea) * eb
        want = _nearest_bf16(mp, exact)
        if exact == 0:
            # the sign of a zero product: sign(a) * sign(b) (silu(a) keeps a's sign)
            want = (0x8000 if (math.copysign(1, av[i]) * math.copysign(1, bv[i])) < 0 else 0)
        got = int(h[i])
        if got != want and _near_boundary(mp, exact):
            near += 1
            assert abs(got - want) == 1 and (got ^ want) & 0x8000 == 0, (av[i], bv[i])
            continue
        assert got == want, (av[i], bv[i], hex(got), hex(want))
    assert near <= 8, near


def test_silu_against_high_precision(oracle_mod):
    """silu in fp64 within 4 fp64 ulp of the 60-digit value, and its
    special values: silu(0) = 0, silu(-800) = -0 (exp(800) overflows),
    silu(800) = 800, silu(+inf) = inf, silu(-inf) and silu(nan) are NaN."""
    mp = _mp()
    xs = np.concatenate([np.linspace(-60, 60, 2401), np.linspace(-1e-3, 1e-3, 101),
                         [-700.0, -300.0, 300.0, 1e-300]])
    for x in xs:
        ref = _mp_silu(mp, mp.mpf(float(x)))
        got = oracle_mod.silu(float(x))
        if ref == 0:
            assert got == 0
            continue
        assert abs(mp.mpf(got) - ref) <= 4 * np.spacing(abs(float(ref))), (x, got, ref)
    assert oracle_mod.silu(0.0) == 0.0
    assert oracle_mod.silu(-800.0) == 0.0 and math.copysign(1.0, oracle_mod.silu(-800.0)) == -1.0
    assert oracle_mod.silu(800.0) == 800.0
    assert oracle_mod.silu(math.inf) == math.inf
    assert math.isnan(oracle_mod.silu(-math.inf)) and math.isnan(oracle_mod.silu(math.nan))


def test_swiglu_bwd_against_high_precision_derivative(oracle_mod):
    """(da, db) equal the 60-digit dh silu'(a) b and dh silu(a) rounded to the
    nearest bf16, with silu'(a) taken by mpmath's numerical differentiation
    of silu (independent of the closed form the oracle evaluates)."""
    mp = _mp()
    g = torch.Generator().manual_seed(31)
    n = 600
    a = torch.cat([torch.randn(n, generator=g) * 3,
                   torch.tensor([0.0, -1.28125, -1.2734375, 20.0, -20.0, -30.0, 45.0, -88.5, -95.0])])
    b = torch.randn(a.numel(), generator=g)
    dh = torch.randn(a.numel(), generator=g)
    a, b, dh = a.to(torch.bfloat16), b.to(torch.bfloat16), dh.to(torch.bfloat16)
    da, db = oracle_mod.swiglu_bwd(wl.bits(dh), wl.bits(a), wl.bits(b))
    av, bv, dv = a.double().numpy(), b.double().numpy(), dh.double().numpy()
    f = lambda t: _mp_silu(mp, t)
    for i in range(av.size):
        ea, eb, ed = mp.mpf(av[i]), mp.mpf(bv[i]), mp.mpf(dv[i])
        d1 = mp.diff(f, ea)
        want_da = _nearest_bf16(mp, ed * eb * d1)
        want_db = _nearest_bf16(mp, ed * f(ea))
        # exact zeros: the sign follows the factors' signs
        if ed * eb * d1 == 0 or ed * f(ea) == 0:
            continue
        for name, got, want, exact in (("da", int(da[i]), want_da, ed * eb * d1),
                                       ("db", int(db[i]), want_db, ed * f(ea))):
            if got != want and _near_boundary(mp, exact):
                assert abs(got - want) == 1, (name, av[i])
                continue
            assert got == want, (name, av[i], bv[i], dv[i], hex(got), hex(want))


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


def _bf(x):
    return torch.tensor(x, dtype=torch.float32).to(torch.bfloat16)


def _f(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).view(torch.bfloat16).double()


def test_swiglu_bwd_against_float64_autograd(oracle_mod):
    """(da, db) against torch autograd of h = silu(a) * b in float64 on the
    same bf16 inputs, rounded to bf16: equal except where torch's float64
    arithmetic and the oracle's land on either side of a bf16 boundary, and
    then by one ulp."""
    shape = (200, 300)
    g = torch.Generator().manual_seed(31)
    a = (torch.randn(shape, generator=g) * 2).to(torch.bfloat16)
    b = torch.randn(shape, generator=g).to(torch.bfloat16)
    dh = torch.randn(shape, generator=g).to(torch.bfloat16)
    da, db = oracle_mod.swiglu_bwd(wl.bits(dh), wl.bits(a), wl.bits(b))
    ad = a.double().requires_grad_()
    bd = b.double().requires_grad_()
    (torch.nn.functional.silu(ad) * bd).backward(dh.double())
    for got, ref in ((_f(da), ad.grad), (_f(db), bd.grad)):
        ref_bf = ref.to(torch.bfloat16).double()
        ulp = torch.from_numpy(np.spacing(np.abs(ref_bf.float().numpy())).astype(np.float64)) * 2 ** 16
        diff = (got - ref_bf).abs()
        assert bool((diff <= ulp * (1 + 1e-9)).all()), float((diff / ulp).max())
        assert float((diff > 0).double().mean()) < 1e-3


def test_silu_derivative_by_finite_differences(oracle_mod):
    """With dh = b = 1, da is bf16(silu'(a)): checked against a central
    difference of the float64 silu (independent of the formula the oracle
    uses), to within one bf16 ulp."""
    xs = np.concatenate([np.linspace(-12, 12, 241), [-0.5, -1e-3, 1e-3, 0.25]])
    a = _bf(xs)
    one = _bf(np.ones_like(xs))
    da, db = oracle_mod.swiglu_bwd(wl.bits(one), wl.bits(a), wl.bits(one))
    silu = lambda v: v / (1.0 + np.exp(-v))
    for v, got in zip(a.double().numpy(), _f(da).numpy()):
        hstep = 1e-6 * max(1.0, abs(v))
        fd = (silu(v + hstep) - silu(v - hstep)) / (2 * hstep)
        ulp = np.spacing(np.float32(abs(fd))) * 2 ** 16 if fd != 0 else 1e-30
        assert abs(got - fd) <= ulp + 1e-9, (v, got, fd)
    # db with dh = 1 is bf16(silu(a))
    for v, got in zip(a.double().numpy(), _f(db).numpy()):
        ref = silu(v)
        assert abs(got - ref) <= np.spacing(np.float32(abs(ref))) * 2 ** 16 + 1e-30, (v, got, ref)


def test_swiglu_bwd_special_cases(oracle_mod):
    """a = 0: sigma = 1/2 and silu'(0) = 1/2 exactly, so da = bf16(dh b / 2)
    and db = 0.  a = 20: silu'(20) = 1 + 4e-8 and sigma = 1 - 2e-9, so da =
    bf16(dh b) and db = bf16(dh a).  dh = 0 gives zeros.  a = -30: both
    gradients tiny and of the sign of -dh b and -dh.  a = -inf or +inf:
    silu' is NaN (0 * inf)."""
    dh = _bf([1.5, -2.0, 0.0, 1.0, 3.0, 1.0, 1.0])
    a = _bf([0.0, 20.0, 5.0, -30.0, 0.0, -math.inf, math.inf])
    b = _bf([3.0, 0.5, 7.0, 2.0, -1.0, 1.0, 1.0])
    da, db = oracle_mod.swiglu_bwd(wl.bits(dh), wl.bits(a), wl.bits(b))
    da, db = _f(da).numpy(), _f(db).numpy()
    assert da[0] == 2.25 and db[0] == 0.0
    assert da[1] == -1.0 and db[1] == -40.0
    assert da[2] == 0.0 and db[2] == 0.0
    assert da[3] < 0 and abs(da[3]) < 1e-10 and db[3] < 0 and abs(db[3]) < 1e-10
    assert da[4] == -1.5 and db[4] == 0.0
    assert math.isnan(da[5]) and math.isnan(db[5])
    assert math.isnan(da[6]) and db[6] == math.inf


def test_swiglu_h_special_values(oracle_mod):
    """h for non-finite and extreme a: silu(+inf) b = inf * sign(b);
    silu(-inf) = NaN; silu(a) = a exactly for a > 37 (exp(-a) < 2^-53), so h
    = bf16(a b); a = -800: h is a zero with the sign of -b."""
    a = _bf([math.inf, math.inf, -math.inf, 40.0, 96.0, -800.0, -800.0])
    b = _bf([2.0, -1.0, 1.0, 1.5, 3.0, 1.0, -1.0])
    h = _f(oracle_mod.swiglu_h(wl.bits(a), wl.bits(b))).numpy()
    assert h[0] == math.inf and h[1] == -math.inf and math.isnan(h[2])
    assert h[3] == 60.0 and h[4] == 288.0
    assert h[5] == 0.0 and math.copysign(1, h[5]) == -1.0
    assert h[6] == 0.0 and math.copysign(1, h[6]) == 1.0


def test_merge_ab_inverts_split_ab(oracle_mod):
    M, F = 4, 384
    rng = np.random.default_rng(5)
    a = rng.integers(0, 1 << 16, (M, F), dtype=np.uint16)
    b = rng.integers(0, 1 << 16, (M, F), dtype=np.uint16)
    ab = oracle_mod.merge_ab(a, b)
    assert ab.shape == (M, 2 * F)
    a2, b2 = oracle_mod.split_ab(ab)
    assert np.array_equal(a, a2) and np.array_equal(b, b2)
    for c in range(F):
        src = 256 * (c // 128) + c % 128
        assert np.array_equal(ab[:, src], a[:, c]) and np.array_equal(ab[:, src + 128], b[:, c])
