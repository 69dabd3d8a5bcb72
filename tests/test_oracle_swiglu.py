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


def _bf(x):
    return torch.tensor(x, dtype=torch.float32).to(torch.bfloat16)


def _f(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).view(torch.bfloat16).double()


def test_swiglu_bwd_against_float64_autograd(oracle_mod):
    """(da, db) against torch autograd of h = silu(a) * b in float64 on the
    same bf16 inputs: equal to the float64 gradient rounded once to bf16
    except within fp32 rounding of a bf16 boundary, and then by one ulp."""
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
        assert float((diff > 0).double().mean()) < 0.02


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
    and db = 0.  a = 20: 1 + exp(-20) rounds to 1 in fp32, so sigma = 1,
    silu' = 1 and da = bf16(dh b), db = bf16(dh a).  dh = 0 gives zeros.
    a = -30: both gradients tiny and of the sign of -dh b and -dh."""
    dh = _bf([1.5, -2.0, 0.0, 1.0, 3.0])
    a = _bf([0.0, 20.0, 5.0, -30.0, 0.0])
    b = _bf([3.0, 0.5, 7.0, 2.0, -1.0])
    da, db = oracle_mod.swiglu_bwd(wl.bits(dh), wl.bits(a), wl.bits(b))
    da, db = _f(da).numpy(), _f(db).numpy()
    assert da[0] == 2.25 and db[0] == 0.0
    assert da[1] == -1.0 and db[1] == -40.0
    assert da[2] == 0.0 and db[2] == 0.0
    assert da[3] < 0 and abs(da[3]) < 1e-10 and db[3] < 0 and abs(db[3]) < 1e-10
    assert da[4] == -1.5 and db[4] == 0.0


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
