"""Pins of the oracle's amax, scale and cast steps.

amax is checked against numpy's max(|x|) of torch's bf16 widening; the cast
against torch's own fp32 multiply and RNE float8_e4m3fn conversion (after a
clamp to +-448, which is what saturation means); and the scaling recipe
against its invariants: max|dequant(q)| == 448 whenever amax >= 1e-12, and
q unchanged when the tensor is multiplied by a power of two.
"""
import numpy as np
import pytest
import torch

from float8_mixed_precision_gb300 import workloads as wl


def _f32(t):
    return t.to(torch.float32).numpy()


@pytest.mark.parametrize("n", [1, 7, 4095, 4097, 65536 + 3])
def test_amax_matches_numpy(oracle_mod, n):
    x = wl.normal((n,), 1.0, 100 + n)
    a, nf = oracle_mod.amax(wl.bits(x))
    assert not nf
    assert a == np.float32(np.abs(_f32(x)).max())


def test_amax_special_cases(oracle_mod):
    z = torch.zeros(1000, dtype=torch.bfloat16)
    assert oracle_mod.amax(wl.bits(z)) == (0.0, False)
    one = z.clone(); one[517] = -3.5
    assert oracle_mod.amax(wl.bits(one)) == (3.5, False)          # negative max
    sub = z.clone(); sub[3] = torch.tensor(1e-39, dtype=torch.bfloat16)
    a, _ = oracle_mod.amax(wl.bits(sub))
    assert a == np.float32(torch.tensor(1e-39, dtype=torch.bfloat16).float().item())  # bf16 subnormal
    bad = z.clone(); bad[9] = float("inf")
    assert oracle_mod.amax(wl.bits(bad))[1] is True
    bad[9] = float("nan")
    assert oracle_mod.amax(wl.bits(bad))[1] is True


def test_scale_values(oracle_mod):
    assert oracle_mod.scale(1.0) == 448.0
    assert oracle_mod.scale(448.0) == 1.0
    assert oracle_mod.scale(0.0) == np.float32(448.0) / np.float32(1e-12)
    assert np.isfinite(oracle_mod.scale(0.0))
    assert oracle_mod.scale(3.0) == np.float32(448.0) / np.float32(3.0)


def _torch_cast(x, s):
    v = x.to(torch.float32) * torch.tensor(s, dtype=torch.float32)
    v = torch.clamp(v, -448.0, 448.0)
    return v.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


@pytest.mark.parametrize("shape,std", [((64, 80), 1.0), ((33, 17), 0.02), ((128, 256), 3e-3)])
def test_cast_matches_torch(oracle_mod, shape, std):
    x = wl.normal(shape, std, 5)
    q = oracle_mod.quantize(wl.bits(x))
    assert q["scale"] == oracle_mod.scale(np.float32(np.abs(_f32(x)).max()))
    want = _torch_cast(x, q["scale"])
    # torch keeps the sign of -0 as 0x80 as well
    assert np.array_equal(q["q"], want)
    assert np.array_equal(q["qt"], q["q"].T)


def test_cast_outliers_and_saturation(oracle_mod):
    x = wl.student_t_outliers((96, 160), 3, 1e-2, 100.0, 9)
    q = oracle_mod.quantize(wl.bits(x))
    assert np.array_equal(q["q"], _torch_cast(x, q["scale"]))
    # a value beyond amax * s (impossible by construction) is checked with an explicit scale
    big = torch.tensor([[1.0, -2.0, 3.0, 1000.0]], dtype=torch.bfloat16)
    qq, _ = oracle_mod.cast_transpose(wl.bits(big), 448.0)
    assert qq.tolist() == [[0x7E, 0xFE, 0x7E, 0x7E]]


def test_max_code_is_448_invariant(oracle_mod):
    dec = np.array([oracle_mod.e4m3_decode(c) for c in range(256)])
    for seed, std in [(1, 1.0), (2, 0.02), (3, 1e-10), (4, 1e30)]:
        x = wl.normal((50, 70), std, seed)
        q = oracle_mod.quantize(wl.bits(x))
        assert q["amax"] >= 1e-12
        vals = np.abs(dec[q["q"]])
        assert vals.max() == 448.0
        assert not np.isnan(vals).any()
    # below the clamp (amax < 1e-12) the scale stays at 448/1e-12 and q shrinks
    x = wl.normal((50, 70), 1e-30, 3)
    q = oracle_mod.quantize(wl.bits(x))
    assert q["amax"] < 1e-12 and q["scale"] == oracle_mod.scale(0.0)
    assert np.abs(dec[q["q"]]).max() < 448.0


def test_power_of_two_scale_invariance(oracle_mod):
    x = wl.normal((40, 64), 1.0, 12)
    q0 = oracle_mod.quantize(wl.bits(x))["q"]
    for k in (-20, -3, 1, 7, 40):
        xk = (x.to(torch.float32) * 2.0 ** k).to(torch.bfloat16)
        assert torch.equal(xk.float() / 2.0 ** k, x.float())   # exact rescale
        assert np.array_equal(oracle_mod.quantize(wl.bits(xk))["q"], q0), k


def test_all_zero_tensor(oracle_mod):
    z = torch.zeros((16, 32), dtype=torch.bfloat16)
    q = oracle_mod.quantize(wl.bits(z))
    assert q["amax"] == 0 and np.isfinite(q["scale"])
    assert (q["q"] == 0).all()
