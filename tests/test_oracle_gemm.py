"""Pins of the oracle's GEMM and of the linear's composition.

- hand-worked 2x2 (forward and backward) and 4x4 (with rounding) examples,
  with every code, scale and output bit derived by hand below;
- the int64 and fp64 sums agree exactly (both are exact);
- agreement with numpy's float64 matmul of torch-decoded E4M3 values (exact
  integers times 2^-18) rounded to bf16 by bit manipulation;
- quantisation quality: SQNR >= 25 dB against the unquantised fp64 product;
- the lossless special case: inputs already on the scaled E4M3 grid give the
  correctly rounded bf16 of the exact bf16 product;
- the sampled row / column entry points return slices of the full product;
- dX and dW use the right operands (a transposed or swapped operand fails
  the unquantised-reference check).
"""
import numpy as np
import pytest
import torch

from float8_mixed_precision_gb300 import workloads as wl


def bf16(vals):
    return torch.tensor(vals, dtype=torch.bfloat16)


def _dec(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _bf16_bits_of_f64(y):
    """RNE fp64 -> bf16 by bit manipulation; valid for zero and normal bf16 results."""
    y = np.asarray(y, np.float64)
    b = y.view(np.uint64)
    sign = (b >> np.uint64(63)).astype(np.uint32)
    exp = ((b >> np.uint64(52)) & np.uint64(0x7FF)).astype(np.int64)
    mant = b & np.uint64((1 << 52) - 1)
    keep = (mant >> np.uint64(45)).astype(np.int64)
    rem = mant & np.uint64((1 << 45) - 1)
    half = np.uint64(1 << 44)
    up = (rem > half) | ((rem == half) & ((keep & 1) == 1))
    keep = keep + up
    exp = exp + (keep >> 7)
    keep = keep & 127
    e16 = exp - 1023 + 127
    zero = (y == 0)
    assert ((e16 >= 1) & (e16 <= 254) | zero).all(), "outside the normal bf16 range"
    out = (sign << 15) | (np.where(zero, 0, e16).astype(np.uint32) << 7) | np.where(zero, 0, keep).astype(np.uint32)
    return out.astype(np.uint16)


def _bits_to_f64(b):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def test_hand_2x2_forward_backward(oracle_mod):
    x = bf16([[1.0, -2.0], [0.5, 4.0]])        # amax 4  -> s_x = 112
    w = bf16([[1.0, 1.0], [0.25, -1.0]])       # amax 1  -> s_w = 448
    dy = bf16([[1.0, 0.0], [0.0, -1.0]])       # amax 1  -> s_dy = 448
    f = oracle_mod.linear_fwd(wl.bits(x), wl.bits(w))
    assert f["x"]["scale"] == 112.0 and f["w"]["scale"] == 448.0
    # 112 = 1.75*2^6 -> 0x6E; -224 = -1.75*2^7 -> 0xF6; 56 = 1.75*2^5 -> 0x66; 448 -> 0x7E
    assert f["x"]["q"].tolist() == [[0x6E, 0xF6], [0x66, 0x7E]]
    assert f["w"]["q"].tolist() == [[0x7E, 0x7E], [0x6E, 0xFE]]
    # Y = X W^T exactly: [[-1, 2.25], [4.5, -3.875]]
    assert f["y"].tolist() == [[0xBF80, 0x4010], [0x4090, 0xC078]]
    b = oracle_mod.linear_bwd(wl.bits(dy), f)
    assert b["dy"]["scale"] == 448.0
    # dX = dY W = [[1, 1], [-0.25, 1]];  dW = dY^T X = [[1, -2], [-0.5, -4]]
    assert b["dx"].tolist() == [[0x3F80, 0x3F80], [0xBE80, 0x3F80]]
    assert b["dw"].tolist() == [[0x3F80, 0xC000], [0xBF00, 0xC080]]


def test_hand_4x4_with_rounding(oracle_mod):
    x = bf16([[1.0, 0.3, 0, 0], [0, 0, 0, 0], [-0.5, 0, 0.0078125, 0], [0, 0, 0, 0.001]])
    w = bf16([[2.0, 0, 0, 0], [0, 2.0, 0, 0], [0, 0, 2.0, 0], [1.0, 1.0, 1.0, 1.0]])
    f = oracle_mod.linear_fwd(wl.bits(x), wl.bits(w))
    assert f["x"]["scale"] == 448.0 and f["w"]["scale"] == 224.0
    # bf16(0.3) = 77/256; *448 = 134.75 -> nearest of {128, 144} is 128 = 0x70
    # 2^-7 * 448 = 3.5 = 1.75*2^1 -> 0x46
    # bf16(0.001) = 1.0234375*2^-10; *448 = 0.44775390625 -> spacing 2^-5 -> 14*2^-5 = 0.4375 -> 0x2E
    assert f["x"]["q"].tolist() == [[0x7E, 0x70, 0, 0], [0, 0, 0, 0], [0xF6, 0, 0x46, 0], [0, 0, 0, 0x2E]]
    assert f["w"]["q"].tolist() == [[0x7E, 0, 0, 0], [0, 0x7E, 0, 0], [0, 0, 0x7E, 0], [0x76, 0x76, 0x76, 0x76]]
    # Y = qX qW^T / (448*224 = 100352):
    #   row 0: 200704/100352 = 2; 57344/100352 = 4/7 -> 0x3F12; 0; 129024/100352 = 9/7 -> 0x3FA5
    #   row 2: -1; 0; 1568/100352 = 2^-6; -49392/100352 = -0.4921875
    #   row 3: 98/100352 = 2^-10 in column 3
    assert f["y"].tolist() == [[0x4000, 0x3F12, 0x0000, 0x3FA5],
                               [0, 0, 0, 0],
                               [0xBF80, 0x0000, 0x3C80, 0xBEFC],
                               [0, 0, 0, 0x3A80]]


def _quantised_pair(M, N, K, seed):
    g = torch.Generator().manual_seed(seed)
    a = torch.randint(0, 256, (M, K), generator=g, dtype=torch.uint8)
    b = torch.randint(0, 256, (N, K), generator=g, dtype=torch.uint8)
    a[(a & 0x7F) == 0x7F] = 0x3C     # no NaN codes
    b[(b & 0x7F) == 0x7F] = 0xC4
    return a.numpy(), b.numpy()


def test_int64_and_fp64_routes_agree(oracle_mod):
    a, b = _quantised_pair(37, 29, 1000, 1)
    for sa, sb in [(1.0, 1.0), (448.0, 3.7e-3), (2.5e4, 1.1e5)]:
        c0 = oracle_mod.gemm(a, b, sa, sb, route=0)
        c1 = oracle_mod.gemm(a, b, sa, sb, route=1)
        assert np.array_equal(c0, c1)


def test_matches_numpy_matmul(oracle_mod):
    a, b = _quantised_pair(40, 24, 512, 2)
    sa, sb = np.float32(3.25), np.float32(0.0625)
    ref = (_dec(a) @ _dec(b).T) / (np.float64(sa) * np.float64(sb))
    assert np.array_equal(oracle_mod.gemm(a, b, sa, sb), _bf16_bits_of_f64(ref))


def _sqnr_db(ref, got):
    return 10 * np.log10((ref ** 2).sum() / ((got - ref) ** 2).sum())


def test_sqnr_against_unquantised(oracle_mod):
    d = wl.custom_linear(96, 256, 80, seed=21)
    f = oracle_mod.linear_fwd(wl.bits(d["x"]), wl.bits(d["w"]))
    b = oracle_mod.linear_bwd(wl.bits(d["dy"]), f)
    x, w, dy = (d[k].to(torch.float64).numpy() for k in ("x", "w", "dy"))
    for ref, got in [(x @ w.T, f["y"]), (dy @ w, b["dx"]), (dy.T @ x, b["dw"])]:
        s = _sqnr_db(ref, _bits_to_f64(got))
        assert s >= 25.0, s
        assert s < 40.0    # it is a quantised result, not the exact product


def test_lossless_special_case(oracle_mod):
    # values on the E4M3 grid times 2^-3 with amax = 56 give s = 8 exactly:
    # x * s lands on the grid and quantisation is lossless
    g = torch.Generator().manual_seed(4)
    grid = _dec(np.arange(0x7F, dtype=np.uint8))
    xs = grid[torch.randint(0, 0x7F, (24, 64), generator=g).numpy()] * np.where(
        torch.rand(24, 64, generator=g).numpy() < 0.5, -1, 1)
    xs[0, 0] = 448.0
    ws = grid[torch.randint(0, 0x7F, (16, 64), generator=g).numpy()]
    ws[3, 5] = -448.0
    x = torch.from_numpy(xs / 8).to(torch.bfloat16)
    w = torch.from_numpy(ws / 2).to(torch.bfloat16)
    assert torch.equal(x.double(), torch.from_numpy(xs / 8))
    f = oracle_mod.linear_fwd(wl.bits(x), wl.bits(w))
    assert f["x"]["scale"] == 8.0 and f["w"]["scale"] == 2.0
    exact = x.double().numpy() @ w.double().numpy().T
    assert np.array_equal(f["y"], _bf16_bits_of_f64(exact))


def test_sampled_rows_and_cols(oracle_mod):
    a, b = _quantised_pair(50, 70, 96, 3)
    full = oracle_mod.gemm(a, b, 5.0, 7.0)
    rows = [0, 13, 49]
    cols = [1, 2, 69]
    assert np.array_equal(oracle_mod.gemm_rows(a, b, 5.0, 7.0, rows), full[rows])
    assert np.array_equal(oracle_mod.gemm_cols(a, b, 5.0, 7.0, cols), full[:, cols].T)


def test_backward_operands(oracle_mod):
    d = wl.custom_linear(48, 32, 64, seed=31)
    f = oracle_mod.linear_fwd(wl.bits(d["x"]), wl.bits(d["w"]))
    b = oracle_mod.linear_bwd(wl.bits(d["dy"]), f)
    assert b["dx"].shape == (48, 32) and b["dw"].shape == (64, 32)
    qx, qw, qdy = _dec(f["x"]["q"]), _dec(f["w"]["q"]), _dec(b["dy"]["q"])
    sx, sw, sdy = (np.float64(v) for v in (f["x"]["scale"], f["w"]["scale"], b["dy"]["scale"]))
    assert np.array_equal(b["dx"], _bf16_bits_of_f64(qdy @ qw / (sdy * sw)))
    assert np.array_equal(b["dw"], _bf16_bits_of_f64(qdy.T @ qx / (sdy * sx)))


def test_empty_and_zero_k(oracle_mod):
    a = np.zeros((3, 0), np.uint8)
    b = np.zeros((5, 0), np.uint8)
    assert (oracle_mod.gemm(a, b, 1.0, 1.0) == 0).all()
    assert oracle_mod.gemm(np.zeros((0, 16), np.uint8), np.zeros((4, 16), np.uint8), 1.0, 1.0).shape == (0, 4)
