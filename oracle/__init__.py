"""CPU oracle for the Float8 training linear (dynamic tensorwise scaling).

TEST INFRASTRUCTURE ONLY.  Only the test-suite, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import this package.  It shares
no code with the CUDA library and never imports it.

The arithmetic lives in ``f8_oracle.c`` (plain C, fp64 / int64, built with
``-ffp-contract=off``); this module builds it with gcc on first use and wraps
it with ctypes.  The linear composition below chains the C steps in the order
of the method:

  forward   amax(X), amax(W) -> s_x, s_w -> q(X), q(W) -> Y = q(X) q(W)^T / (s_x s_w)
  backward  amax(dY) -> s_dy -> q(dY) -> dX = q(dY) q(W) / (s_dy s_w)
                                        dW = q(dY)^T q(X) / (s_dy s_x)

Sources: "TorchTitan" paper summary (atlas.scime.ai), Approach and ablation
table (Float8 as a composable transformation of the Llama 3.1 8B linears);
wassimseifeddine.com/posts/torchtitan, "Float8 Training" (torchao Float8);
stanleyjacob.dev/oss/torchtitan, Part XI item 9 (the E4M3 / E5M2 formats).
The pages do not print the scaling recipe; the reading taken here (one fp32
scale 448/amax per tensor, recomputed every call) is the plainest one.

Every function takes and returns numpy arrays; bf16 tensors travel as their
uint16 bit patterns, E4M3 tensors as uint8 codes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "f8_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``f8_oracle.c`` into ``_build/liboracle.so`` (gcc, OpenMP if present)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        u8p = ctypes.POINTER(ctypes.c_uint8)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        i64p = ctypes.POINTER(ctypes.c_int64)
        i64 = ctypes.c_int64
        f32 = ctypes.c_float
        lib.or_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.or_bf16_to_f32.restype = f32
        lib.or_f64_to_bf16.argtypes = [ctypes.c_double]
        lib.or_f64_to_bf16.restype = ctypes.c_uint16
        lib.or_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.or_e4m3_decode.restype = ctypes.c_double
        lib.or_e4m3_encode.argtypes = [f32]
        lib.or_e4m3_encode.restype = ctypes.c_uint8
        lib.or_amax.argtypes = [u16p, i64, ctypes.POINTER(ctypes.c_int)]
        lib.or_amax.restype = f32
        lib.or_scale.argtypes = [f32]
        lib.or_scale.restype = f32
        lib.or_cast_transpose.argtypes = [u16p, i64, i64, f32, u8p, u8p]
        lib.or_cast_transpose.restype = None
        lib.or_gemm.argtypes = [u8p, u8p, i64, i64, i64, f32, f32, u16p, ctypes.c_int]
        lib.or_gemm.restype = None
        lib.or_gemm_rows.argtypes = [u8p, u8p, i64, i64, i64, f32, f32, i64p, i64, u16p]
        lib.or_gemm_rows.restype = None
        lib.or_gemm_cols.argtypes = [u8p, u8p, i64, i64, i64, f32, f32, i64p, i64, u16p]
        lib.or_gemm_cols.restype = None
        lib.or_e5m2_decode.argtypes = [ctypes.c_uint8]
        lib.or_e5m2_decode.restype = ctypes.c_double
        lib.or_e5m2_encode.argtypes = [f32]
        lib.or_e5m2_encode.restype = ctypes.c_uint8
        lib.or_scale_fmt.argtypes = [f32, ctypes.c_int]
        lib.or_scale_fmt.restype = f32
        lib.or_cast_transpose_fmt.argtypes = [u16p, i64, i64, f32, ctypes.c_int, u8p, u8p]
        lib.or_cast_transpose_fmt.restype = None
        lib.or_gemm_rows_fmt.argtypes = [u8p, ctypes.c_int, u8p, ctypes.c_int, i64, i64, i64, f32, f32,
                                         i64p, i64, u16p]
        lib.or_gemm_rows_fmt.restype = None
        lib.or_silu.argtypes = [ctypes.c_double]
        lib.or_silu.restype = ctypes.c_double
        lib.or_swiglu_h.argtypes = [u16p, u16p, i64, u16p]
        lib.or_swiglu_h.restype = None
        lib.or_swiglu_bwd.argtypes = [u16p, u16p, u16p, i64, u16p, u16p]
        lib.or_swiglu_bwd.restype = None
        lib.or_num_threads.argtypes = []
        lib.or_num_threads.restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(arr: np.ndarray, ctype):
    if arr is None:
        return None
    assert arr.flags["C_CONTIGUOUS"]
    return arr.ctypes.data_as(ctypes.POINTER(ctype))


def _u16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x)
    assert x.dtype == np.uint16, "bf16 tensors are passed as uint16 bit patterns"
    return x


def _u8(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x)
    assert x.dtype == np.uint8, "E4M3 tensors are passed as uint8 codes"
    return x


# --------------------------------------------------------------------------
# scalar codecs
# --------------------------------------------------------------------------

def bf16_to_f32(bits: int) -> float:
    return float(_load().or_bf16_to_f32(int(bits)))


def f64_to_bf16(y: float) -> int:
    return int(_load().or_f64_to_bf16(float(y)))


def e4m3_decode(code: int) -> float:
    return float(_load().or_e4m3_decode(int(code)))


def e4m3_encode(v: float) -> int:
    """v is taken as an fp32 value (the cast's operand is an fp32 product)."""
    return int(_load().or_e4m3_encode(float(np.float32(v))))


E4M3, E5M2 = 0, 1
FMT_MAX = {E4M3: 448.0, E5M2: 57344.0}


def e5m2_decode(code: int) -> float:
    return float(_load().or_e5m2_decode(int(code)))


def e5m2_encode(v: float) -> int:
    """v is taken as an fp32 value."""
    return int(_load().or_e5m2_encode(float(np.float32(v))))


def num_threads() -> int:
    return int(_load().or_num_threads())


# --------------------------------------------------------------------------
# tensor steps
# --------------------------------------------------------------------------

def amax(x_bits: np.ndarray) -> tuple[np.float32, bool]:
    """max |x| over a bf16 tensor (fp32) and whether any entry was non-finite."""
    x = _u16(x_bits).reshape(-1)
    nf = ctypes.c_int(0)
    a = _load().or_amax(_ptr(x, ctypes.c_uint16), x.size, ctypes.byref(nf))
    return np.float32(a), bool(nf.value)


def scale(a: float) -> np.float32:
    return np.float32(_load().or_scale(float(np.float32(a))))


def cast_transpose(x_bits: np.ndarray, s: float) -> tuple[np.ndarray, np.ndarray]:
    """(q [rows, cols], q^T [cols, rows]) of a 2-D bf16 tensor under scale s."""
    x = _u16(x_bits)
    rows, cols = x.shape
    q = np.empty((rows, cols), np.uint8)
    qt = np.empty((cols, rows), np.uint8)
    _load().or_cast_transpose(_ptr(x, ctypes.c_uint16), rows, cols, float(np.float32(s)),
                              _ptr(q, ctypes.c_uint8), _ptr(qt, ctypes.c_uint8))
    return q, qt


def scale_fmt(a: float, fmt: int) -> np.float32:
    return np.float32(_load().or_scale_fmt(float(np.float32(a)), int(fmt)))


def cast_transpose_fmt(x_bits: np.ndarray, s: float, fmt: int) -> tuple[np.ndarray, np.ndarray]:
    x = _u16(x_bits)
    rows, cols = x.shape
    q = np.empty((rows, cols), np.uint8)
    qt = np.empty((cols, rows), np.uint8)
    _load().or_cast_transpose_fmt(_ptr(x, ctypes.c_uint16), rows, cols, float(np.float32(s)),
                                  int(fmt), _ptr(q, ctypes.c_uint8), _ptr(qt, ctypes.c_uint8))
    return q, qt


def gemm_rows_fmt(a_q, fa: int, b_q, fb: int, sa, sb, rows=None) -> np.ndarray:
    """Rows of C = bf16(A B^T / (sa sb)) with A codes in format fa and B in fb
    (exact __int128 sums); all rows if ``rows`` is None."""
    a = _u8(a_q)
    b = _u8(b_q)
    M, K = a.shape
    N = b.shape[0]
    r = np.arange(M, dtype=np.int64) if rows is None else np.ascontiguousarray(np.asarray(rows, np.int64))
    out = np.empty((r.size, N), np.uint16)
    _load().or_gemm_rows_fmt(_ptr(a, ctypes.c_uint8), int(fa), _ptr(b, ctypes.c_uint8), int(fb), M, N,
                             K, float(np.float32(sa)), float(np.float32(sb)), _ptr(r, ctypes.c_int64),
                             r.size, _ptr(out, ctypes.c_uint16))
    return out


def gemm(a_q: np.ndarray, b_q: np.ndarray, sa: float, sb: float, route: int = 0) -> np.ndarray:
    """C = bf16(A B^T / (sa sb)); A [M,K], B [N,K] E4M3 codes; returns uint16 [M,N]."""
    a = _u8(a_q)
    b = _u8(b_q)
    M, K = a.shape
    N, K2 = b.shape
    assert K == K2
    c = np.empty((M, N), np.uint16)
    _load().or_gemm(_ptr(a, ctypes.c_uint8), _ptr(b, ctypes.c_uint8), M, N, K,
                    float(np.float32(sa)), float(np.float32(sb)), _ptr(c, ctypes.c_uint16),
                    int(route))
    return c


def gemm_rows(a_q, b_q, sa, sb, rows) -> np.ndarray:
    """Rows ``rows`` of gemm(a_q, b_q, sa, sb): uint16 [len(rows), N]."""
    a = _u8(a_q)
    b = _u8(b_q)
    M, K = a.shape
    N = b.shape[0]
    r = np.ascontiguousarray(np.asarray(rows, np.int64))
    assert r.size == 0 or (r.min() >= 0 and r.max() < M)
    out = np.empty((r.size, N), np.uint16)
    _load().or_gemm_rows(_ptr(a, ctypes.c_uint8), _ptr(b, ctypes.c_uint8), M, N, K,
                         float(np.float32(sa)), float(np.float32(sb)),
                         _ptr(r, ctypes.c_int64), r.size, _ptr(out, ctypes.c_uint16))
    return out


def gemm_cols(a_q, b_q, sa, sb, cols) -> np.ndarray:
    """Columns ``cols`` of gemm(a_q, b_q, sa, sb), transposed: uint16 [len(cols), M]."""
    a = _u8(a_q)
    b = _u8(b_q)
    M, K = a.shape
    N = b.shape[0]
    cidx = np.ascontiguousarray(np.asarray(cols, np.int64))
    assert cidx.size == 0 or (cidx.min() >= 0 and cidx.max() < N)
    out = np.empty((cidx.size, M), np.uint16)
    _load().or_gemm_cols(_ptr(a, ctypes.c_uint8), _ptr(b, ctypes.c_uint8), M, N, K,
                         float(np.float32(sa)), float(np.float32(sb)),
                         _ptr(cidx, ctypes.c_int64), cidx.size, _ptr(out, ctypes.c_uint16))
    return out


def silu(x: float) -> float:
    """silu(x) = x / (1 + exp(-x)) in fp64."""
    return float(_load().or_silu(float(x)))


def swiglu_h(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """bf16 bits of h = bf16(silu(a) * b): the product formed in fp64 from the
    bf16 inputs and rounded once to bf16."""
    a = _u16(a_bits)
    b = _u16(b_bits)
    assert a.shape == b.shape
    h = np.empty(a.shape, np.uint16)
    _load().or_swiglu_h(_ptr(a, ctypes.c_uint16), _ptr(b, ctypes.c_uint16), a.size,
                        _ptr(h, ctypes.c_uint16))
    return h


def swiglu_bwd(dh_bits: np.ndarray, a_bits: np.ndarray, b_bits: np.ndarray):
    """bf16 bits of (da, db), the gradient of h = silu(a) * b for an upstream
    dh: db = bf16(dh * silu(a)), da = bf16(dh * b * silu'(a)) with
    silu'(a) = sigma (1 + a (1 - sigma)), each formed in fp64 and rounded
    once to bf16."""
    dh, a, b = _u16(dh_bits), _u16(a_bits), _u16(b_bits)
    assert dh.shape == a.shape == b.shape
    da = np.empty(a.shape, np.uint16)
    db = np.empty(a.shape, np.uint16)
    _load().or_swiglu_bwd(_ptr(dh, ctypes.c_uint16), _ptr(a, ctypes.c_uint16),
                          _ptr(b, ctypes.c_uint16), a.size, _ptr(da, ctypes.c_uint16),
                          _ptr(db, ctypes.c_uint16))
    return da, db


# --------------------------------------------------------------------------
# the linear layer, step by step
# --------------------------------------------------------------------------

def quantize(x_bits: np.ndarray, fmt: int = E4M3) -> dict:
    """amax -> scale -> (q, q^T) for one bf16 tensor in format fmt."""
    a, nonfinite = amax(x_bits)
    if fmt == E4M3:
        s = scale(a)
        q, qt = cast_transpose(x_bits, s)
    else:
        s = scale_fmt(a, fmt)
        q, qt = cast_transpose_fmt(x_bits, s, fmt)
    return {"amax": a, "scale": s, "q": q, "qt": qt, "nonfinite": nonfinite, "fmt": fmt}


def linear_fwd(x_bits: np.ndarray, w_bits: np.ndarray) -> dict:
    """Y = X W^T for X [M,K], W [N,K] (bf16 bits); returns Y bits and every intermediate."""
    qx = quantize(x_bits)
    qw = quantize(w_bits)
    y = gemm(qx["q"], qw["q"], qx["scale"], qw["scale"])
    return {"x": qx, "w": qw, "y": y}


def linear_fwd_swiglu(a_bits: np.ndarray, b_bits: np.ndarray, w_bits: np.ndarray) -> dict:
    """The forward of a linear whose input is h = silu(a) * b: h is formed
    elementwise, then quantised and multiplied exactly as linear_fwd does."""
    h = swiglu_h(a_bits, b_bits)
    out = linear_fwd(h, w_bits)
    out["h"] = h
    return out


def split_ab(ab_bits: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """a, b [M, F] of the group {w1, w3}'s output AB [M, 2F] when W13 takes
    its rows from W1 and W3 alternately in blocks of 128: column c of a is
    column 256 (c // 128) + c % 128 of AB, column c of b the one 128 to its
    right."""
    ab = _u16(ab_bits)
    M, N = ab.shape
    v = ab.reshape(M, N // 256, 2, 128)
    return (np.ascontiguousarray(v[:, :, 0, :].reshape(M, N // 2)),
            np.ascontiguousarray(v[:, :, 1, :].reshape(M, N // 2)))


def linear_fwd_w13_swiglu(x_bits: np.ndarray, w13_bits: np.ndarray) -> dict:
    """The input side of a SwiGLU FFN: AB = linear_fwd(X, W13) (one Float8
    linear for the group {w1, w3}, one scale over W13), then h = bf16(silu(a)
    * b) from AB's bf16 a and b, then h quantised for the w2 linear."""
    out = linear_fwd(x_bits, w13_bits)
    a, b = split_ab(out["y"])
    out["h"] = swiglu_h(a, b)
    out["qh"] = quantize(out["h"])
    return out


def merge_ab(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """The inverse of split_ab: a and b [M, F] into one [M, 2F] whose column
    blocks of 128 come from a and b alternately."""
    a, b = _u16(a_bits), _u16(b_bits)
    M, F = a.shape
    out = np.empty((M, F // 128, 2, 128), np.uint16)
    out[:, :, 0, :] = a.reshape(M, F // 128, 128)
    out[:, :, 1, :] = b.reshape(M, F // 128, 128)
    return out.reshape(M, 2 * F)


def linear_bwd_w13_swiglu(dh_bits: np.ndarray, fwd: dict) -> dict:
    """The backward of linear_fwd_w13_swiglu for the gradient dh of h: the
    SwiGLU gradient (da, db) from dh and the forward's bf16 a and b, merged
    into d(AB) in AB's column order, then linear_bwd of the group."""
    a, b = split_ab(fwd["y"])
    da, db = swiglu_bwd(dh_bits, a, b)
    dab = merge_ab(da, db)
    out = linear_bwd(dab, fwd)
    out["dab"] = dab
    return out


def linear_bwd(dy_bits: np.ndarray, fwd: dict, dy_fmt: int = E4M3) -> dict:
    """dX = dY W, dW = dY^T X using the forward's quantised X and W; dY is
    quantised in format dy_fmt (E4M3 or E5M2)."""
    qdy = quantize(dy_bits, dy_fmt)
    qx, qw = fwd["x"], fwd["w"]
    if dy_fmt != E4M3:
        dx = gemm_rows_fmt(qdy["q"], dy_fmt, qw["qt"], E4M3, qdy["scale"], qw["scale"])
        dw = gemm_rows_fmt(qdy["qt"], dy_fmt, qx["qt"], E4M3, qdy["scale"], qx["scale"])
        return {"dy": qdy, "dx": dx, "dw": dw}
    # dX[m,k] = sum_n dY[m,n] W[n,k]: A = q(dY) [M,N], B = q(W)^T [K,N]
    dx = gemm(qdy["q"], qw["qt"], qdy["scale"], qw["scale"])
    # dW[n,k] = sum_m dY[m,n] X[m,k]: A = q(dY)^T [N,M], B = q(X)^T [K,M]
    dw = gemm(qdy["qt"], qx["qt"], qdy["scale"], qx["scale"])
    return {"dy": qdy, "dx": dx, "dw": dw}
