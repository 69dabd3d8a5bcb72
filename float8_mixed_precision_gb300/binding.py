"""Python binding of libf8's C ABI (include/f8.h): argument marshalling only.

Every function here has the name of the C entry point it calls.  torch is
used to allocate device memory for outputs the caller did not pass and to
find the current CUDA stream; all arithmetic runs in libf8's kernels.  There
is no fallback: if ``_lib/libf8.so`` is missing the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# F8_LIBRARY selects another build of the same library (the checked build,
# _lib/libf8_checked.so); it must exist like the default one.
LIB_PATH = os.environ.get("F8_LIBRARY") or os.path.join(_HERE, "_lib", "libf8.so")

F8_OK = 0
F8_ERR_INVALID = 1
F8_ERR_ALIGN = 2
F8_ERR_SHAPE = 3
F8_ERR_CUDA = 4
F8_ERR_TIMEOUT = 5
F8_ERR_NONFINITE = 6
F8_ERR_UNSUPPORTED = 7
F8_ERR_BOUNDS = 8

# every symbol include/f8.h declares
EXPORTS = ("f8_amax", "f8_cast_transpose", "f8_gemm", "f8_linear_workspace_bytes",
           "f8_linear_fwd", "f8_linear_bwd", "f8_last_device_status", "f8_status_string",
           "f8_selftest_wait_timeout", "f8_set_wait_limit_ns", "f8_linear_fwd_noalloc",
           "f8_quantize", "f8_quantize_workspace_bytes", "f8_quantize_fmt", "f8_gemm_fmt",
           "f8_linear_bwd_fmt", "f8_quantize_swiglu", "f8_linear_fwd_swiglu",
           "f8_linear_fwd_w13_swiglu", "f8_gemm_w13_swiglu", "f8_linear_bwd_w13_swiglu",
           "f8_quantize_swiglu_bwd", "f8_kernel_launches", "f8_selftest_bounds",
           "f8_gemm_grouped", "f8_quantize_multi", "f8_quantize_multi_workspace_bytes",
           "f8_linear_group_workspace_bytes", "f8_linear_fwd_group", "f8_linear_bwd_group",
           "f8_transpose_u8", "f8_linear_fwd_qw", "f8_linear_fwd_qw_workspace_bytes")

F8_MAX_GROUPED_GEMMS = 8
F8_MAX_MULTI_TENSORS = 8
F8_MAX_GROUP_LINEARS = 4

F8_E4M3 = 0
F8_E5M2 = 1


class F8Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {f8_status_string(status)}")


class _Saved(ctypes.Structure):
    _fields_ = [("x_t", ctypes.c_void_p), ("w_t", ctypes.c_void_p),
                ("amax_x", ctypes.c_void_p), ("scale_x", ctypes.c_void_p),
                ("amax_w", ctypes.c_void_p), ("scale_w", ctypes.c_void_p)]


class _GemmProblem(ctypes.Structure):
    _fields_ = [("a", ctypes.c_void_p), ("b", ctypes.c_void_p), ("M", ctypes.c_int64),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("scale_a", ctypes.c_void_p),
                ("scale_b", ctypes.c_void_p), ("c", ctypes.c_void_p), ("fmt_a", ctypes.c_int),
                ("fmt_b", ctypes.c_int)]


class _QuantTensor(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("amax_out", ctypes.c_void_p), ("scale_out", ctypes.c_void_p),
                ("q", ctypes.c_void_p), ("q_t", ctypes.c_void_p)]


class _GroupLinear(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int64), ("w", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("dy", ctypes.c_void_p), ("dx", ctypes.c_void_p), ("dw", ctypes.c_void_p),
                ("saved", _Saved)]


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libf8 (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libf8 is not built ({LIB_PATH} missing): run "
                "`python -m float8_mixed_precision_gb300.build` (needs nvcc)")
        L = ctypes.CDLL(LIB_PATH)
        vp, i64, u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64
        st = ctypes.c_int
        L.f8_amax.argtypes = [vp, i64, vp, vp]
        L.f8_amax.restype = st
        L.f8_cast_transpose.argtypes = [vp, i64, i64, vp, vp, vp, vp, vp]
        L.f8_cast_transpose.restype = st
        L.f8_gemm.argtypes = [vp, vp, i64, i64, i64, vp, vp, vp, vp]
        L.f8_gemm.restype = st
        L.f8_linear_workspace_bytes.argtypes = [i64, i64, i64]
        L.f8_linear_workspace_bytes.restype = ctypes.c_size_t
        L.f8_linear_fwd.argtypes = [vp, vp, i64, i64, i64, vp, ctypes.POINTER(_Saved), vp,
                                    ctypes.c_size_t, vp]
        L.f8_linear_fwd.restype = st
        L.f8_linear_bwd.argtypes = [vp, ctypes.POINTER(_Saved), i64, i64, i64, vp, vp, vp,
                                    ctypes.c_size_t, vp]
        L.f8_linear_bwd.restype = st
        L.f8_last_device_status.argtypes = [vp]
        L.f8_last_device_status.restype = st
        L.f8_status_string.argtypes = [st]
        L.f8_status_string.restype = ctypes.c_char_p
        L.f8_selftest_wait_timeout.argtypes = [u64, vp]
        L.f8_selftest_wait_timeout.restype = st
        L.f8_set_wait_limit_ns.argtypes = [u64]
        L.f8_set_wait_limit_ns.restype = None
        L.f8_quantize_workspace_bytes.argtypes = []
        L.f8_quantize_workspace_bytes.restype = ctypes.c_size_t
        L.f8_quantize.argtypes = [vp, i64, i64, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
        L.f8_quantize.restype = st
        L.f8_quantize_fmt.argtypes = [vp, i64, i64, ctypes.c_int, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
        L.f8_quantize_fmt.restype = st
        L.f8_gemm_fmt.argtypes = [vp, ctypes.c_int, vp, ctypes.c_int, i64, i64, i64, vp, vp, vp, vp]
        L.f8_gemm_fmt.restype = st
        L.f8_linear_bwd_fmt.argtypes = [vp, ctypes.c_int, ctypes.POINTER(_Saved), i64, i64, i64, vp, vp,
                                        vp, ctypes.c_size_t, vp]
        L.f8_linear_bwd_fmt.restype = st
        L.f8_quantize_swiglu.argtypes = [vp, vp, vp, i64, i64, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
        L.f8_quantize_swiglu.restype = st
        L.f8_linear_fwd_swiglu.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp, ctypes.POINTER(_Saved),
                                           vp, ctypes.c_size_t, vp]
        L.f8_linear_fwd_swiglu.restype = st
        L.f8_linear_fwd_w13_swiglu.argtypes = [vp, vp, i64, i64, i64, vp, vp, ctypes.POINTER(_Saved),
                                               vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
        L.f8_linear_fwd_w13_swiglu.restype = st
        L.f8_linear_bwd_w13_swiglu.argtypes = [vp, vp, ctypes.POINTER(_Saved), i64, i64, i64, vp,
                                               ctypes.c_int, vp, vp, vp, ctypes.c_size_t, vp]
        L.f8_linear_bwd_w13_swiglu.restype = st
        L.f8_quantize_swiglu_bwd.argtypes = [vp, vp, i64, i64, vp, ctypes.c_int, vp, vp, vp, vp, vp,
                                             ctypes.c_size_t, vp]
        L.f8_quantize_swiglu_bwd.restype = st
        L.f8_selftest_bounds.argtypes = [vp]
        L.f8_selftest_bounds.restype = st
        L.f8_kernel_launches.argtypes = []
        L.f8_kernel_launches.restype = ctypes.c_ulonglong
        L.f8_gemm_w13_swiglu.argtypes = [vp, vp, i64, i64, i64, vp, vp, vp, vp, vp, vp]
        L.f8_gemm_w13_swiglu.restype = st
        L.f8_linear_fwd_noalloc.argtypes = [vp, vp, i64, i64, i64, vp, ctypes.POINTER(_Saved), vp]
        L.f8_linear_fwd_noalloc.restype = st
        L.f8_gemm_grouped.argtypes = [ctypes.POINTER(_GemmProblem), ctypes.c_int, vp]
        L.f8_gemm_grouped.restype = st
        L.f8_quantize_multi_workspace_bytes.argtypes = []
        L.f8_quantize_multi_workspace_bytes.restype = ctypes.c_size_t
        L.f8_quantize_multi.argtypes = [ctypes.POINTER(_QuantTensor), ctypes.c_int, ctypes.c_int, vp,
                                        ctypes.c_size_t, vp]
        L.f8_quantize_multi.restype = st
        L.f8_linear_group_workspace_bytes.argtypes = [i64, i64, ctypes.POINTER(i64), ctypes.c_int]
        L.f8_linear_group_workspace_bytes.restype = ctypes.c_size_t
        L.f8_linear_fwd_group.argtypes = [vp, i64, i64, ctypes.POINTER(_GroupLinear), ctypes.c_int, vp,
                                          ctypes.c_size_t, vp]
        L.f8_linear_fwd_group.restype = st
        L.f8_linear_bwd_group.argtypes = [ctypes.POINTER(_GroupLinear), ctypes.c_int, i64, i64,
                                          ctypes.c_int, vp, ctypes.c_size_t, vp]
        L.f8_linear_bwd_group.restype = st
        L.f8_transpose_u8.argtypes = [vp, i64, i64, vp, vp]
        L.f8_transpose_u8.restype = st
        L.f8_linear_fwd_qw_workspace_bytes.argtypes = [i64, i64]
        L.f8_linear_fwd_qw_workspace_bytes.restype = ctypes.c_size_t
        L.f8_linear_fwd_qw.argtypes = [vp, vp, i64, i64, i64, vp, ctypes.POINTER(_Saved), vp,
                                       ctypes.c_size_t, vp]
        L.f8_linear_fwd_qw.restype = st
        _lib = L
        return L


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _need(what: str, dtype, *ts) -> None:
    """TypeError unless every given tensor is 2-D of `dtype`: the C calls
    read the bytes as that type and take the shape from the tensor."""
    for t in ts:
        if t is not None and (t.dtype != dtype or t.dim() != 2):
            raise TypeError(f"{what} takes 2-D {str(dtype).replace('torch.', '')} tensors")


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libf8 takes device tensors only")
    if not t.is_contiguous():
        raise ValueError("libf8 takes contiguous (row-major) tensors only")
    return t.data_ptr()


def _check(status: int, where: str):
    if status != F8_OK:
        raise F8Error(status, where)


def f8_selftest_bounds(stream=None) -> int:
    """F8_OK in the checked build (the next status read is F8_ERR_BOUNDS),
    F8_ERR_UNSUPPORTED in a release build; returns the status, never raises."""
    return int(lib().f8_selftest_bounds(_stream(stream)))


def f8_kernel_launches() -> int:
    """Kernels libf8 has launched in this process so far."""
    return int(lib().f8_kernel_launches())


def f8_status_string(status: int) -> str:
    return lib().f8_status_string(int(status)).decode()


def f8_last_device_status(stream=None) -> int:
    """Synchronise the stream and read (and clear) the device status word."""
    return int(lib().f8_last_device_status(_stream(stream)))


def f8_set_wait_limit_ns(limit_ns: int) -> None:
    lib().f8_set_wait_limit_ns(int(limit_ns))


def f8_selftest_wait_timeout(limit_ns: int, stream=None) -> None:
    _check(lib().f8_selftest_wait_timeout(int(limit_ns), _stream(stream)), "f8_selftest_wait_timeout")


def f8_amax(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """max |x| of a bf16 tensor as a device fp32 scalar tensor."""
    if x.dtype != torch.bfloat16:
        raise TypeError("f8_amax takes a bf16 tensor")
    if out is None:
        out = torch.empty((), dtype=torch.float32, device=x.device)
    _check(lib().f8_amax(_ptr(x), x.numel(), _ptr(out), _stream(stream)), "f8_amax")
    return out


def f8_cast_transpose(x: torch.Tensor, amax: torch.Tensor, scale_out: torch.Tensor | None = None,
                      q: torch.Tensor | None = None, q_t: torch.Tensor | None = None,
                      want_q: bool = True, want_t: bool = True, stream=None):
    """(q [rows, cols] uint8, q_t [cols, rows] uint8, scale fp32 scalar) of a 2-D bf16 tensor."""
    if x.dtype != torch.bfloat16 or x.dim() != 2:
        raise TypeError("f8_cast_transpose takes a 2-D bf16 tensor")
    rows, cols = x.shape
    dev = x.device
    if scale_out is None:
        scale_out = torch.empty((), dtype=torch.float32, device=dev)
    if q is None and want_q:
        q = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
    if q_t is None and want_t:
        q_t = torch.empty((cols, rows), dtype=torch.uint8, device=dev)
    _check(lib().f8_cast_transpose(_ptr(x), rows, cols, _ptr(amax), _ptr(scale_out), _ptr(q),
                                   _ptr(q_t), _stream(stream)), "f8_cast_transpose")
    return q, q_t, scale_out


def f8_quantize_workspace_bytes() -> int:
    return int(lib().f8_quantize_workspace_bytes())


def f8_quantize(x: torch.Tensor, amax_out: torch.Tensor | None = None,
                scale_out: torch.Tensor | None = None, q: torch.Tensor | None = None,
                q_t: torch.Tensor | None = None, ws: torch.Tensor | None = None,
                want_q: bool = True, want_t: bool = True, fmt: int = F8_E4M3, stream=None):
    """amax, scale and both FP8 layouts of a 2-D bf16 tensor (the linear's
    own two-launch quantisation): returns (q, q_t, scale, amax).  ``fmt``
    picks E4M3 (f8_quantize) or E5M2 (f8_quantize_fmt)."""
    if x.dtype != torch.bfloat16 or x.dim() != 2:
        raise TypeError("f8_quantize takes a 2-D bf16 tensor")
    rows, cols = x.shape
    dev = x.device
    if amax_out is None:
        amax_out = torch.empty((), dtype=torch.float32, device=dev)
    if scale_out is None:
        scale_out = torch.empty((), dtype=torch.float32, device=dev)
    if q is None and want_q:
        q = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
    if q_t is None and want_t:
        q_t = torch.empty((cols, rows), dtype=torch.uint8, device=dev)
    if ws is None:
        ws = torch.empty(f8_quantize_workspace_bytes(), dtype=torch.uint8, device=dev)
    if fmt == F8_E4M3:
        _check(lib().f8_quantize(_ptr(x), rows, cols, _ptr(amax_out), _ptr(scale_out), _ptr(q),
                                 _ptr(q_t), _ptr(ws), ws.numel(), _stream(stream)), "f8_quantize")
    else:
        _check(lib().f8_quantize_fmt(_ptr(x), rows, cols, int(fmt), _ptr(amax_out), _ptr(scale_out),
                                     _ptr(q), _ptr(q_t), _ptr(ws), ws.numel(), _stream(stream)),
               "f8_quantize_fmt")
    return q, q_t, scale_out, amax_out


def f8_gemm(a: torch.Tensor, b: torch.Tensor, scale_a: torch.Tensor, scale_b: torch.Tensor,
            out: torch.Tensor | None = None, fmt_a: int = F8_E4M3, fmt_b: int = F8_E4M3,
            stream=None) -> torch.Tensor:
    """bf16(a b^T / (scale_a scale_b)) for FP8 codes a [M,K], b [N,K] (uint8);
    formats other than E4M3 go through f8_gemm_fmt."""
    _need("f8_gemm", torch.uint8, a, b)
    M, K = a.shape
    N, K2 = b.shape
    if K != K2:
        raise ValueError("contraction sizes differ")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    if fmt_a == F8_E4M3 and fmt_b == F8_E4M3:
        _check(lib().f8_gemm(_ptr(a), _ptr(b), M, N, K, _ptr(scale_a), _ptr(scale_b), _ptr(out),
                             _stream(stream)), "f8_gemm")
    else:
        _check(lib().f8_gemm_fmt(_ptr(a), int(fmt_a), _ptr(b), int(fmt_b), M, N, K, _ptr(scale_a),
                                 _ptr(scale_b), _ptr(out), _stream(stream)), "f8_gemm_fmt")
    return out


def f8_gemm_grouped(problems, stream=None) -> list:
    """Up to F8_MAX_GROUPED_GEMMS GEMMs under the grouped-launch planner
    (f8_gemm_grouped).  Each problem is
    (a, b, scale_a, scale_b, out, fmt_a, fmt_b) as for f8_gemm (out, fmt_a
    and fmt_b may be None / omitted); returns the outputs."""
    for p in problems:
        _need("f8_gemm_grouped", torch.uint8, p[0], p[1])
    arr = (_GemmProblem * len(problems))()
    outs = []
    for i, p in enumerate(problems):
        a, b, sa, sb = p[:4]
        out = p[4] if len(p) > 4 else None
        fa = p[5] if len(p) > 5 else F8_E4M3
        fb = p[6] if len(p) > 6 else F8_E4M3
        M, K = a.shape
        N, K2 = b.shape
        if K != K2:
            raise ValueError("contraction sizes differ")
        if out is None:
            out = torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
        arr[i] = _GemmProblem(_ptr(a), _ptr(b), M, N, K, _ptr(sa), _ptr(sb), _ptr(out), int(fa),
                              int(fb))
        outs.append(out)
    _check(lib().f8_gemm_grouped(arr, len(problems), _stream(stream)), "f8_gemm_grouped")
    return outs


def f8_linear_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(lib().f8_linear_workspace_bytes(M, N, K))


@dataclass
class LinearSaved:
    """Device buffers the forward pass leaves for the backward pass.  A
    member of a group (group_saved) shares x_t and x_scalars with the
    group's other members; its scalars[0:2] are then unused."""
    x_t: torch.Tensor      # [K, M] uint8
    w_t: torch.Tensor      # [K, N] uint8
    scalars: torch.Tensor  # [4] fp32: amax_x, scale_x, amax_w, scale_w
    x_scalars: torch.Tensor | None = None  # [2] fp32 amax_x, scale_x shared by a group

    @classmethod
    def empty(cls, M: int, N: int, K: int, device) -> "LinearSaved":
        return cls(torch.empty((K, M), dtype=torch.uint8, device=device),
                   torch.empty((K, N), dtype=torch.uint8, device=device),
                   torch.empty(4, dtype=torch.float32, device=device))

    def c_struct(self) -> _Saved:
        p = self.scalars.data_ptr()
        px = self.x_scalars.data_ptr() if self.x_scalars is not None else p
        return _Saved(self.x_t.data_ptr(), self.w_t.data_ptr(), px, px + 4, p + 8, p + 12)

    @property
    def amax_x(self):
        return (self.x_scalars if self.x_scalars is not None else self.scalars)[0]

    @property
    def scale_x(self):
        return (self.x_scalars if self.x_scalars is not None else self.scalars)[1]

    @property
    def amax_w(self): return self.scalars[2]

    @property
    def scale_w(self): return self.scalars[3]


def workspace(M: int, N: int, K: int, device) -> torch.Tensor:
    return torch.empty(max(f8_linear_workspace_bytes(M, N, K), 1), dtype=torch.uint8, device=device)


def f8_quantize_multi_workspace_bytes() -> int:
    return int(lib().f8_quantize_multi_workspace_bytes())


def f8_quantize_multi(xs, fmt: int = F8_E4M3, outs=None, ws: torch.Tensor | None = None,
                      want_q: bool = True, want_t: bool = True, stream=None) -> list:
    """Each 2-D bf16 tensor of ``xs`` quantised with its own amax and scale
    (f8_quantize_multi): returns [(q, q_t, scale, amax), ...].  ``outs`` may
    give those buffers per tensor."""
    n = len(xs)
    arr = (_QuantTensor * n)()
    res = []
    for i, x in enumerate(xs):
        if x.dtype != torch.bfloat16 or x.dim() != 2:
            raise TypeError("f8_quantize_multi takes 2-D bf16 tensors")
        rows, cols = x.shape
        dev = x.device
        if outs is not None:
            q, q_t, sc, am = outs[i]
        else:
            q = torch.empty((rows, cols), dtype=torch.uint8, device=dev) if want_q else None
            q_t = torch.empty((cols, rows), dtype=torch.uint8, device=dev) if want_t else None
            sc = torch.empty((), dtype=torch.float32, device=dev)
            am = torch.empty((), dtype=torch.float32, device=dev)
        arr[i] = _QuantTensor(_ptr(x), rows, cols, _ptr(am), _ptr(sc), _ptr(q), _ptr(q_t))
        res.append((q, q_t, sc, am))
    if ws is None:
        ws = torch.empty(f8_quantize_multi_workspace_bytes(), dtype=torch.uint8, device=xs[0].device)
    _check(lib().f8_quantize_multi(arr, n, int(fmt), _ptr(ws), ws.numel(), _stream(stream)),
           "f8_quantize_multi")
    return res


def f8_linear_group_workspace_bytes(M: int, K: int, Ns) -> int:
    arr = (ctypes.c_int64 * len(Ns))(*Ns)
    return int(lib().f8_linear_group_workspace_bytes(M, K, arr, len(Ns)))


def group_workspace(M: int, K: int, Ns, device) -> torch.Tensor:
    return torch.empty(max(f8_linear_group_workspace_bytes(M, K, Ns), 1), dtype=torch.uint8,
                       device=device)


def group_saved(M: int, K: int, Ns, device) -> list:
    """Saved buffers of a group of linears sharing X [M, K]: one q(X)^T and
    one (amax_x, scale_x) shared, q(W_i)^T and (amax_w, scale_w) per member."""
    x_t = torch.empty((K, M), dtype=torch.uint8, device=device)
    xs = torch.empty(2, dtype=torch.float32, device=device)
    return [LinearSaved(x_t, torch.empty((K, N), dtype=torch.uint8, device=device),
                        torch.empty(4, dtype=torch.float32, device=device), xs) for N in Ns]


def _group_array(saved, Ns, w=None, y=None, dy=None, dx=None, dw=None):
    n = len(saved)
    arr = (_GroupLinear * n)()
    for i in range(n):
        arr[i] = _GroupLinear(Ns[i], _ptr(w[i]) if w else None, _ptr(y[i]) if y else None,
                              _ptr(dy[i]) if dy else None, _ptr(dx[i]) if dx else None,
                              _ptr(dw[i]) if dw else None, saved[i].c_struct())
    return arr


def f8_linear_fwd_group(x: torch.Tensor, ws_: list, ys: list | None = None, saved: list | None = None,
                        ws: torch.Tensor | None = None, stream=None):
    """Y_i = X W_i^T for linears sharing X (f8_linear_fwd_group): X quantised
    once, each W_i with its own scale; returns (ys, saved)."""
    _need("f8_linear_fwd_group", torch.bfloat16, x, *ws_)
    M, K = x.shape
    Ns = [w.shape[0] for w in ws_]
    for w in ws_:
        if w.shape[1] != K:
            raise ValueError("in-feature sizes differ")
    dev = x.device
    if ys is None:
        ys = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for N in Ns]
    if saved is None:
        saved = group_saved(M, K, Ns, dev)
    if ws is None:
        ws = group_workspace(M, K, Ns, dev)
    arr = _group_array(saved, Ns, w=ws_, y=ys)
    _check(lib().f8_linear_fwd_group(_ptr(x), M, K, arr, len(Ns), _ptr(ws), ws.numel(),
                                     _stream(stream)), "f8_linear_fwd_group")
    return ys, saved


def f8_linear_bwd_group(dys: list, saved: list, K: int, dxs: list | None = None,
                        dws: list | None = None, ws: torch.Tensor | None = None,
                        fmt: int = F8_E4M3, want_dx: bool = True, want_dw: bool = True, stream=None):
    """dX_i = dY_i W_i, dW_i = dY_i^T X for the group of f8_linear_fwd_group
    (f8_linear_bwd_group); returns (dxs, dws) (lists, or None if not wanted)."""
    _need("f8_linear_bwd_group", torch.bfloat16, *dys)
    M = dys[0].shape[0]
    Ns = [dy.shape[1] for dy in dys]
    dev = dys[0].device
    if want_dx and dxs is None:
        dxs = [torch.empty((M, K), dtype=torch.bfloat16, device=dev) for _ in Ns]
    if want_dw and dws is None:
        dws = [torch.empty((N, K), dtype=torch.bfloat16, device=dev) for N in Ns]
    if ws is None:
        ws = group_workspace(M, K, Ns, dev)
    arr = _group_array(saved, Ns, dy=dys, dx=dxs if want_dx else None, dw=dws if want_dw else None)
    _check(lib().f8_linear_bwd_group(arr, len(Ns), M, K, int(fmt), _ptr(ws), ws.numel(),
                                     _stream(stream)), "f8_linear_bwd_group")
    return (dxs if want_dx else None), (dws if want_dw else None)


def f8_linear_fwd(x: torch.Tensor, w: torch.Tensor, y: torch.Tensor | None = None,
                  saved: LinearSaved | None = None, ws: torch.Tensor | None = None, stream=None):
    """Y = X W^T through the Float8 path; returns (Y, saved)."""
    _need("f8_linear_fwd", torch.bfloat16, x, w)
    M, K = x.shape
    N, K2 = w.shape
    if K != K2:
        raise ValueError("in-feature sizes differ")
    dev = x.device
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    if saved is None:
        saved = LinearSaved.empty(M, N, K, dev)
    if ws is None:
        ws = workspace(M, N, K, dev)
    s = saved.c_struct()
    _check(lib().f8_linear_fwd(_ptr(x), _ptr(w), M, N, K, _ptr(y), ctypes.byref(s), _ptr(ws),
                               ws.numel(), _stream(stream)), "f8_linear_fwd")
    return y, saved


def f8_linear_fwd_noalloc(x: torch.Tensor, w: torch.Tensor, y: torch.Tensor | None = None,
                          saved: LinearSaved | None = None, stream=None):
    """f8_linear_fwd without a workspace argument: the C entry point uses a
    static device array instead, for callers that cannot allocate device memory."""
    _need("f8_linear_fwd_noalloc", torch.bfloat16, x, w)
    M, K = x.shape
    N, K2 = w.shape
    if K != K2:
        raise ValueError("in-feature sizes differ")
    dev = x.device
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    if saved is None:
        saved = LinearSaved.empty(M, N, K, dev)
    s = saved.c_struct()
    _check(lib().f8_linear_fwd_noalloc(_ptr(x), _ptr(w), M, N, K, _ptr(y), ctypes.byref(s),
                                       _stream(stream)), "f8_linear_fwd_noalloc")
    return y, saved


def f8_quantize_swiglu(a: torch.Tensor, b: torch.Tensor, h: torch.Tensor | None = None,
                       amax_out=None, scale_out=None, q=None, q_t=None, ws=None, stream=None):
    """h = bf16(silu(a) * b) with its amax from the producing pass, then its
    E4M3 cast: returns (q, q_t, scale, amax, h)."""
    if a.shape != b.shape or a.dtype != torch.bfloat16 or b.dtype != torch.bfloat16 or a.dim() != 2:
        raise TypeError("f8_quantize_swiglu takes two 2-D bf16 tensors of one shape")
    rows, cols = a.shape
    dev = a.device
    amax_out = torch.empty((), dtype=torch.float32, device=dev) if amax_out is None else amax_out
    scale_out = torch.empty((), dtype=torch.float32, device=dev) if scale_out is None else scale_out
    q = torch.empty((rows, cols), dtype=torch.uint8, device=dev) if q is None else q
    q_t = torch.empty((cols, rows), dtype=torch.uint8, device=dev) if q_t is None else q_t
    if ws is None:
        ws = torch.empty(f8_quantize_workspace_bytes(), dtype=torch.uint8, device=dev)
    h = torch.empty_like(a) if h is None else h
    _check(lib().f8_quantize_swiglu(_ptr(a), _ptr(b), _ptr(h), rows, cols, _ptr(amax_out),
                                    _ptr(scale_out), _ptr(q), _ptr(q_t), _ptr(ws), ws.numel(),
                                    _stream(stream)), "f8_quantize_swiglu")
    return q, q_t, scale_out, amax_out, h


def f8_linear_fwd_swiglu(a: torch.Tensor, b: torch.Tensor, w: torch.Tensor,
                         y: torch.Tensor | None = None, saved: LinearSaved | None = None,
                         ws: torch.Tensor | None = None, h: torch.Tensor | None = None, stream=None):
    """Y = h W^T with h = silu(a) * b produced with its amax; returns (Y, saved)."""
    _need("f8_linear_fwd_swiglu", torch.bfloat16, a, b, w)
    M, K = a.shape
    N, K2 = w.shape
    if K != K2 or a.shape != b.shape:
        raise ValueError("shapes do not match")
    dev = a.device
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    if saved is None:
        saved = LinearSaved.empty(M, N, K, dev)
    if ws is None:
        ws = workspace(M, N, K, dev)
    h = torch.empty_like(a) if h is None else h
    s = saved.c_struct()
    _check(lib().f8_linear_fwd_swiglu(_ptr(a), _ptr(b), _ptr(h), _ptr(w), M, N, K, _ptr(y),
                                      ctypes.byref(s), _ptr(ws), ws.numel(), _stream(stream)),
           "f8_linear_fwd_swiglu")
    return y, saved


def interleave_w13(w1: torch.Tensor, w3: torch.Tensor) -> torch.Tensor:
    """W13 [2F, K] in the row order f8_linear_fwd_w13_swiglu takes: blocks of
    128 rows of W1 and of W3, alternating (a layout copy, no arithmetic)."""
    F, K = w1.shape
    if w3.shape != w1.shape or F % 128:
        raise ValueError("w1 and w3 must both be [F, K] with F % 128 == 0")
    return torch.stack((w1.reshape(F // 128, 128, K), w3.reshape(F // 128, 128, K)),
                       dim=1).reshape(2 * F, K)


def split_ab(ab: torch.Tensor) -> tuple[torch.Tensor, torch.Tensor]:
    """Views a, b [M, F] (strided) of an interleaved AB [M, 2F]."""
    M, N = ab.shape
    v = ab.view(M, N // 256, 2, 128)
    return v[:, :, 0, :].reshape(M, N // 2), v[:, :, 1, :].reshape(M, N // 2)


def f8_linear_fwd_w13_swiglu(x: torch.Tensor, w13: torch.Tensor, ab: torch.Tensor | None = None,
                             h: torch.Tensor | None = None, saved: LinearSaved | None = None,
                             amax_h: torch.Tensor | None = None,
                             scale_h: torch.Tensor | None = None, h_q: torch.Tensor | None = None,
                             h_t: torch.Tensor | None = None, ws: torch.Tensor | None = None,
                             stream=None):
    """AB = X W13^T (Float8 linear), h = silu(a) * b and its E4M3 copies from
    the GEMM epilogue; returns (ab, h, saved, h_q, h_t, scale_h, amax_h)."""
    _need("f8_linear_fwd_w13_swiglu", torch.bfloat16, x, w13)
    M, K = x.shape
    N, K2 = w13.shape
    if K != K2 or N % 256:
        raise ValueError("w13 must be [2F, K] with F % 128 == 0")
    F = N // 2
    dev = x.device
    ab = torch.empty((M, N), dtype=torch.bfloat16, device=dev) if ab is None else ab
    h = torch.empty((M, F), dtype=torch.bfloat16, device=dev) if h is None else h
    saved = LinearSaved.empty(M, N, K, dev) if saved is None else saved
    amax_h = torch.empty(1, dtype=torch.float32, device=dev) if amax_h is None else amax_h
    scale_h = torch.empty(1, dtype=torch.float32, device=dev) if scale_h is None else scale_h
    h_q = torch.empty((M, F), dtype=torch.uint8, device=dev) if h_q is None else h_q
    h_t = torch.empty((F, M), dtype=torch.uint8, device=dev) if h_t is None else h_t
    ws = workspace(M, N, K, dev) if ws is None else ws
    s = saved.c_struct()
    _check(lib().f8_linear_fwd_w13_swiglu(_ptr(x), _ptr(w13), M, F, K, _ptr(ab), _ptr(h),
                                          ctypes.byref(s), _ptr(amax_h), _ptr(scale_h), _ptr(h_q),
                                          _ptr(h_t), _ptr(ws), ws.numel(), _stream(stream)),
           "f8_linear_fwd_w13_swiglu")
    return ab, h, saved, h_q, h_t, scale_h, amax_h


def f8_linear_bwd_w13_swiglu(dh: torch.Tensor, ab: torch.Tensor, saved: LinearSaved,
                             dab: torch.Tensor | None = None, dx: torch.Tensor | None = None,
                             dw: torch.Tensor | None = None, ws: torch.Tensor | None = None,
                             want_dx: bool = True, want_dw: bool = True, dy_fmt: int = F8_E4M3,
                             stream=None):
    """d(AB) from dh and the forward's AB (quantised in format dy_fmt), then
    dX, dW13 of the w1+w3 group; returns (dx, dw, dab)."""
    _need("f8_linear_bwd_w13_swiglu", torch.bfloat16, dh, ab)
    M, F = dh.shape
    K = saved.x_t.shape[0]
    if ab.shape != (M, 2 * F):
        raise ValueError("ab must be [M, 2F] for dh [M, F]")
    dev = dh.device
    dab = torch.empty_like(ab) if dab is None else dab
    if dx is None and want_dx:
        dx = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    if dw is None and want_dw:
        dw = torch.empty((2 * F, K), dtype=torch.bfloat16, device=dev)
    ws = workspace(M, 2 * F, K, dev) if ws is None else ws
    s = saved.c_struct()
    _check(lib().f8_linear_bwd_w13_swiglu(_ptr(dh), _ptr(ab), ctypes.byref(s), M, F, K, _ptr(dab),
                                          int(dy_fmt), _ptr(dx), _ptr(dw), _ptr(ws), ws.numel(),
                                          _stream(stream)), "f8_linear_bwd_w13_swiglu")
    return dx, dw, dab


def f8_quantize_swiglu_bwd(dh: torch.Tensor, ab: torch.Tensor, dab: torch.Tensor | None = None,
                           amax_out=None, scale_out=None, q=None, q_t=None, ws=None,
                           fmt: int = F8_E4M3, stream=None):
    """d(AB) from dh and the forward's AB with its amax, then its cast to
    format fmt: returns (q, q_t, scale, amax, dab)."""
    _need("f8_quantize_swiglu_bwd", torch.bfloat16, dh, ab)
    M, F = dh.shape
    if ab.shape != (M, 2 * F):
        raise ValueError("ab must be [M, 2F] for dh [M, F]")
    dev = dh.device
    dab = torch.empty_like(ab) if dab is None else dab
    amax_out = torch.empty((), dtype=torch.float32, device=dev) if amax_out is None else amax_out
    scale_out = torch.empty((), dtype=torch.float32, device=dev) if scale_out is None else scale_out
    q = torch.empty((M, 2 * F), dtype=torch.uint8, device=dev) if q is None else q
    q_t = torch.empty((2 * F, M), dtype=torch.uint8, device=dev) if q_t is None else q_t
    if ws is None:
        ws = torch.empty(f8_quantize_workspace_bytes(), dtype=torch.uint8, device=dev)
    _check(lib().f8_quantize_swiglu_bwd(_ptr(dh), _ptr(ab), M, F, _ptr(dab), int(fmt),
                                        _ptr(amax_out), _ptr(scale_out), _ptr(q), _ptr(q_t),
                                        _ptr(ws), ws.numel(), _stream(stream)),
           "f8_quantize_swiglu_bwd")
    return q, q_t, scale_out, amax_out, dab


def f8_gemm_w13_swiglu(x_q: torch.Tensor, w13_q: torch.Tensor, scale_x: torch.Tensor,
                       scale_w13: torch.Tensor, ab: torch.Tensor | None = None,
                       h: torch.Tensor | None = None, amax_h: torch.Tensor | None = None,
                       stream=None):
    """AB = q(X) q(W13)^T / (s_x s_w13) and h = silu(a) * b with max |h|;
    returns (ab, h, amax_h)."""
    _need("f8_gemm_w13_swiglu", torch.uint8, x_q, w13_q)
    M, K = x_q.shape
    N, K2 = w13_q.shape
    if K != K2 or N % 256:
        raise ValueError("w13_q must be [2F, K] with F % 128 == 0")
    dev = x_q.device
    ab = torch.empty((M, N), dtype=torch.bfloat16, device=dev) if ab is None else ab
    h = torch.empty((M, N // 2), dtype=torch.bfloat16, device=dev) if h is None else h
    amax_h = torch.empty(1, dtype=torch.float32, device=dev) if amax_h is None else amax_h
    _check(lib().f8_gemm_w13_swiglu(_ptr(x_q), _ptr(w13_q), M, N // 2, K, _ptr(scale_x),
                                    _ptr(scale_w13), _ptr(ab), _ptr(h), _ptr(amax_h),
                                    _stream(stream)), "f8_gemm_w13_swiglu")
    return ab, h, amax_h


def f8_linear_bwd(dy: torch.Tensor, saved: LinearSaved, K: int | None = None,
                  dx: torch.Tensor | None = None, dw: torch.Tensor | None = None,
                  ws: torch.Tensor | None = None, want_dx: bool = True, want_dw: bool = True,
                  dy_fmt: int = F8_E4M3, stream=None):
    """(dX, dW) of the linear whose forward produced ``saved``; ``dy_fmt``
    E5M2 routes through f8_linear_bwd_fmt."""
    _need("f8_linear_bwd", torch.bfloat16, dy)
    M, N = dy.shape
    K = saved.x_t.shape[0]
    dev = dy.device
    if dx is None and want_dx:
        dx = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    if dw is None and want_dw:
        dw = torch.empty((N, K), dtype=torch.bfloat16, device=dev)
    if ws is None:
        ws = workspace(M, N, K, dev)
    s = saved.c_struct()
    if dy_fmt == F8_E4M3:
        _check(lib().f8_linear_bwd(_ptr(dy), ctypes.byref(s), M, N, K, _ptr(dx), _ptr(dw), _ptr(ws),
                                   ws.numel(), _stream(stream)), "f8_linear_bwd")
    else:
        _check(lib().f8_linear_bwd_fmt(_ptr(dy), int(dy_fmt), ctypes.byref(s), M, N, K, _ptr(dx),
                                       _ptr(dw), _ptr(ws), ws.numel(), _stream(stream)),
               "f8_linear_bwd_fmt")
    return dx, dw


def f8_transpose_u8(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """out[c, r] = x[r, c] for a 2-D uint8 tensor (f8_transpose_u8)."""
    if x.dtype != torch.uint8 or x.dim() != 2:
        raise TypeError("f8_transpose_u8 takes a 2-D uint8 tensor")
    rows, cols = x.shape
    if out is None:
        out = torch.empty((cols, rows), dtype=torch.uint8, device=x.device)
    _check(lib().f8_transpose_u8(_ptr(x), rows, cols, _ptr(out), _stream(stream)), "f8_transpose_u8")
    return out


def f8_linear_fwd_qw_workspace_bytes(M: int, K: int) -> int:
    return int(lib().f8_linear_fwd_qw_workspace_bytes(M, K))


def f8_linear_fwd_qw(x: torch.Tensor, w_q: torch.Tensor, saved: LinearSaved,
                     y: torch.Tensor | None = None, ws: torch.Tensor | None = None, stream=None):
    """Y = X W^T for a weight that arrives quantised (w_q [N, K] uint8, with
    saved.w_t = q(W)^T and saved's amax_w / scale_w set by the caller);
    writes saved's X part; returns Y."""
    _need("f8_linear_fwd_qw", torch.bfloat16, x)
    _need("f8_linear_fwd_qw", torch.uint8, w_q)
    M, K = x.shape
    N, K2 = w_q.shape
    if K != K2:
        raise ValueError("in-feature sizes differ")
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    if ws is None:
        ws = torch.empty(max(f8_linear_fwd_qw_workspace_bytes(M, K), 1), dtype=torch.uint8,
                         device=x.device)
    s = saved.c_struct()
    _check(lib().f8_linear_fwd_qw(_ptr(x), _ptr(w_q), M, N, K, _ptr(y), ctypes.byref(s), _ptr(ws),
                                  ws.numel(), _stream(stream)), "f8_linear_fwd_qw")
    return y
