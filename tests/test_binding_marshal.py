"""The Python binding's marshalling, without a GPU: every wrapper is called on
small CPU tensors against a stand-in for libf8 that checks the argument count
of each C call against the argtypes the real library was given, records the
call and returns F8_OK.  Nothing runs on a device; this catches wrappers whose
C call no longer matches include/f8.h."""
import ctypes

import pytest
import torch

from float8_mixed_precision_gb300 import binding


class _Recorder:
    def __init__(self, real):
        self.real = real
        self.calls = []

    def __getattr__(self, name):
        fn = getattr(self.real, name)

        def call(*args):
            assert len(args) == len(fn.argtypes), (name, len(args), len(fn.argtypes))
            self.calls.append(name)
            if fn.restype is ctypes.c_size_t:
                return 4096
            return 0
        return call


@pytest.fixture()
def rec(monkeypatch):
    from float8_mixed_precision_gb300 import build
    build.build()
    real = binding.lib()
    r = _Recorder(real)
    monkeypatch.setattr(binding, "lib", lambda: r)
    monkeypatch.setattr(binding, "_ptr", lambda t: None if t is None else t.data_ptr())
    monkeypatch.setattr(binding, "_stream", lambda s: 0)
    return r


def _bf(*shape):
    return torch.zeros(shape, dtype=torch.bfloat16)


def test_every_wrapper_marshals(rec):
    M, N, K, F = 32, 48, 64, 128
    x, w, dy = _bf(M, K), _bf(N, K), _bf(M, N)
    binding.f8_amax(x)
    binding.f8_cast_transpose(x, torch.ones(1), torch.ones(1))
    binding.f8_quantize(x)
    binding.f8_quantize(x, fmt=binding.F8_E5M2)
    q = torch.zeros((M, K), dtype=torch.uint8)
    binding.f8_gemm(q, torch.zeros((N, K), dtype=torch.uint8), torch.ones(1), torch.ones(1))
    binding.f8_gemm(q, torch.zeros((N, K), dtype=torch.uint8), torch.ones(1), torch.ones(1),
                    fmt_a=binding.F8_E5M2)
    qb = torch.zeros((N, K), dtype=torch.uint8)
    binding.f8_gemm_grouped([(q, qb, torch.ones(1), torch.ones(1)),
                             (qb, q, torch.ones(1), torch.ones(1), None, binding.F8_E5M2)])
    y, saved = binding.f8_linear_fwd(x, w)
    binding.f8_linear_fwd_noalloc(x, w)
    binding.f8_linear_bwd(dy, saved)
    binding.f8_linear_bwd(dy, saved, dy_fmt=binding.F8_E5M2)
    binding.f8_quantize_swiglu(x, x)
    binding.f8_linear_fwd_swiglu(x, x, w)
    binding.f8_linear_fwd_w13_swiglu(x, _bf(2 * F, K))
    binding.f8_gemm_w13_swiglu(q, torch.zeros((2 * F, K), dtype=torch.uint8), torch.ones(1),
                               torch.ones(1))
    _, _, saved13, _, _, _, _ = binding.f8_linear_fwd_w13_swiglu(x, _bf(2 * F, K))
    binding.f8_linear_bwd_w13_swiglu(_bf(M, F), _bf(M, 2 * F), saved13)
    binding.f8_quantize_swiglu_bwd(_bf(M, F), _bf(M, 2 * F))
    binding.f8_selftest_wait_timeout(1000)
    binding.f8_selftest_bounds()
    binding.f8_quantize_multi([x, w, dy])
    binding.f8_quantize_multi([x], fmt=binding.F8_E5M2, want_q=False)
    binding.f8_gemm_grouped([(q, qb, torch.ones(1), torch.ones(1))] * 5)
    ys, gsaved = binding.f8_linear_fwd_group(x, [w, _bf(2 * N, K)])
    binding.f8_linear_bwd_group([dy, _bf(M, 2 * N)], gsaved, K)
    binding.f8_linear_bwd_group([dy, _bf(M, 2 * N)], gsaved, K, want_dx=False)
    assert gsaved[0].x_t is gsaved[1].x_t and gsaved[0].x_scalars is gsaved[1].x_scalars
    binding.f8_transpose_u8(torch.zeros((N, K), dtype=torch.uint8))
    binding.f8_linear_fwd_qw(x, torch.zeros((N, K), dtype=torch.uint8), saved)
    wrapped = {n for n in binding.EXPORTS if hasattr(binding, n)}
    called = set(rec.calls)
    assert wrapped - {"f8_status_string", "f8_last_device_status", "f8_set_wait_limit_ns",
                      "f8_kernel_launches",
                      "f8_linear_workspace_bytes", "f8_quantize_workspace_bytes",
                      "f8_quantize_multi_workspace_bytes",
                      "f8_linear_fwd_qw_workspace_bytes"} <= called, \
        sorted(wrapped - called)


def test_wrappers_reject_wrong_dtypes(rec):
    """Every wrapper that hands a tensor's bytes to the C ABI refuses a
    tensor of the wrong type or rank before any C call (the kernels would
    read fp32 or fp8 bytes as bf16, or the reverse)."""
    M, N, K, F = 32, 48, 64, 128
    f32 = torch.zeros((M, K), dtype=torch.float32)
    x, w, dy = _bf(M, K), _bf(N, K), _bf(M, N)
    q, qb = torch.zeros((M, K), dtype=torch.uint8), torch.zeros((N, K), dtype=torch.uint8)
    saved = binding.LinearSaved(torch.zeros((K, M), dtype=torch.uint8),
                                torch.zeros((K, N), dtype=torch.uint8), torch.zeros(4))
    one = torch.ones(1)
    bad = [
        lambda: binding.f8_linear_fwd(f32, w),
        lambda: binding.f8_linear_fwd(x, w.float()),
        lambda: binding.f8_linear_fwd(x.reshape(-1), w),
        lambda: binding.f8_linear_fwd_noalloc(f32, w),
        lambda: binding.f8_linear_bwd(dy.float(), saved),
        lambda: binding.f8_gemm(x, qb, one, one),
        lambda: binding.f8_gemm(q, w, one, one),
        lambda: binding.f8_gemm_grouped([(q, qb.float(), one, one)]),
        lambda: binding.f8_linear_fwd_group(f32, [w]),
        lambda: binding.f8_linear_fwd_group(x, [w, w.float()]),
        lambda: binding.f8_linear_bwd_group([dy.float()], [saved], K),
        lambda: binding.f8_linear_fwd_qw(f32, qb, saved),
        lambda: binding.f8_linear_fwd_qw(x, w, saved),
        lambda: binding.f8_linear_fwd_swiglu(_bf(M, F), _bf(M, F).float(), _bf(N, F)),
        lambda: binding.f8_linear_fwd_w13_swiglu(f32, _bf(2 * F, K)),
        lambda: binding.f8_linear_bwd_w13_swiglu(_bf(M, F).float(), _bf(M, 2 * F), saved),
        lambda: binding.f8_quantize_swiglu_bwd(_bf(M, F), _bf(M, 2 * F).float()),
        lambda: binding.f8_gemm_w13_swiglu(x, torch.zeros((2 * F, K), dtype=torch.uint8), one, one),
    ]
    for i, call in enumerate(bad):
        with pytest.raises(TypeError):
            call()
        assert rec.calls == [], (i, rec.calls)
