"""f8_linear_fwd_noalloc: the forward pass for callers that cannot allocate
device memory (e.g. a plugin inside a framework that owns all device memory,
or a service with a fixed device-memory budget).  Its workspace is a static
device array inside the library instead of a caller-provided buffer; it
runs f8_linear_fwd's own code on that array.

Checked here through the C ABI:
- two calls in a row (different shapes and inputs, so the second call runs
  on the first call's leftover scratch) each give Y and the saved tensors
  bit-identical to the workspace entry point f8_linear_fwd, and Y within the
  GEMM bar of the oracle, with the saved scales and E4M3 bytes equal to the
  oracle's;
- after a warm-up call (whose first use of the library's module on the
  device may map its static arrays), a call changes the device's free memory
  by nothing: it allocates no device memory;
- a problem whose workspace exceeds the static array is refused before
  anything is launched.
This file is collected last so a run that stops at the first failure has
already run every other test; it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from float8_mixed_precision_gb300 import workloads as wl
from tolerance import check_close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def f8():
    import float8_mixed_precision_gb300 as m
    from float8_mixed_precision_gb300 import build
    build.build()
    oracle.build()
    m.lib()
    return m


def _noalloc_c(f8, x, w, M, N, K, y, saved):
    """Direct C-ABI call of f8_linear_fwd_noalloc into caller-allocated outputs."""
    s = saved.c_struct()
    st = f8.lib().f8_linear_fwd_noalloc(x.data_ptr(), w.data_ptr(), M, N, K, y.data_ptr(),
                                        ctypes.byref(s), torch.cuda.current_stream().cuda_stream)
    assert st == 0, f8.f8_status_string(st)


def test_two_calls_match_the_workspace_entry_point_and_the_oracle(f8):
    for i, (M, N, K) in enumerate([(1024, 768, 2048), (512, 1536, 1024)]):
        d = wl.custom_linear(M, K, N, seed=900 + i)
        x, w = d["x"].to(DEV), d["w"].to(DEV)
        y_ref, saved_ref = f8.f8_linear_fwd(x, w)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
        saved = f8.LinearSaved.empty(M, N, K, DEV)
        _noalloc_c(f8, x, w, M, N, K, y, saved)
        assert f8.f8_last_device_status() == 0
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16)), f"call {i + 1}: Y differs"
        assert torch.equal(saved.scalars, saved_ref.scalars)
        assert torch.equal(saved.x_t, saved_ref.x_t) and torch.equal(saved.w_t, saved_ref.w_t)
        fwd = oracle.linear_fwd(wl.bits(d["x"]), wl.bits(d["w"]))
        assert saved.scalars.cpu().tolist() == [float(fwd["x"]["amax"]), float(fwd["x"]["scale"]),
                                                float(fwd["w"]["amax"]), float(fwd["w"]["scale"])]
        assert np.array_equal(saved.x_t.cpu().numpy(), fwd["x"]["qt"])
        assert np.array_equal(saved.w_t.cpu().numpy(), fwd["w"]["qt"])
        check_close(y, fwd["y"], what=f"noalloc call {i + 1} Y")


def test_a_call_allocates_no_device_memory(f8):
    M, N, K = 512, 1024, 1024
    d = wl.custom_linear(M, K, N, seed=950)
    x, w = d["x"].to(DEV), d["w"].to(DEV)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    saved = f8.LinearSaved.empty(M, N, K, DEV)
    _noalloc_c(f8, x, w, M, N, K, y, saved)     # warm-up: module and array mapped
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    _noalloc_c(f8, x, w, M, N, K, y, saved)
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert f8.f8_last_device_status() == 0
    assert free1 == free0, (free0, free1)


def test_too_large_is_refused(f8):
    M, N, K = 8192, 4096, 8192       # 64 MiB + 32 MiB of E4M3 copies > 64 MiB
    assert M * K + N * K > 64 * 1024 * 1024
    s = f8.binding._Saved(256, 256, 256, 260, 264, 268)
    st = f8.lib().f8_linear_fwd_noalloc(256, 256, M, N, K, 256, ctypes.byref(s), None)
    assert st == f8.binding.F8_ERR_SHAPE
