"""The checked build (device bounds checks compiled in, -DF8_BOUNDS_CHECK)
runs the kernel, linear, E5M2, SwiGLU, W13, paired-quantisation, grouped
(multi-tensor quantisation, grouped GEMMs, shared-input linears), FP8
all-gather (byte transpose), past-2^31-element and PyTorch-module parity
tests in a child process.  Every manually indexed global access is tested
against its buffer first, and every one of those tests asserts a clean
device status, so a single index outside its buffer would fail the run as
F8_ERR_BOUNDS.  The check mechanism itself is shown to fire by
f8_selftest_bounds, which fails one check without touching memory.  The
full-size workload tests stay out (their shapes are covered at the same
launch configurations by the smaller cases of the same kernels), to keep
the run to a few minutes.  Collected last (zz) because it builds a second
library."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def checked_lib():
    from float8_mixed_precision_gb300 import build
    return build.build(checked=True)


def _child(env_lib, args, timeout):
    env = dict(os.environ, F8_LIBRARY=env_lib)
    return subprocess.run([sys.executable] + args, cwd=ROOT, env=env, capture_output=True,
                          text=True, timeout=timeout)


def test_release_build_has_no_checks():
    import float8_mixed_precision_gb300 as f8
    from float8_mixed_precision_gb300 import build
    build.build()
    f8.lib()
    if os.environ.get("F8_LIBRARY"):
        pytest.skip("run against another build")
    assert f8.f8_selftest_bounds() == f8.binding.F8_ERR_UNSUPPORTED
    assert f8.f8_last_device_status() == 0


def test_checked_build_selftest_fires(checked_lib):
    code = ("import float8_mixed_precision_gb300 as f8; "
            "assert f8.f8_selftest_bounds() == 0; "
            "s = f8.f8_last_device_status(); "
            "assert s == f8.binding.F8_ERR_BOUNDS, s; "
            "assert f8.f8_last_device_status() == 0; print('ok')")
    r = _child(checked_lib, ["-c", code], 300)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr


def test_parity_suites_under_checked_build(checked_lib):
    tests = ["tests/test_gpu_kernels.py", "tests/test_gpu_linear.py", "tests/test_gpu_e5m2.py",
             "tests/test_gpu_swiglu.py", "tests/test_gpu_w13.py", "tests/test_gpu_quant_pair.py",
             "tests/test_gpu_group.py", "tests/test_gpu_fsdp.py", "tests/test_gpu_max_size.py",
             "tests/test_gpu_nn.py"]
    r = _child(checked_lib, ["-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
                             "-k", "not full_size and not every_output and not llama8b and not all_gather",
                             *tests],
               1500)
    tail = (r.stdout + r.stderr)[-3000:]
    assert r.returncode == 0, tail
    import re
    m = re.search(r"(\d+) passed", r.stdout)
    assert m is not None and int(m.group(1)) >= 100, tail
