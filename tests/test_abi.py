"""The C ABI without a GPU: the library loads, exports every function
include/f8.h declares, and rejects bad arguments on the host before it
touches the device (so these calls return without any CUDA work)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from float8_mixed_precision_gb300 import build
    build.build()
    import float8_mixed_precision_gb300 as f8
    return f8.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "f8.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(f8_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_five_path_calls():
    names = _declared()
    for n in ("f8_amax", "f8_cast_transpose", "f8_gemm", "f8_linear_fwd", "f8_linear_bwd"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    import float8_mixed_precision_gb300 as f8
    names = _declared()
    assert set(names) == set(f8.EXPORTS)
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    import float8_mixed_precision_gb300 as f8
    for s in range(8):
        assert f8.f8_status_string(s).startswith("F8_")
    assert "UNKNOWN" in f8.f8_status_string(99)


def test_workspace_bytes(L):
    import float8_mixed_precision_gb300 as f8
    M, N, K = 8192, 1024, 4096
    ws = f8.f8_linear_workspace_bytes(M, N, K)
    assert ws >= M * K + N * K and ws >= 2 * M * N
    assert f8.f8_linear_workspace_bytes(0, 1, 1) == 0


FAKE = 1 << 40          # an aligned address that is never dereferenced
FAKE_MIS = FAKE + 8     # 8-byte aligned, not 16


@pytest.mark.parametrize("args,want", [
    ((FAKE, FAKE, 16, 16, 17, FAKE, FAKE, FAKE, None), 3),     # K % 16
    ((FAKE, FAKE, -1, 16, 16, FAKE, FAKE, FAKE, None), 1),     # negative M
    ((FAKE, FAKE, 16, 16, 16, None, FAKE, FAKE, None), 1),     # missing scale
    ((FAKE_MIS, FAKE, 16, 16, 16, FAKE, FAKE, FAKE, None), 2), # misaligned A
    ((FAKE, FAKE, 16, 16, 16, FAKE, FAKE, FAKE_MIS, None), 2), # misaligned C
    ((None, FAKE, 16, 16, 16, FAKE, FAKE, FAKE, None), 1),     # NULL A
    ((FAKE, FAKE, 1 << 29, 1 << 29, 16, FAKE, FAKE, FAKE, None), 3),  # 2^36 tiles
])
def test_gemm_rejects_bad_arguments_on_host(L, args, want):
    assert L.f8_gemm(*args) == want


def test_other_calls_reject_bad_arguments_on_host(L):
    assert L.f8_amax(FAKE, -5, FAKE, None) == 1
    assert L.f8_amax(FAKE_MIS, 5, FAKE, None) == 2
    assert L.f8_amax(FAKE, 5, None, None) == 1
    assert L.f8_cast_transpose(FAKE, 4, -1, FAKE, None, FAKE, FAKE, None) == 1
    assert L.f8_cast_transpose(FAKE, 4, 4, None, None, FAKE, FAKE, None) == 1
    assert L.f8_cast_transpose(FAKE, 4, 4, FAKE, None, FAKE_MIS, FAKE, None) == 2
    from float8_mixed_precision_gb300.binding import _Saved
    s = _Saved(FAKE, FAKE, FAKE, FAKE + 4, FAKE + 8, FAKE + 12)
    ws = 1 << 30
    assert L.f8_linear_fwd(FAKE, FAKE, 16, 16, 24, FAKE, ctypes.byref(s), FAKE, ws, None) == 3
    big = 1 << 29                                      # dX would have 2^35 tiles
    assert L.f8_linear_fwd(FAKE, FAKE, big, 16, big, FAKE, ctypes.byref(s), FAKE, ws, None) == 3
    assert L.f8_linear_fwd(FAKE, FAKE, 0, 16, 16, FAKE, ctypes.byref(s), FAKE, ws, None) == 1
    assert L.f8_linear_fwd(FAKE, FAKE, 16, 16, 16, FAKE, None, FAKE, ws, None) == 1
    assert L.f8_linear_fwd(FAKE, FAKE, 16, 16, 16, FAKE, ctypes.byref(s), FAKE, 10, None) == 1
    assert L.f8_linear_fwd(FAKE, FAKE, 16, 16, 16, FAKE, ctypes.byref(s), FAKE + 16, ws, None) == 2
    bad = _Saved(FAKE, None, FAKE, FAKE, FAKE, FAKE)
    assert L.f8_linear_bwd(FAKE, ctypes.byref(bad), 16, 16, 16, FAKE, FAKE, FAKE, ws, None) == 1
    assert L.f8_linear_bwd(FAKE, ctypes.byref(s), 16, 16, 16, FAKE_MIS, FAKE, FAKE, ws, None) == 2


def test_w13_swiglu_rejects_bad_arguments_on_host(L):
    from float8_mixed_precision_gb300.binding import _Saved
    s = _Saved(FAKE, FAKE, FAKE, FAKE + 4, FAKE + 8, FAKE + 12)
    ws = 1 << 30
    f = L.f8_linear_fwd_w13_swiglu
    ok = (FAKE, FAKE, 256, 128, 64, FAKE, FAKE, ctypes.byref(s), FAKE, FAKE + 4, FAKE, FAKE, FAKE,
          ws, None)

    def call(**kw):
        a = list(ok)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return f(*a)

    assert call(a3=192) == 3            # F % 128
    assert call(a3=0) == 1              # F = 0
    assert call(a2=24) == 3             # M % 16
    assert call(a4=40) == 3             # K % 16
    assert call(a5=None) == 1           # AB missing
    assert call(a6=None) == 1           # h missing
    assert call(a7=None) == 1           # saved missing
    assert call(a10=None) == 1          # h_q missing
    assert call(a13=10) == 1            # workspace too small
    assert call(a6=FAKE_MIS) == 2       # h misaligned
    assert call(a12=FAKE + 16) == 2     # workspace not 256-byte aligned


def test_gemm_w13_swiglu_rejects_bad_arguments_on_host(L):
    f = L.f8_gemm_w13_swiglu
    assert f(FAKE, FAKE, 256, 192, 64, FAKE, FAKE, FAKE, FAKE, FAKE, None) == 3   # F % 128
    assert f(FAKE, FAKE, 256, 128, 0, FAKE, FAKE, FAKE, FAKE, FAKE, None) == 1    # K = 0
    assert f(FAKE, FAKE, 256, 128, 64, FAKE, FAKE, FAKE, FAKE, None, None) == 1   # amax_h
    assert f(FAKE, FAKE, 256, 128, 64, FAKE, FAKE, FAKE_MIS, FAKE, FAKE, None) == 2


def test_package_exposes_every_binding_wrapper():
    """Each C entry point that has a Python wrapper is reachable from the
    package itself (no GPU needed: nothing is called)."""
    import float8_mixed_precision_gb300 as f8
    from float8_mixed_precision_gb300 import binding
    for n in binding.EXPORTS:
        if hasattr(binding, n):
            assert hasattr(f8, n), n
    for n in ("interleave_w13", "split_ab", "LinearSaved", "workspace"):
        assert hasattr(f8, n), n


def test_w13_swiglu_bwd_rejects_bad_arguments_on_host(L):
    from float8_mixed_precision_gb300.binding import _Saved
    s = _Saved(FAKE, FAKE, FAKE, FAKE + 4, FAKE + 8, FAKE + 12)
    f = L.f8_linear_bwd_w13_swiglu
    ws = 1 << 30
    assert f(FAKE, FAKE, ctypes.byref(s), 256, 192, 64, FAKE, 0, FAKE, FAKE, FAKE, ws, None) == 3
    assert f(FAKE, FAKE, ctypes.byref(s), 256, 128, 64, None, 0, FAKE, FAKE, FAKE, ws, None) == 1
    assert f(FAKE, FAKE, None, 256, 128, 64, FAKE, 0, FAKE, FAKE, FAKE, ws, None) == 1
    assert f(FAKE, FAKE, ctypes.byref(s), 256, 128, 64, FAKE, 0, FAKE, FAKE, FAKE, 10, None) == 1
    assert f(FAKE_MIS, FAKE, ctypes.byref(s), 256, 128, 64, FAKE, 0, FAKE, FAKE, FAKE, ws, None) == 2
    assert f(FAKE, FAKE, ctypes.byref(s), 256, 128, 64, FAKE, 2, FAKE, FAKE, FAKE, ws, None) == 1


def test_gemm_grouped_rejects_bad_arguments_on_host(L):
    from float8_mixed_precision_gb300.binding import _GemmProblem
    ok = _GemmProblem(FAKE, FAKE, 256, 256, 256, FAKE, FAKE + 4, FAKE, 0, 0)
    arr = (_GemmProblem * 3)(ok, ok, ok)
    f = L.f8_gemm_grouped
    assert f(None, 1, None) == 1                  # no array
    assert f(arr, 0, None) == 1                   # count outside 1..8
    big = (_GemmProblem * 9)(*([ok] * 9))
    assert f(big, 9, None) == 1

    def with_field(name, value):
        p = _GemmProblem(FAKE, FAKE, 256, 256, 256, FAKE, FAKE + 4, FAKE, 0, 0)
        setattr(p, name, value)
        return (_GemmProblem * 2)(ok, p)

    assert f(with_field("K", 24), 2, None) == 3       # K % 16
    assert f(with_field("M", -1), 2, None) == 1
    assert f(with_field("fmt_a", 2), 2, None) == 1    # no such format
    assert f(with_field("scale_b", None), 2, None) == 1
    assert f(with_field("c", None), 2, None) == 1
    assert f(with_field("b", FAKE_MIS), 2, None) == 2


def test_struct_layouts_match_the_header(tmp_path):
    """The ctypes mirrors of f8_linear_saved and f8_gemm_problem have the
    size and field offsets that a C compiler gives the header's structs
    (compiled here against include/f8.h; no CUDA headers needed)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from float8_mixed_precision_gb300.binding import _GemmProblem, _GroupLinear, _QuantTensor, _Saved
    structs = {"f8_linear_saved": _Saved, "f8_gemm_problem": _GemmProblem,
               "f8_quant_tensor": _QuantTensor, "f8_group_linear": _GroupLinear}
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "f8.h"', "int main(void) {"]
    for cname, cls in structs.items():
        lines.append(f'printf("{cname} size %zu\\n", sizeof({cname}));')
        for field, _ in cls._fields_:
            lines.append(f'printf("{cname} {field} %zu\\n", offsetof({cname}, {field}));')
    lines.append('printf("f8_format size %zu\\n", sizeof(f8_format));')
    lines += ["return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c99", "-I", os.path.join(ROOT, "include"), "-o", str(exe), str(src)],
                   check=True)
    got = {}
    for ln in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.splitlines():
        name, field, value = ln.split()
        got[(name, field)] = int(value)
    for cname, cls in structs.items():
        assert got[(cname, "size")] == ctypes.sizeof(cls), cname
        for field, _ in cls._fields_:
            assert got[(cname, field)] == getattr(cls, field).offset, (cname, field)
    assert got[("f8_format", "size")] == ctypes.sizeof(ctypes.c_int)


def test_quantize_multi_rejects_bad_arguments_on_host(L):
    from float8_mixed_precision_gb300.binding import _QuantTensor
    ok = _QuantTensor(FAKE, 256, 256, FAKE, FAKE + 4, FAKE, FAKE)
    arr = (_QuantTensor * 9)(*([ok] * 9))
    f = L.f8_quantize_multi
    ws = L.f8_quantize_multi_workspace_bytes()
    assert ws > 0
    assert f(None, 1, 0, FAKE, ws, None) == 1          # no array
    assert f(arr, 0, 0, FAKE, ws, None) == 1           # count outside 1..8
    assert f(arr, 9, 0, FAKE, ws, None) == 1
    assert f(arr, 2, 2, FAKE, ws, None) == 1           # no such format
    assert f(arr, 2, 0, None, ws, None) == 1           # no workspace
    assert f(arr, 2, 0, FAKE, ws - 1, None) == 1       # workspace too small
    assert f(arr, 2, 0, FAKE_MIS, ws, None) == 2       # misaligned workspace

    def with_field(name, value):
        p = _QuantTensor(FAKE, 256, 256, FAKE, FAKE + 4, FAKE, FAKE)
        setattr(p, name, value)
        return (_QuantTensor * 2)(ok, p)

    assert f(with_field("rows", -1), 2, 0, FAKE, ws, None) == 1
    assert f(with_field("amax_out", None), 2, 0, FAKE, ws, None) == 1
    assert f(with_field("x", None), 2, 0, FAKE, ws, None) == 1
    assert f(with_field("q", FAKE_MIS), 2, 0, FAKE, ws, None) == 2


def test_linear_group_rejects_bad_arguments_on_host(L):
    from float8_mixed_precision_gb300.binding import _GroupLinear, _Saved
    s0 = _Saved(FAKE, FAKE + 4096, FAKE, FAKE + 4, FAKE + 8, FAKE + 12)
    s1 = _Saved(FAKE, FAKE + 8192, FAKE, FAKE + 4, FAKE + 16, FAKE + 20)
    m0 = _GroupLinear(256, FAKE, FAKE, FAKE, FAKE, FAKE, s0)
    m1 = _GroupLinear(512, FAKE, FAKE, FAKE, FAKE, FAKE, s1)
    arr = (_GroupLinear * 5)(m0, m1, m0, m1, m0)
    Ns = (ctypes.c_int64 * 2)(256, 512)
    wsb = L.f8_linear_group_workspace_bytes(512, 256, Ns, 2)
    assert wsb > 0
    assert L.f8_linear_group_workspace_bytes(512, 256, Ns, 0) == 0
    assert L.f8_linear_group_workspace_bytes(0, 256, Ns, 2) == 0
    fwd, bwd = L.f8_linear_fwd_group, L.f8_linear_bwd_group
    assert fwd(FAKE, 512, 256, None, 2, FAKE, wsb, None) == 1     # no array
    assert fwd(FAKE, 512, 256, arr, 5, FAKE, wsb, None) == 1      # count outside 1..4
    assert fwd(FAKE, 512, 256, arr, 2, FAKE, 4096, None) == 1     # workspace too small
    assert bwd(arr, 2, 512, 256, 0, FAKE, wsb - 1, None) == 1     # (the backward needs wsb)
    assert fwd(FAKE, 500, 256, arr, 2, FAKE, wsb, None) == 3      # M % 16
    assert fwd(None, 512, 256, arr, 2, FAKE, wsb, None) == 1
    assert fwd(FAKE_MIS, 512, 256, arr, 2, FAKE, wsb, None) == 2
    assert bwd(arr, 2, 512, 256, 2, FAKE, wsb, None) == 1         # no such format
    assert bwd(arr, 2, 512, 256, 0, FAKE_MIS, wsb, None) == 2     # workspace alignment
    # the members must share q(X)^T and the X scalars
    s_other = _Saved(FAKE + 65536, FAKE + 8192, FAKE, FAKE + 4, FAKE + 16, FAKE + 20)
    bad = (_GroupLinear * 2)(m0, _GroupLinear(512, FAKE, FAKE, FAKE, FAKE, FAKE, s_other))
    assert fwd(FAKE, 512, 256, bad, 2, FAKE, wsb, None) == 1
    assert bwd(bad, 2, 512, 256, 0, FAKE, wsb, None) == 1
    nody = (_GroupLinear * 2)(m0, _GroupLinear(512, FAKE, FAKE, None, FAKE, FAKE, s1))
    assert bwd(nody, 2, 512, 256, 0, FAKE, wsb, None) == 1


def test_transpose_and_fwd_qw_reject_bad_arguments_on_host(L):
    from float8_mixed_precision_gb300.binding import _Saved
    t = L.f8_transpose_u8
    assert t(FAKE, -1, 4, FAKE, None) == 1
    assert t(None, 4, 4, FAKE, None) == 1
    assert t(FAKE, 0, 4, None, None) == 0          # nothing to do
    s = _Saved(FAKE, FAKE, FAKE, FAKE + 4, FAKE + 8, FAKE + 12)
    f = L.f8_linear_fwd_qw
    wsb = L.f8_linear_fwd_qw_workspace_bytes(256, 512)
    assert wsb >= 256 * 512 and L.f8_linear_fwd_qw_workspace_bytes(0, 512) == 0
    assert f(FAKE, FAKE, 256, 128, 500, FAKE, ctypes.byref(s), FAKE, wsb, None) == 3   # K % 16
    assert f(FAKE, None, 256, 128, 512, FAKE, ctypes.byref(s), FAKE, wsb, None) == 1
    assert f(FAKE, FAKE, 256, 128, 512, FAKE, ctypes.byref(s), FAKE, wsb - 1, None) == 1
    assert f(FAKE, FAKE_MIS, 256, 128, 512, FAKE, ctypes.byref(s), FAKE, wsb, None) == 2
    assert f(FAKE, FAKE, 256, 128, 512, FAKE, None, FAKE, wsb, None) == 1
