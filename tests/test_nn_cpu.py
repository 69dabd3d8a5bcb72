"""float8_mixed_precision_gb300.nn without a GPU: which linears
to_float8_linears swaps, that the swapped modules share the original weight
Parameters, and that Float8Linear refuses what the ABI cannot take (wrong
dtype, sizes that are not multiples of 16, host tensors) instead of
computing anything in torch."""
import pytest
import torch

from float8_mixed_precision_gb300 import nn as f8nn


@pytest.fixture(scope="module", autouse=True)
def _built():
    from float8_mixed_precision_gb300 import build
    build.build()


def _lin(i, o, bias=False, dtype=torch.bfloat16):
    return torch.nn.Linear(i, o, bias=bias, dtype=dtype)


def _model():
    return torch.nn.ModuleDict({
        "attn": torch.nn.ModuleDict({"wq": _lin(64, 64), "wk": _lin(64, 16), "wo": _lin(64, 64)}),
        "ffn": torch.nn.Sequential(_lin(64, 128), torch.nn.SiLU(), _lin(128, 64)),
        "head": _lin(64, 100),                 # 100 is not a multiple of 16
        "proj": _lin(64, 64, bias=True),       # a bias
        "fp32": _lin(64, 64, dtype=torch.float32),
    })


def test_swaps_eligible_linears_sharing_weights():
    m = _model()
    before = {n: mod.weight for n, mod in m.named_modules() if isinstance(mod, torch.nn.Linear)}
    f8nn.to_float8_linears(m)
    swapped = {n for n, mod in m.named_modules() if isinstance(mod, f8nn.Float8Linear)}
    assert swapped == {"attn.wq", "attn.wk", "attn.wo", "ffn.0", "ffn.2"}
    for n in swapped:
        assert m.get_submodule(n).weight is before[n]
    for n in ("head", "proj", "fp32"):
        assert type(m.get_submodule(n)) is torch.nn.Linear
    assert sum(1 for _ in m.parameters()) == sum(1 for _ in _model().parameters())


def test_keep_filter():
    m = _model()
    f8nn.to_float8_linears(m, keep=lambda name, lin: name.startswith("ffn"))
    assert isinstance(m["ffn"][0], f8nn.Float8Linear) and isinstance(m["ffn"][2], f8nn.Float8Linear)
    assert type(m["attn"]["wq"]) is torch.nn.Linear


def test_refusals():
    with pytest.raises(ValueError):
        f8nn.Float8Linear(64, 100)
    with pytest.raises(ValueError):
        f8nn.Float8Linear.from_linear(_lin(64, 64, bias=True))
    with pytest.raises(ValueError):
        f8nn.to_float8_linears(_lin(64, 64))
    layer = f8nn.Float8Linear(64, 64)
    with pytest.raises(TypeError):
        layer(torch.zeros((16, 64), dtype=torch.float32))
    with pytest.raises(ValueError):
        layer(torch.zeros((15, 64), dtype=torch.bfloat16))       # 15 tokens
    with pytest.raises(ValueError):
        layer(torch.zeros((16, 48), dtype=torch.bfloat16))       # wrong in_features
    with pytest.raises(ValueError, match="device tensors"):
        layer(torch.zeros((2, 8, 64), dtype=torch.bfloat16))     # host tensors: no CPU path


def test_group_construction_and_refusals():
    lins = [_lin(64, 64), _lin(64, 16), _lin(64, 16)]
    g = f8nn.Float8LinearGroup.from_linears(lins)
    assert g.out_features == [64, 16, 16]
    assert all(w is l.weight for w, l in zip(g.weights, lins))
    with pytest.raises(ValueError):
        f8nn.Float8LinearGroup.from_linears([_lin(64, 64), _lin(32, 64)])
    with pytest.raises(ValueError):
        f8nn.Float8LinearGroup.from_linears([_lin(64, 64, bias=True)])
    with pytest.raises(ValueError):
        f8nn.Float8LinearGroup(64, [16] * 5)
    with pytest.raises(TypeError):
        g(torch.zeros((16, 64), dtype=torch.float32))
    with pytest.raises(ValueError, match="device tensors"):
        g(torch.zeros((16, 64), dtype=torch.bfloat16))


def test_interleave_w13_layout():
    F, D = 256, 32
    w1 = torch.arange(F * D, dtype=torch.float32).reshape(F, D)
    w3 = -w1
    w13 = f8nn.interleave_w13(w1, w3)
    assert w13.shape == (2 * F, D)
    for j in range(F // 128):
        assert torch.equal(w13[256 * j:256 * j + 128], w1[128 * j:128 * j + 128])
        assert torch.equal(w13[256 * j + 128:256 * j + 256], w3[128 * j:128 * j + 128])
    with pytest.raises(ValueError):
        f8nn.interleave_w13(w1[:100], w3[:100])


def test_swiglu_module_construction():
    w1, w3, w2 = _lin(64, 256), _lin(64, 256), _lin(256, 64)
    ffn = f8nn.Float8SwiGLU.from_linears(w1, w3, w2)
    assert ffn.w2 is w2.weight and ffn.w13.shape == (512, 64)
    with pytest.raises(ValueError):
        f8nn.Float8SwiGLU(64, 200)
    with pytest.raises(TypeError):
        ffn(torch.zeros((16, 64), dtype=torch.float32))
    with pytest.raises(ValueError, match="device tensors"):
        ffn(torch.zeros((16, 64), dtype=torch.bfloat16))


def test_grad_format_option():
    assert f8nn.Float8Linear(64, 64).grad_format == f8nn.binding.F8_E4M3
    assert f8nn.Float8Linear(64, 64, grad_format="e5m2").grad_format == f8nn.binding.F8_E5M2
    with pytest.raises(ValueError):
        f8nn.Float8Linear(64, 64, grad_format="fp16")
    m = _model()
    f8nn.to_float8_linears(m, grad_format="e5m2")
    assert m["attn"]["wq"].grad_format == f8nn.binding.F8_E5M2


def test_example_module_imports():
    import importlib
    mod = importlib.import_module("float8_mixed_precision_gb300.example_block")
    assert callable(mod.main)
