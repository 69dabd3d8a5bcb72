"""float8_mixed_precision_gb300.nn on the GPU: Float8Linear under autograd
gives exactly the outputs and gradients of the C-ABI calls it wraps, and a
model converted by to_float8_linears trains through libf8.

- One layer, input [2, 256, 512] -> 768: Y, dX and dW bit-identical to
  f8_linear_fwd / f8_linear_bwd on the flattened tensors, and Y within the
  GEMM bar of the oracle's linear.
- A two-linear SwiGLU-free MLP (x -> w1 -> silu -> w2) after conversion:
  the loss's gradients bit-identical to the same chain composed by hand
  from the C-ABI calls and torch's silu backward, with libf8 launching the
  backward's kernels (its launch counter grows during backward, which
  autograd runs on its own device thread).
- A layer whose input needs no gradient gets dW only (no dX GEMM).
- A converted model's training step captured in a CUDA graph and replayed
  gives the eager step's output and gradients.
"""
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


def _eq(a, b):
    return torch.equal(a.contiguous().view(torch.int16), b.contiguous().view(torch.int16))


def test_layer_matches_the_abi_calls(f8):
    from float8_mixed_precision_gb300 import nn as f8nn
    B, T, K, N = 2, 256, 512, 768
    d = wl.custom_linear(B * T, K, N, seed=81, dy_std=0.1)
    x = d["x"].to(DEV).reshape(B, T, K).requires_grad_(True)
    layer = f8nn.Float8Linear(K, N, weight=torch.nn.Parameter(d["w"].to(DEV)))
    g = d["dy"].to(DEV).reshape(B, T, N)
    y = layer(x)
    y.backward(g)
    assert f8.f8_last_device_status() == 0
    y_ref, saved = f8.f8_linear_fwd(d["x"].to(DEV), d["w"].to(DEV))
    dx_ref, dw_ref = f8.f8_linear_bwd(d["dy"].to(DEV), saved)
    assert y.shape == (B, T, N) and x.grad.shape == (B, T, K)
    assert _eq(y.reshape(-1, N), y_ref)
    assert _eq(x.grad.reshape(-1, K), dx_ref)
    assert _eq(layer.weight.grad, dw_ref)
    fwd = oracle.linear_fwd(wl.bits(d["x"]), wl.bits(d["w"]))
    check_close(y.reshape(-1, N), fwd["y"], what="Float8Linear Y")


def test_converted_mlp_gradients(f8):
    from float8_mixed_precision_gb300 import nn as f8nn
    M, D, H = 512, 256, 768
    torch.manual_seed(0)
    model = torch.nn.Sequential(
        torch.nn.Linear(D, H, bias=False, dtype=torch.bfloat16, device=DEV),
        torch.nn.SiLU(),
        torch.nn.Linear(H, D, bias=False, dtype=torch.bfloat16, device=DEV))
    with torch.no_grad():
        for lin in (model[0], model[2]):
            lin.weight.normal_(0.0, 0.02)
    w1, w2 = model[0].weight.detach().clone(), model[2].weight.detach().clone()
    f8nn.to_float8_linears(model)
    assert isinstance(model[0], f8nn.Float8Linear) and isinstance(model[2], f8nn.Float8Linear)
    x = wl.normal((M, D), 1.0, 82).to(DEV).requires_grad_(True)
    g = wl.normal((M, D), 0.05, 83).to(DEV)
    torch.cuda.synchronize()
    y = model(x)
    n0 = f8.f8_kernel_launches()
    (y * g).sum().backward()
    torch.cuda.synchronize()
    assert f8.f8_kernel_launches() > n0
    assert f8.f8_last_device_status() == 0
    # the same chain from the C-ABI calls
    a1, s1 = f8.f8_linear_fwd(x.detach(), w1)
    a1r = a1.clone().requires_grad_(True)
    h = torch.nn.functional.silu(a1r)
    y2, s2 = f8.f8_linear_fwd(h.detach(), w2)
    assert _eq(y, y2)
    dy2 = (g * torch.ones_like(y2)).to(torch.bfloat16)
    dh, dw2 = f8.f8_linear_bwd(dy2, s2)
    (da1,) = torch.autograd.grad(h, a1r, dh)
    dx, dw1 = f8.f8_linear_bwd(da1, s1)
    assert _eq(model[2].weight.grad, dw2)
    assert _eq(model[0].weight.grad, dw1)
    assert _eq(x.grad, dx)


def test_frozen_input_gets_weight_gradient_only(f8):
    from float8_mixed_precision_gb300 import nn as f8nn
    M, K, N = 256, 256, 512
    layer = f8nn.Float8Linear(K, N, device=DEV)
    x = wl.normal((M, K), 1.0, 84).to(DEV)               # requires no gradient
    y = layer(x)
    y.backward(wl.normal((M, N), 0.1, 85).to(DEV))
    assert f8.f8_last_device_status() == 0
    assert layer.weight.grad is not None and x.grad is None


def test_training_step_in_a_cuda_graph(f8):
    """A converted model's forward and backward captured once in a CUDA
    graph (torch.cuda.graph, static input and gradient buffers) and
    replayed: the output and the weight gradients of a replay equal an eager
    step's bit for bit."""
    from float8_mixed_precision_gb300 import nn as f8nn
    M, D, H = 256, 256, 512
    model = torch.nn.Sequential(
        torch.nn.Linear(D, H, bias=False, dtype=torch.bfloat16, device=DEV),
        torch.nn.SiLU(),
        torch.nn.Linear(H, D, bias=False, dtype=torch.bfloat16, device=DEV))
    with torch.no_grad():
        for lin in (model[0], model[2]):
            lin.weight.normal_(0.0, 0.02)
    f8nn.to_float8_linears(model)
    x = wl.normal((M, D), 1.0, 86).to(DEV)
    g = wl.normal((M, D), 0.05, 87).to(DEV)

    def step():
        for p in model.parameters():
            p.grad = None
        y = model(x)
        y.backward(g)
        return y

    y_eager = step().detach().clone()
    grads_eager = [p.grad.clone() for p in model.parameters()]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):                 # warm-up on the capture stream
            step()
    torch.cuda.current_stream().wait_stream(side)
    for p in model.parameters():
        p.grad = None
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        y_static = model(x)
        y_static.backward(g)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert f8.f8_last_device_status() == 0
    assert _eq(y_static, y_eager)
    for p, ge in zip(model.parameters(), grads_eager):
        assert _eq(p.grad, ge)


def test_group_matches_separate_layers(f8):
    """Float8LinearGroup over q, k, v-like members (512 -> 512, 128, 128),
    input [2, 128, 512]: each output and weight gradient bit-identical to
    f8_linear_fwd / f8_linear_bwd of that member, dX the member-order sum of
    the members' dX; a member whose output is unused gets a zero dY."""
    from float8_mixed_precision_gb300 import nn as f8nn
    B, T, K, Ns = 2, 128, 512, [512, 128, 128]
    x0 = wl.normal((B * T, K), 1.0, 91).to(DEV)
    ws = [wl.normal((n, K), 0.02, 92 + i).to(DEV) for i, n in enumerate(Ns)]
    gs = [wl.normal((B * T, n), 0.1, 96 + i).to(DEV) for i, n in enumerate(Ns)]
    group = f8nn.Float8LinearGroup(K, Ns, weights=[torch.nn.Parameter(w.clone()) for w in ws])
    x = x0.reshape(B, T, K).clone().requires_grad_(True)
    ys = group(x)
    torch.autograd.backward([ys[0], ys[1]], [gs[0].reshape(B, T, -1), gs[1].reshape(B, T, -1)])
    assert f8.f8_last_device_status() == 0
    dx_sum = None
    for i, (w, y) in enumerate(zip(ws, ys)):
        y_ref, saved = f8.f8_linear_fwd(x0, w)
        assert _eq(y.reshape(-1, Ns[i]), y_ref), i
        dy = gs[i] if i < 2 else torch.zeros_like(gs[i])
        dx_i, dw_i = f8.f8_linear_bwd(dy, saved)
        assert _eq(group.weights[i].grad, dw_i), i
        dx_sum = dx_i if dx_sum is None else dx_sum + dx_i
    assert _eq(x.grad.reshape(-1, K), dx_sum)


def test_swiglu_module(f8):
    """Float8SwiGLU (dim 512, hidden 1024, 2 x 128 tokens): output and the
    gradients of X, W13 and W2 bit-identical to the same chain of C-ABI
    calls (w1+w3 linear with the SwiGLU epilogue, W2 quantised, GEMM on
    q(h); f8_linear_bwd, then f8_linear_bwd_w13_swiglu); and the output near
    an fp32 evaluation of the FFN on the bf16 inputs (FP8 error, relative
    Frobenius below 0.12)."""
    from float8_mixed_precision_gb300 import nn as f8nn
    B, T, D, F = 2, 128, 512, 1024
    x0 = wl.normal((B * T, D), 1.0, 101).to(DEV)
    w1 = wl.normal((F, D), 0.02, 102).to(DEV)
    w3 = wl.normal((F, D), 0.02, 103).to(DEV)
    w2 = wl.normal((D, F), 0.02, 104).to(DEV)
    g = wl.normal((B * T, D), 0.1, 105).to(DEV)
    w13 = f8nn.interleave_w13(w1, w3)
    ffn = f8nn.Float8SwiGLU(D, F, w13=torch.nn.Parameter(w13.clone()),
                            w2=torch.nn.Parameter(w2.clone()))
    x = x0.reshape(B, T, D).clone().requires_grad_(True)
    y = ffn(x)
    y.backward(g.reshape(B, T, D))
    assert f8.f8_last_device_status() == 0
    # the chain by hand
    s2 = f8.LinearSaved.empty(B * T, D, F, DEV)
    ab, _, s13, h_q, _, _, _ = f8.f8_linear_fwd_w13_swiglu(
        x0, w13, amax_h=s2.scalars[0:1], scale_h=s2.scalars[1:2], h_t=s2.x_t)
    w2q, _, _, _ = f8.f8_quantize(w2, s2.scalars[2:3], s2.scalars[3:4], q_t=s2.w_t)
    y_ref = f8.f8_gemm(h_q, w2q, s2.scalars[1:2], s2.scalars[3:4])
    dh, dw2 = f8.f8_linear_bwd(g, s2)
    dx, dw13, _ = f8.f8_linear_bwd_w13_swiglu(dh, ab, s13)
    assert _eq(y.reshape(-1, D), y_ref)
    assert _eq(x.grad.reshape(-1, D), dx)
    assert _eq(ffn.w13.grad, dw13)
    assert _eq(ffn.w2.grad, dw2)
    ref = (torch.nn.functional.silu(x0.float() @ w1.float().t()) * (x0.float() @ w3.float().t())) \
        @ w2.float().t()
    rel = (y.reshape(-1, D).float() - ref).norm() / ref.norm()
    assert rel < 0.12, rel


def test_layer_with_e5m2_gradients(f8):
    """grad_format="e5m2": dY quantised to E5M2 (scale 57344/amax), dX and
    dW bit-identical to f8_linear_bwd with dy_fmt E5M2."""
    from float8_mixed_precision_gb300 import nn as f8nn
    M, K, N = 256, 512, 384
    d = wl.custom_linear(M, K, N, seed=111, dy_std=0.1)
    x = d["x"].to(DEV).requires_grad_(True)
    layer = f8nn.Float8Linear(K, N, weight=torch.nn.Parameter(d["w"].to(DEV)), grad_format="e5m2")
    layer(x).backward(d["dy"].to(DEV))
    assert f8.f8_last_device_status() == 0
    _, saved = f8.f8_linear_fwd(d["x"].to(DEV), d["w"].to(DEV))
    dx, dw = f8.f8_linear_bwd(d["dy"].to(DEV), saved, dy_fmt=f8.F8_E5M2)
    assert _eq(x.grad, dx) and _eq(layer.weight.grad, dw)
    _, saved4 = f8.f8_linear_fwd(d["x"].to(DEV), d["w"].to(DEV))
    dx4, _ = f8.f8_linear_bwd(d["dy"].to(DEV), saved4)
    assert not _eq(dx, dx4)          # the format really changed the gradient


def test_cached_weight_quantisation(f8):
    """cache_weight=True: two micro-batches (gradient accumulation) reuse
    one quantisation of W and give outputs, dX and the accumulated dW
    bit-identical to the layer without the cache; an in-place update of the
    weight (as an optimiser step makes) invalidates the cache, and the next
    forward matches the uncached layer on the updated weight."""
    from float8_mixed_precision_gb300 import nn as f8nn
    M, K, N = 512, 1024, 768
    w0 = wl.normal((N, K), 0.02, 121).to(DEV)
    cached = f8nn.Float8Linear(K, N, weight=torch.nn.Parameter(w0.clone()), cache_weight=True)
    plain = f8nn.Float8Linear(K, N, weight=torch.nn.Parameter(w0.clone()))
    xs = [wl.normal((M, K), 1.0, 122 + i).to(DEV) for i in range(2)]
    gs = [wl.normal((M, N), 0.1, 124 + i).to(DEV) for i in range(2)]
    keys = []
    for layer in (cached, plain):
        for x, g in zip(xs, gs):
            xr = x.clone().requires_grad_(True)
            y = layer(xr)
            y.backward(g)
            layer.__dict__.setdefault("_outs", []).append((y.detach(), xr.grad))
            if layer is cached:
                keys.append(layer._wcache[0])
    assert f8.f8_last_device_status() == 0
    assert keys[0] == keys[1]                          # one quantisation for both micro-batches
    for (yc, dxc), (yp, dxp) in zip(cached._outs, plain._outs):
        assert _eq(yc, yp) and _eq(dxc, dxp)
    assert _eq(cached.weight.grad, plain.weight.grad)
    with torch.no_grad():                              # the optimiser's in-place update
        for layer in (cached, plain):
            layer.weight.add_(layer.weight.grad, alpha=-0.01)
    y_c, y_p = cached(xs[0]), plain(xs[0])
    assert cached._wcache[0] != keys[0]
    assert f8.f8_last_device_status() == 0
    assert _eq(y_c, y_p)
