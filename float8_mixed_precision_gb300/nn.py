"""PyTorch modules over libf8: a Float8 linear layer for training.

The atlas.scime.ai summary of the TorchTitan paper (Approach) treats Float8
as a per-linear transformation composed onto a model, and its ablation
table measures it on Llama 3.1 8B.  This module is that transformation for
modules whose linears have no bias (as in Llama):

- Float8Linear: Y = X W^T with the forward and backward of a Float8 linear
  (f8_linear_fwd, f8_linear_bwd): dynamic tensorwise E4M3 scaling of X, W
  and dY, three FP8 GEMMs, bf16 outputs.  Autograd gets dX and dW from
  libf8; nothing of the layer's arithmetic runs in torch.
- Float8LinearGroup: linears that read one input (q, k, v; w1, w3), each
  its own Float8 linear, with X quantised once and shared GEMM launches
  (f8_linear_fwd_group, f8_linear_bwd_group).
- Float8SwiGLU: the Llama FFN with the w1+w3 GEMM's epilogue forming h
  and its amax, and the SwiGLU backward forming d(AB) with its amax.
- to_float8_linears: swaps eligible nn.Linear modules of a model for
  Float8Linear modules that share their weight Parameter.

Inputs and weights must be bf16 CUDA tensors with every size a multiple of
16 (the ABI's rule); anything else raises, there is no fallback path.
"""
from __future__ import annotations

from typing import Callable

import torch

from . import binding


class _Float8LinearFn(torch.autograd.Function):
    """One Float8 linear: forward saves q(X)^T, q(W)^T and their scalars
    (f8_linear_fwd); backward quantises dY and runs the dgrad and wgrad
    GEMMs (f8_linear_bwd)."""

    @staticmethod
    def forward(ctx, x: torch.Tensor, weight: torch.Tensor, dy_fmt: int) -> torch.Tensor:
        lead = x.shape[:-1]
        x2 = x.reshape(-1, x.shape[-1]).contiguous()
        y, saved = binding.f8_linear_fwd(x2, weight.contiguous())
        ctx.f8_saved = saved
        ctx.dy_fmt = dy_fmt
        ctx.x_shape = x.shape
        ctx.needs = (ctx.needs_input_grad[0], ctx.needs_input_grad[1])
        return y.reshape(*lead, weight.shape[0])

    @staticmethod
    def backward(ctx, dy: torch.Tensor):
        want_dx, want_dw = ctx.needs
        if not (want_dx or want_dw):
            return None, None, None
        dy2 = dy.reshape(-1, dy.shape[-1]).contiguous()
        dx, dw = binding.f8_linear_bwd(dy2, ctx.f8_saved, want_dx=want_dx, want_dw=want_dw,
                                       dy_fmt=ctx.dy_fmt)
        ctx.f8_saved = None
        return (dx.reshape(ctx.x_shape) if want_dx else None), (dw if want_dw else None), None


class _Float8GroupFn(torch.autograd.Function):
    """Linears that read one input: X quantised once, each W_i and dY_i with
    its own scale (f8_linear_fwd_group, f8_linear_bwd_group); dX is the sum
    of the members' dX_i, as autograd would form it for separate layers."""

    @staticmethod
    def forward(ctx, x: torch.Tensor, *weights: torch.Tensor):
        lead = x.shape[:-1]
        x2 = x.reshape(-1, x.shape[-1]).contiguous()
        ys, saved = binding.f8_linear_fwd_group(x2, [w.contiguous() for w in weights])
        ctx.f8_saved = saved
        ctx.x_shape = x.shape
        ctx.needs = tuple(ctx.needs_input_grad)
        return tuple(y.reshape(*lead, y.shape[-1]) for y in ys)

    @staticmethod
    def backward(ctx, *dys: torch.Tensor):
        want_dx, want_dw = ctx.needs[0], any(ctx.needs[1:])
        if not (want_dx or want_dw):
            return (None,) * len(ctx.needs)
        dys2 = [dy.reshape(-1, dy.shape[-1]).contiguous() for dy in dys]
        dxs, dws = binding.f8_linear_bwd_group(dys2, ctx.f8_saved, ctx.x_shape[-1],
                                               want_dx=want_dx, want_dw=want_dw)
        ctx.f8_saved = None
        dx = None
        if want_dx:
            dx = dxs[0]
            for d in dxs[1:]:
                dx = dx + d
            dx = dx.reshape(ctx.x_shape)
        dws = dws if want_dw else [None] * (len(ctx.needs) - 1)
        return (dx, *[dw if need else None for dw, need in zip(dws, ctx.needs[1:])])


class _Float8LinearQWFn(torch.autograd.Function):
    """The linear on a weight quantised earlier (f8_linear_fwd_qw: only X is
    quantised here), then f8_linear_bwd as usual."""

    @staticmethod
    def forward(ctx, x: torch.Tensor, weight: torch.Tensor, w_q: torch.Tensor, w_t: torch.Tensor,
                w_scalars: torch.Tensor, dy_fmt: int) -> torch.Tensor:
        lead, K = x.shape[:-1], x.shape[-1]
        x2 = x.reshape(-1, K).contiguous()
        M = x2.shape[0]
        # W's amax and scale sit in w_scalars[2:4]; X's go to a buffer of
        # this call's own
        saved = binding.LinearSaved(torch.empty((K, M), dtype=torch.uint8, device=x.device), w_t,
                                    w_scalars, torch.empty(2, dtype=torch.float32, device=x.device))
        y = binding.f8_linear_fwd_qw(x2, w_q, saved)
        ctx.f8_saved = saved
        ctx.dy_fmt = dy_fmt
        ctx.x_shape = x.shape
        ctx.needs = (ctx.needs_input_grad[0], ctx.needs_input_grad[1])
        return y.reshape(*lead, w_q.shape[0])

    @staticmethod
    def backward(ctx, dy: torch.Tensor):
        dx, dw, _ = _Float8LinearFn.backward(ctx, dy)
        return dx, dw, None, None, None, None


def _grad_format(name: str) -> int:
    """The FP8 format of dY: "e4m3" (scale 448/amax) or "e5m2" (scale
    57344/amax, the wider-range gradient format of the FP8 formats paper)."""
    formats = {"e4m3": binding.F8_E4M3, "e5m2": binding.F8_E5M2}
    if name not in formats:
        raise ValueError("grad_format is 'e4m3' or 'e5m2'")
    return formats[name]


def _check_sizes(in_features: int, out_features: int) -> None:
    if in_features % 16 or out_features % 16:
        raise ValueError("Float8Linear needs in_features and out_features that are multiples of 16")


class Float8Linear(torch.nn.Module):
    """A bias-free linear layer, y = x W^T, computed by the Float8 path.

    `weight` is [out_features, in_features] bf16, as in nn.Linear.  The
    input's last dimension is in_features; its other dimensions are
    flattened into the GEMM's M, which must be a multiple of 16."""

    def __init__(self, in_features: int, out_features: int, device=None,
                 weight: torch.nn.Parameter | None = None, grad_format: str = "e4m3",
                 cache_weight: bool = False):
        super().__init__()
        _check_sizes(in_features, out_features)
        self.in_features = in_features
        self.out_features = out_features
        self.grad_format = _grad_format(grad_format)
        # cache_weight: q(W), q(W)^T and W's scalars are kept and reused
        # while the weight's storage and version are unchanged (e.g. across
        # the micro-batches of one optimiser step); an in-place update of
        # the weight bumps its version and the next forward quantises again
        self.cache_weight = cache_weight
        self._wcache = None
        if weight is None:
            weight = torch.nn.Parameter(torch.empty((out_features, in_features),
                                                    dtype=torch.bfloat16, device=device))
            torch.nn.init.normal_(weight, std=0.02)
        if tuple(weight.shape) != (out_features, in_features) or weight.dtype != torch.bfloat16:
            raise TypeError("Float8Linear's weight is a bf16 [out_features, in_features] tensor")
        self.weight = weight

    @classmethod
    def from_linear(cls, linear: torch.nn.Linear, grad_format: str = "e4m3",
                    cache_weight: bool = False) -> "Float8Linear":
        """The Float8 counterpart of `linear`, sharing its weight Parameter."""
        if linear.bias is not None:
            raise ValueError("Float8Linear has no bias")
        return cls(linear.in_features, linear.out_features, weight=linear.weight,
                   grad_format=grad_format, cache_weight=cache_weight)

    def quantized_weight(self):
        """(q(W) [out, in], q(W)^T [in, out], scalars [4] with W's amax and
        scale at [2:4]) for the weight as it is now: f8_quantize once per
        weight version, then the cached tensors."""
        w = self.weight
        key = (w.data_ptr(), w._version)
        if self._wcache is None or self._wcache[0] != key:
            scalars = torch.zeros(4, dtype=torch.float32, device=w.device)
            q, qt, _, _ = binding.f8_quantize(w.detach(), scalars[2:3], scalars[3:4])
            self._wcache = (key, q, qt, scalars)
        return self._wcache[1:]

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        if x.dtype != torch.bfloat16:
            raise TypeError("Float8Linear takes bf16 inputs")
        if x.shape[-1] != self.in_features:
            raise ValueError("the input's last dimension is not in_features")
        if (x.numel() // self.in_features) % 16:
            raise ValueError("Float8Linear needs a token count (the input's leading dimensions) "
                             "that is a multiple of 16")
        if self.cache_weight:
            w_q, w_t, w_scalars = self.quantized_weight()
            return _Float8LinearQWFn.apply(x, self.weight, w_q, w_t, w_scalars, self.grad_format)
        return _Float8LinearFn.apply(x, self.weight, self.grad_format)

    def extra_repr(self) -> str:
        grads = "e5m2" if self.grad_format == binding.F8_E5M2 else "e4m3"
        return (f"in_features={self.in_features}, out_features={self.out_features}, "
                f"float8=e4m3, gradients={grads}")


class Float8LinearGroup(torch.nn.Module):
    """Bias-free linears that read the same input, such as the q, k and v
    projections of attention or w1 and w3 of a SwiGLU FFN: forward returns
    one output per member.  Each member stays a Float8 linear with its own
    weight and gradient scales; X is quantised once, and the members' GEMMs
    share launches where the tile schedule gains.  Outputs and weight
    gradients equal separate Float8Linear layers' bit for bit; dX is the sum
    of the members' dX in member order.  At most four members."""

    def __init__(self, in_features: int, out_features: list[int], device=None,
                 weights: list[torch.nn.Parameter] | None = None):
        super().__init__()
        if not 1 <= len(out_features) <= binding.F8_MAX_GROUP_LINEARS:
            raise ValueError(f"a group has 1 to {binding.F8_MAX_GROUP_LINEARS} members")
        for n in out_features:
            _check_sizes(in_features, n)
        self.in_features = in_features
        self.out_features = list(out_features)
        if weights is None:
            weights = []
            for n in out_features:
                w = torch.nn.Parameter(torch.empty((n, in_features), dtype=torch.bfloat16,
                                                   device=device))
                torch.nn.init.normal_(w, std=0.02)
                weights.append(w)
        for w, n in zip(weights, out_features):
            if tuple(w.shape) != (n, in_features) or w.dtype != torch.bfloat16:
                raise TypeError("each weight is a bf16 [out_features, in_features] tensor")
        self.weights = torch.nn.ParameterList(weights)

    @classmethod
    def from_linears(cls, linears: list[torch.nn.Linear]) -> "Float8LinearGroup":
        """The group of `linears` (same in_features, no bias), sharing their
        weight Parameters."""
        if any(l.bias is not None for l in linears):
            raise ValueError("Float8LinearGroup has no bias")
        if len({l.in_features for l in linears}) != 1:
            raise ValueError("the members of a group read the same input")
        return cls(linears[0].in_features, [l.out_features for l in linears],
                   weights=[l.weight for l in linears])

    def forward(self, x: torch.Tensor) -> tuple[torch.Tensor, ...]:
        if x.dtype != torch.bfloat16:
            raise TypeError("Float8LinearGroup takes bf16 inputs")
        if x.shape[-1] != self.in_features:
            raise ValueError("the input's last dimension is not in_features")
        if (x.numel() // self.in_features) % 16:
            raise ValueError("Float8LinearGroup needs a token count that is a multiple of 16")
        return _Float8GroupFn.apply(x, *self.weights)

    def extra_repr(self) -> str:
        return f"in_features={self.in_features}, out_features={self.out_features}, float8=e4m3"


def interleave_w13(w1: torch.Tensor, w3: torch.Tensor) -> torch.Tensor:
    """W13 [2F, D] from W1 and W3 [F, D]: blocks of 128 rows taken from W1
    and W3 alternately, the layout whose 256-column output tiles hold 128
    columns of a = X W1^T next to the matching 128 of b = X W3^T."""
    if w1.shape != w3.shape or w1.shape[0] % 128:
        raise ValueError("W1 and W3 are [F, D] with F a multiple of 128")
    F, D = w1.shape
    return torch.stack([w1.reshape(F // 128, 128, D), w3.reshape(F // 128, 128, D)],
                       dim=1).reshape(2 * F, D)


class _Float8SwiGLUFn(torch.autograd.Function):
    """y = W2 h with h = silu(X W1^T) * (X W3^T), the Llama FFN:
    forward f8_linear_fwd_w13_swiglu (the w1+w3 group as one Float8 linear
    whose GEMM epilogue writes a, b, h and max|h|, then the cast of h), W2's
    quantisation and the w2 GEMM on q(h); backward f8_linear_bwd (dh and dW2)
    then f8_linear_bwd_w13_swiglu (d(AB) with its amax from dh, a and b,
    then dX and dW13)."""

    @staticmethod
    def forward(ctx, x: torch.Tensor, w13: torch.Tensor, w2: torch.Tensor) -> torch.Tensor:
        lead, D = x.shape[:-1], x.shape[-1]
        x2 = x.reshape(-1, D).contiguous()
        M, F = x2.shape[0], w2.shape[1]
        s2 = binding.LinearSaved.empty(M, D, F, x.device)   # w2: X part = h
        ab, _, s13, h_q, _, _, _ = binding.f8_linear_fwd_w13_swiglu(
            x2, w13.contiguous(), amax_h=s2.scalars[0:1], scale_h=s2.scalars[1:2], h_t=s2.x_t)
        w2q, _, _, _ = binding.f8_quantize(w2.contiguous(), s2.scalars[2:3], s2.scalars[3:4],
                                           q_t=s2.w_t)
        y = binding.f8_gemm(h_q, w2q, s2.scalars[1:2], s2.scalars[3:4])
        ctx.f8 = (ab, s13, s2)
        ctx.x_shape = x.shape
        return y.reshape(*lead, D)

    @staticmethod
    def backward(ctx, dy: torch.Tensor):
        ab, s13, s2 = ctx.f8
        ctx.f8 = None
        dh, dw2 = binding.f8_linear_bwd(dy.reshape(-1, dy.shape[-1]).contiguous(), s2)
        dx, dw13, _ = binding.f8_linear_bwd_w13_swiglu(dh, ab, s13)
        return dx.reshape(ctx.x_shape), dw13, dw2


class Float8SwiGLU(torch.nn.Module):
    """The SwiGLU FFN of a Llama block, y = W2 (silu(W1 x) * (W3 x)), with
    every GEMM a Float8 one and the SiLU, the product and the amax of h in
    the epilogue of the w1+w3 GEMM (the amax-with-the-producer row).  The
    w1+w3 group is one Float8 linear (one scale over W13); w2 is a Float8
    linear of its own.  Its parameters are `w13` [2F, D], W1 and W3
    interleaved by 128 rows (interleave_w13), and `w2` [D, F]; F a multiple
    of 128, D of 16, and the token count of 16."""

    def __init__(self, dim: int, hidden: int, device=None, w13: torch.nn.Parameter | None = None,
                 w2: torch.nn.Parameter | None = None):
        super().__init__()
        if hidden % 128 or dim % 16:
            raise ValueError("Float8SwiGLU needs hidden % 128 == 0 and dim % 16 == 0")
        self.dim, self.hidden = dim, hidden
        if w13 is None:
            w13 = torch.nn.Parameter(torch.empty((2 * hidden, dim), dtype=torch.bfloat16,
                                                 device=device))
            torch.nn.init.normal_(w13, std=0.02)
        if w2 is None:
            w2 = torch.nn.Parameter(torch.empty((dim, hidden), dtype=torch.bfloat16, device=device))
            torch.nn.init.normal_(w2, std=0.02)
        if tuple(w13.shape) != (2 * hidden, dim) or tuple(w2.shape) != (dim, hidden) or \
                w13.dtype != torch.bfloat16 or w2.dtype != torch.bfloat16:
            raise TypeError("w13 is bf16 [2 hidden, dim] and w2 bf16 [dim, hidden]")
        self.w13, self.w2 = w13, w2

    @classmethod
    def from_linears(cls, w1: torch.nn.Linear, w3: torch.nn.Linear,
                     w2: torch.nn.Linear) -> "Float8SwiGLU":
        """From a model's three FFN linears: w2's weight Parameter is shared,
        W13 is a new Parameter holding W1 and W3 interleaved."""
        if any(l.bias is not None for l in (w1, w3, w2)):
            raise ValueError("Float8SwiGLU has no biases")
        w13 = torch.nn.Parameter(interleave_w13(w1.weight.detach(), w3.weight.detach()))
        return cls(w1.in_features, w1.out_features, w13=w13, w2=w2.weight)

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        if x.dtype != torch.bfloat16:
            raise TypeError("Float8SwiGLU takes bf16 inputs")
        if x.shape[-1] != self.dim:
            raise ValueError("the input's last dimension is not dim")
        if (x.numel() // self.dim) % 16:
            raise ValueError("Float8SwiGLU needs a token count that is a multiple of 16")
        return _Float8SwiGLUFn.apply(x, self.w13, self.w2)

    def extra_repr(self) -> str:
        return f"dim={self.dim}, hidden={self.hidden}, float8=e4m3"


def eligible(linear: torch.nn.Module) -> bool:
    """An nn.Linear Float8Linear can stand in for: no bias, a bf16 weight,
    both sizes multiples of 16."""
    return (isinstance(linear, torch.nn.Linear) and linear.bias is None
            and linear.weight.dtype == torch.bfloat16
            and linear.in_features % 16 == 0 and linear.out_features % 16 == 0)


def to_float8_linears(module: torch.nn.Module,
                      keep: Callable[[str, torch.nn.Module], bool] | None = None,
                      grad_format: str = "e4m3", cache_weights: bool = False) -> torch.nn.Module:
    """Replaces, in place, every eligible nn.Linear below `module` for which
    `keep(qualified_name, linear)` is true (all of them when `keep` is None)
    with a Float8Linear sharing its weight Parameter (dY in `grad_format`;
    `cache_weights` as Float8Linear's cache_weight); returns `module`."""
    def visit(parent: torch.nn.Module, prefix: str) -> None:
        for name, child in list(parent.named_children()):
            qual = f"{prefix}.{name}" if prefix else name
            if eligible(child) and (keep is None or keep(qual, child)):
                setattr(parent, name, Float8Linear.from_linear(child, grad_format, cache_weights))
            else:
                visit(child, qual)

    if eligible(module) and (keep is None or keep("", module)):
        raise ValueError("the module itself is a linear: use Float8Linear.from_linear")
    visit(module, "")
    return module
