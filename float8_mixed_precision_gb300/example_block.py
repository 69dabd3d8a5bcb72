"""Example: the linears of one Llama-3.1-8B block trained through
float8_mixed_precision_gb300.nn, timed eager and as a captured CUDA graph.

    python -m float8_mixed_precision_gb300.example_block [--steps 20]

The block's linears at M = 8192 tokens: q, k, v as one Float8LinearGroup
(X quantised once, a scale per weight), wo as a Float8Linear, and the SwiGLU
FFN as a Float8SwiGLU on the fused path (h and its amax from the w1+w3
GEMM's epilogue, the SwiGLU backward with its amax).  Attention and the
norms are not part of the example: each module gets its own random bf16
input and output gradient, and a step is every module's forward and
backward.  TFLOP/s counts 6 M N K per linear, as the benchmark does.
"""
from __future__ import annotations

import argparse

import torch

from . import binding
from . import nn as f8nn


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--steps", type=int, default=20)
    args = ap.parse_args(argv)
    dev = torch.device("cuda", 0)
    M, D, F = 8192, 4096, 14336
    gen = torch.Generator(device=dev).manual_seed(0)

    def rnd(shape, std):
        return (torch.randn(shape, generator=gen, device=dev) * std).to(torch.bfloat16)

    qkv = f8nn.Float8LinearGroup(D, [4096, 1024, 1024], device=dev)
    wo = f8nn.Float8Linear(D, D, device=dev)
    ffn = f8nn.Float8SwiGLU(D, F, device=dev)
    xs = [rnd((M, D), 1.0).requires_grad_(True) for _ in range(3)]
    grads = [rnd((M, 4096), 0.01), rnd((M, 1024), 0.01), rnd((M, 1024), 0.01),
             rnd((M, D), 0.01), rnd((M, D), 0.01)]
    params = list(qkv.parameters()) + list(wo.parameters()) + list(ffn.parameters()) + xs
    flops = 6 * M * D * (4096 + 2 * 1024) + 6 * M * D * D + 3 * 6 * M * D * F

    def forward_backward():
        q, k, v = qkv(xs[0])
        o = wo(xs[1])
        y = ffn(xs[2])
        torch.autograd.backward([q, k, v, o, y], grads)

    def step():
        for p in params:
            p.grad = None
        forward_backward()

    def timed(fn):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.steps):
            fn()
        b.record()
        b.synchronize()
        return a.elapsed_time(b) / args.steps

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    ms = timed(step)
    print(f"eager autograd: {ms:.3f} ms per step, {flops / ms / 1e9:,.0f} TFLOP/s")

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            step()
    torch.cuda.current_stream().wait_stream(side)
    for p in params:
        p.grad = None
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        forward_backward()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    ms = timed(graph.replay)
    print(f"CUDA graph:     {ms:.3f} ms per step, {flops / ms / 1e9:,.0f} TFLOP/s")
    status = binding.f8_last_device_status()
    if status != 0:
        raise RuntimeError(binding.f8_status_string(status))


if __name__ == "__main__":
    main()
