"""FP8 all-gather of a row-sharded weight, as FSDP2's Float8 all-gather does
it (discuss.pytorch.org torchtitan index, topic "[Distributed w/ Torchtitan]
Enabling Float8 All-Gather in FSDP2": float8 saves network bandwidth with a
reduced message size).

Rank r of R holds rows [r N/R, (r+1) N/R) of W [N, K] (bf16).  Dynamic
tensorwise scaling needs one scale for the whole W, so the gather is:

  1. amax of the local shard                                  (device)
  2. all-reduce(MAX) of that one fp32 over the ranks           (collective)
  3. scale = fmax / max(amax, 1e-12); the shard cast to E4M3   (device)
  4. all-gather of the shard's E4M3 bytes into q(W) [N, K]     (collective)
  5. q(W)^T [K, N] from the gathered q(W), for the dgrad GEMM  (device)

The gathered q(W) equals the quantisation of the whole W (the same amax, so
the same scale and the same per-element cast), at 1 byte per element on the
wire instead of bf16's 2.  f8_linear_fwd_qw then runs the linear on it.

This module holds the protocol only.  The device steps come from `ops`
(default: libf8's kernels through the binding); the collectives are
torch.distributed's, on whatever process group the caller passes (NCCL on
GPUs).  A test may pass other ops (it runs the protocol on CPU gloo ranks).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable


@dataclass
class GatherOps:
    """The device steps of the gather: amax(shard) -> fp32 scalar tensor;
    cast(shard, amax) -> (q_shard [n, K] uint8, scale fp32 scalar tensor)
    using that amax; transpose(q [N, K]) -> q^T [K, N]."""
    amax: Callable
    cast: Callable
    transpose: Callable


def libf8_ops() -> GatherOps:
    """The gather's device steps on libf8's kernels (f8_amax,
    f8_cast_transpose with the gathered amax, f8_transpose_u8)."""
    from . import binding

    def cast(shard, amax):
        q, _, scale = binding.f8_cast_transpose(shard, amax, want_t=False)
        return q, scale

    return GatherOps(amax=binding.f8_amax, cast=cast, transpose=binding.f8_transpose_u8)


def fp8_all_gather_weight(w_shard, group=None, ops: GatherOps | None = None):
    """Steps 1-5 above for this rank's shard w_shard [N / R, K] (bf16; every
    rank's shard of the same shape).  Returns (q_w [N, K], q_w_t [K, N],
    amax, scale): the whole weight's E4M3 copies and its scalars, the same
    on every rank."""
    import torch
    import torch.distributed as dist

    ops = ops or libf8_ops()
    world = dist.get_world_size(group)
    amax = ops.amax(w_shard).reshape(1).clone()
    dist.all_reduce(amax, op=dist.ReduceOp.MAX, group=group)
    q_shard, scale = ops.cast(w_shard, amax.reshape(()))
    n, K = q_shard.shape
    q_w = torch.empty((world * n, K), dtype=torch.uint8, device=q_shard.device)
    dist.all_gather_into_tensor(q_w, q_shard.contiguous(), group=group)
    q_w_t = ops.transpose(q_w)
    return q_w, q_w_t, amax.reshape(()), scale


def gathered_saved(q_w_t, amax, scale, M: int):
    """A LinearSaved for f8_linear_fwd_qw / f8_linear_bwd whose weight part
    is the gathered q(W)^T and scalars (the X part is filled by the forward)."""
    import torch

    from .binding import LinearSaved
    K, N = q_w_t.shape
    dev = q_w_t.device
    scalars = torch.empty(4, dtype=torch.float32, device=dev)
    scalars[2] = amax
    scalars[3] = scale
    return LinearSaved(torch.empty((K, M), dtype=torch.uint8, device=dev), q_w_t, scalars)
