"""Seeded synthetic inputs for the Float8 training linear.

This module holds only shapes, distributions and random draws.  It contains
none of the method's arithmetic (no amax, scale, cast or GEMM), so that the
CUDA path and the CPU oracle can both be fed from it without sharing any of
the computation under test.

Every tensor is drawn in fp32 on the CPU from ``torch.Generator().manual_seed``
and rounded to bf16 with torch's round-to-nearest-even conversion; callers
receive the same bytes whichever side they feed.

Workloads (Llama 3.1 shapes; M = sequence 8192 x local batch 1, as in the
torchtitan walkthrough's llama3_8b training run):
  1 tiny     X [256,256] ~N(0,1), W [512,256] ~N(0,0.02), dY [256,512] ~N(0,1)
  2 attn8b   wq, wo 4096->4096 and wk, wv 4096->1024; X ~N(0,1), W ~N(0,0.02),
             dY ~N(0,0.01)
  3 ffn8b    w1, w3 4096->14336, w2 14336->4096; X ~N(0,1) (RMSNorm output),
             the w2 input is silu(a)*b with a, b ~N(0,1); W ~N(0,0.02);
             dY ~N(0,0.01)
  4 ffn70b   w1, w3 8192->28672, w2 28672->8192; activations ~N(0,1),
             weights ~N(0,0.02), dY ~N(0,0.01)
  5 block8b  the 7 linears of 2 and 3 with outlier activations: X, dY and
             the w2 input are Student-t(nu=3) with 0.1% of the entries
             (uniform, without replacement) multiplied by 100; W ~N(0,0.02)
The second parameter of N(mu, sigma) is the standard deviation.
Shared inputs (fused_groups): q, k, v read one X, as do w1 and w3; merging
each group into one linear with the concatenated weight leaves the work
unchanged and quantises the shared X once.
Seed of tensor t (X=0, W=1, dY=2, a=3, b=4) of linear l in workload c:
1000*(c-1) + 10*l + t, so workload 1 starts from seed 0.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

SEQ = 8192  # tokens per micro-batch: seq 8192 x local batch 1


@dataclass(frozen=True)
class Linear:
    name: str
    M: int  # tokens
    K: int  # in-features
    N: int  # out-features
    x_kind: str = "normal"   # "normal" | "swiglu" | "student_t"
    dy_kind: str = "normal"  # "normal" | "student_t"
    x_std: float = 1.0
    w_std: float = 0.02
    dy_std: float = 0.01

    @property
    def flops(self) -> int:
        """fwd + dgrad + wgrad: three GEMMs of 2*M*N*K each."""
        return 6 * self.M * self.N * self.K


def _attn(M, kind="normal", dy_kind="normal"):
    return [Linear("wq", M, 4096, 4096, kind, dy_kind), Linear("wk", M, 4096, 1024, kind, dy_kind),
            Linear("wv", M, 4096, 1024, kind, dy_kind), Linear("wo", M, 4096, 4096, kind, dy_kind)]


def _ffn(M, d, h, kind="normal", w2_kind="swiglu", dy_kind="normal"):
    return [Linear("w1", M, d, h, kind, dy_kind), Linear("w3", M, d, h, kind, dy_kind),
            Linear("w2", M, h, d, w2_kind, dy_kind)]


WORKLOADS = {
    1: ("tiny", [Linear("tiny", 256, 256, 512, dy_std=1.0)]),
    2: ("llama3.1-8b-attention-proj", _attn(SEQ)),
    3: ("llama3.1-8b-swiglu-ffn", _ffn(SEQ, 4096, 14336)),
    4: ("llama3.1-70b-shape-ffn", _ffn(SEQ, 8192, 28672, w2_kind="normal")),
    5: ("llama3.1-8b-block-outliers",
        _attn(SEQ, "student_t", "student_t")
        + _ffn(SEQ, 4096, 14336, "student_t", "student_t", "student_t")),
}


def workload(c: int) -> tuple[str, list[Linear]]:
    return WORKLOADS[c]


def seed_of(c: int, l: int, t: int) -> int:
    return 1000 * (c - 1) + 10 * l + t


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(seed)
    return g


def normal(shape, std: float, seed: int) -> torch.Tensor:
    """bf16 tensor of N(0, std^2) draws."""
    x = torch.randn(shape, generator=_gen(seed), dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def swiglu_input(shape, seed_a: int, seed_b: int) -> torch.Tensor:
    """bf16(silu(a) * b) with a, b ~N(0,1), evaluated in fp32."""
    a = torch.randn(shape, generator=_gen(seed_a), dtype=torch.float32)
    b = torch.randn(shape, generator=_gen(seed_b), dtype=torch.float32)
    return (torch.nn.functional.silu(a) * b).to(torch.bfloat16)


def student_t_outliers(shape, nu: int, frac: float, factor: float, seed: int) -> torch.Tensor:
    """Student-t(nu) draws (z / sqrt(chi2_nu / nu)); a fraction ``frac`` of
    the entries, chosen uniformly without replacement, multiplied by ``factor``."""
    g = _gen(seed)
    n = math.prod(shape)
    z = torch.randn(n, generator=g, dtype=torch.float32)
    chi2 = torch.zeros(n, dtype=torch.float32)
    for _ in range(nu):
        e = torch.randn(n, generator=g, dtype=torch.float32)
        chi2.addcmul_(e, e)
    t = z / torch.sqrt(chi2 / nu)
    k = int(round(frac * n))
    if k:
        idx = torch.randperm(n, generator=g)[:k]
        t[idx] *= factor
    return t.reshape(shape).to(torch.bfloat16)


def swiglu_ab(c: int, l: int) -> tuple[torch.Tensor, torch.Tensor]:
    """The a and b (bf16) whose silu(a) * b is the input of linear l of
    workload c, for linears with x_kind "swiglu"."""
    lin = WORKLOADS[c][1][l]
    shape = (lin.M, lin.K)
    a = torch.randn(shape, generator=_gen(seed_of(c, l, 3)), dtype=torch.float32)
    b = torch.randn(shape, generator=_gen(seed_of(c, l, 4)), dtype=torch.float32)
    return a.to(torch.bfloat16), b.to(torch.bfloat16)


def _activation(kind: str, shape, std: float, c: int, l: int, t: int) -> torch.Tensor:
    if kind == "normal":
        return normal(shape, std, seed_of(c, l, t))
    if kind == "student_t":
        return student_t_outliers(shape, 3, 1e-3, 100.0, seed_of(c, l, t))
    if kind == "swiglu":
        return swiglu_input(shape, seed_of(c, l, 3), seed_of(c, l, 4))
    raise ValueError(kind)


def linear_inputs(c: int, l: int, lin: Linear | None = None) -> dict[str, torch.Tensor]:
    """X [M,K], W [N,K], dY [M,N] (bf16, CPU) of linear ``l`` of workload ``c``."""
    if lin is None:
        lin = WORKLOADS[c][1][l]
    x = _activation(lin.x_kind, (lin.M, lin.K), lin.x_std, c, l, 0)
    w = normal((lin.N, lin.K), lin.w_std, seed_of(c, l, 1))
    dy = _activation(lin.dy_kind, (lin.M, lin.N), lin.dy_std, c, l, 2)
    return {"x": x, "w": w, "dy": dy}


# Linears of a workload that read the same input in a Llama block: q, k and v
# read the attention-norm output, w1 and w3 the FFN-norm output.
SHARED_INPUT_GROUPS = {2: [["wq", "wk", "wv"], ["wo"]],
                       3: [["w1", "w3"], ["w2"]],
                       4: [["w1", "w3"], ["w2"]],
                       5: [["wq", "wk", "wv"], ["wo"], ["w1", "w3"], ["w2"]]}


def fused_groups(c: int) -> list[tuple[Linear, list[int]]]:
    """Workload ``c`` with the linears that share an input merged into one
    linear with the concatenated weight [sum N_i, K] (same total work): each
    entry is (merged Linear, indices of the member linears)."""
    lins = WORKLOADS[c][1]
    by_name = {l.name: i for i, l in enumerate(lins)}
    out = []
    for names in SHARED_INPUT_GROUPS[c]:
        idx = [by_name[n] for n in names]
        first = lins[idx[0]]
        out.append((Linear("+".join(names), first.M, first.K, sum(lins[i].N for i in idx),
                           first.x_kind, first.dy_kind, first.x_std, first.w_std, first.dy_std), idx))
    return out


def fused_group_inputs(c: int, idx: list[int]) -> dict[str, torch.Tensor]:
    """X of the group's first linear (the shared input), the members' W
    stacked along N, and their dY concatenated along N."""
    parts = [linear_inputs(c, i) for i in idx]
    return {"x": parts[0]["x"], "w": torch.cat([p["w"] for p in parts], 0),
            "dy": torch.cat([p["dy"] for p in parts], 1)}


def interleave_128(t1: torch.Tensor, t3: torch.Tensor, dim: int) -> torch.Tensor:
    """Blocks of 128 along `dim` taken from t1 and t3 alternately (the row
    order of W13, and the column order of AB and its gradient): a copy, no
    arithmetic."""
    n = t1.shape[dim]
    assert t3.shape == t1.shape and n % 128 == 0
    a = t1.unflatten(dim, (n // 128, 128))
    b = t3.unflatten(dim, (n // 128, 128))
    return torch.stack((a, b), dim=dim + 1).flatten(dim, dim + 2)


def w13_group_inputs(c: int, idx: list[int]) -> dict[str, torch.Tensor]:
    """The group {w1, w3} of workload c for the SwiGLU-epilogue linear: X of
    w1, W13 with W1 and W3 rows interleaved by 128, and the group's dY
    [M, 2F] with dY1 and dY3 columns interleaved the same way."""
    p1, p3 = linear_inputs(c, idx[0]), linear_inputs(c, idx[1])
    return {"x": p1["x"], "w": interleave_128(p1["w"], p3["w"], 0),
            "dy": interleave_128(p1["dy"], p3["dy"], 1)}


def custom_linear(M: int, K: int, N: int, seed: int, x_std=1.0, w_std=0.02, dy_std=1.0):
    """Inputs for an arbitrary (M, K, N), e.g. ragged parity cases."""
    return {"x": normal((M, K), x_std, seed), "w": normal((N, K), w_std, seed + 1),
            "dy": normal((M, N), dy_std, seed + 2)}


def bits(t: torch.Tensor):
    """uint16 bit patterns of a bf16 CPU tensor, as a numpy array (a view)."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view("uint16")
