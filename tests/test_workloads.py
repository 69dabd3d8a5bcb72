"""The seeded input recipe (no GPU): shapes, seeds, distributions, and the
shared-input groups keep the workload's work and bytes."""
import numpy as np
import pytest
import torch

from float8_mixed_precision_gb300 import workloads as wl


def test_seeds_and_tiny_workload():
    assert wl.seed_of(1, 0, 0) == 0
    d = wl.linear_inputs(1, 0)
    assert d["x"].shape == (256, 256) and d["w"].shape == (512, 256) and d["dy"].shape == (256, 512)
    assert all(t.dtype == torch.bfloat16 for t in d.values())
    again = wl.linear_inputs(1, 0)
    assert all(torch.equal(d[k], again[k]) for k in d)


def test_flops_of_workloads():
    tot = {c: sum(l.flops for l in wl.workload(c)[1]) for c in wl.WORKLOADS}
    assert tot[1] == 6 * 256 * 256 * 512
    assert abs(tot[2] / 1e9 - 2061.6) < 0.1
    assert abs(tot[3] / 1e9 - 8658.7) < 0.1
    assert abs(tot[4] / 1e9 - 34634.7) < 0.1
    assert tot[5] == tot[2] + tot[3]


def test_distributions():
    x = wl.normal((200_000,), 0.02, 1).float()
    assert abs(x.std().item() - 0.02) < 5e-4
    h = wl.swiglu_input((100_000,), 3, 4).float()
    a = torch.randn(100_000, generator=torch.Generator().manual_seed(3))
    b = torch.randn(100_000, generator=torch.Generator().manual_seed(4))
    assert torch.equal(h, (torch.nn.functional.silu(a) * b).to(torch.bfloat16).float())
    t = wl.student_t_outliers((1000, 100), 3, 1e-3, 100.0, 5).float()
    n_big = int((t.abs() > 40).sum())
    assert 60 <= n_big <= 200         # ~100 entries scaled by 100, plus the t tail


@pytest.mark.parametrize("c", [2, 3, 5])
def test_fused_groups_keep_the_work(c):
    groups = wl.fused_groups(c)
    lins = wl.workload(c)[1]
    assert sum(g.flops for g, _ in groups) == sum(l.flops for l in lins)
    assert sorted(i for _, idx in groups for i in idx) == list(range(len(lins)))
    for g, idx in groups:
        assert all(lins[i].K == g.K and lins[i].M == g.M for i in idx)


def test_fused_group_inputs_are_concatenations():
    groups = wl.fused_groups(2)
    g, idx = groups[0]
    d = wl.fused_group_inputs(2, idx)
    parts = [wl.linear_inputs(2, i) for i in idx]
    assert torch.equal(d["x"], parts[0]["x"])
    assert torch.equal(d["w"][:4096], parts[0]["w"]) and torch.equal(d["w"][4096:5120], parts[1]["w"])
    assert torch.equal(d["dy"][:, 5120:], parts[2]["dy"])
