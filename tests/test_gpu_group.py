"""GPU parity of the grouped paths: several tensors quantised in one launch
pair, several GEMMs in shared launches, and linears that share their input.

- f8_quantize_multi: every tensor's amax, scale and both code layouts
  bit-exact against the oracle's quantize of that tensor (E4M3 and E5M2),
  and equal to f8_quantize on it; shapes that are not multiples of 128 take
  the per-tensor fallback with the same results.
- f8_gemm_grouped with up to eight problems: every output bit-identical to
  f8_gemm_fmt on its problem (same tiles, same K order), with one K extent
  (one class), two (the list schedule) and three or more (several launches),
  ragged M and N tails, both kernels, and a launch forced over problems the
  planner would keep apart (F8_GEMM_GROUP=2); small cases against the
  oracle within the GEMM bar.
- f8_linear_fwd_group / f8_linear_bwd_group: every output and saved tensor
  bit-identical to f8_linear_fwd / f8_linear_bwd on each member with the same
  X, and within the GEMM bar of the oracle's linear of each member; the
  Llama-3.1-8B q, k, v group at full size on sampled rows; the launch counts
  the planner promises (q, k, v forward: two quantisation launches and one
  GEMM launch).
"""
import os

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


def _bf(shape, std, seed):
    return wl.normal(shape, std, seed)


def _eq(a, b):
    return torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("shapes", [[(256, 384), (128, 128), (1024, 256)],
                                    [(128, 256)] * 8,
                                    [(256, 384), (130, 96)]])
def test_quantize_multi_bytes(f8, shapes, fmt):
    xs = [_bf(s, 1.0 + i, 100 + i) for i, s in enumerate(shapes)]
    xs[0][3, 5] = 300.0            # saturating outlier in one tensor only
    got = f8.f8_quantize_multi([x.to(DEV) for x in xs], fmt=fmt)
    assert f8.f8_last_device_status() == 0
    for x, (q, qt, sc, am) in zip(xs, got):
        ref = oracle.quantize(wl.bits(x), fmt)
        assert am.item() == float(ref["amax"]) and sc.item() == float(ref["scale"])
        assert np.array_equal(q.cpu().numpy(), ref["q"])
        assert np.array_equal(qt.cpu().numpy(), ref["qt"])
        q1, qt1, sc1, am1 = f8.f8_quantize(x.to(DEV), fmt=fmt)
        assert _eq(q, q1) and _eq(qt, qt1) and sc.item() == sc1.item()


def test_quantize_multi_launches_two_kernels(f8):
    xs = [_bf((256, 256), 1.0, i).to(DEV) for i in range(5)]
    n0 = f8.f8_kernel_launches()
    f8.f8_quantize_multi(xs)
    assert f8.f8_kernel_launches() - n0 == 2
    assert f8.f8_last_device_status() == 0


def _problems(specs, seed):
    """FP8 operands and scales for GEMM specs (M, N, K, fmt_a)."""
    out = []
    for i, (M, N, K, fa) in enumerate(specs):
        a = _bf((M, K), 1.0, seed + 10 * i).to(DEV)
        b = _bf((N, K), 0.05, seed + 10 * i + 1).to(DEV)
        qa, _, sa, _ = _quant(a, fa)
        qb, _, sb, _ = _quant(b, 0)
        out.append((qa, qb, sa, sb, M, N, K, fa))
    return out


def _quant(x, fmt):
    import float8_mixed_precision_gb300 as m
    return m.f8_quantize(x, fmt=fmt, want_t=False)


@pytest.mark.parametrize("specs", [
    # one K extent: one class, round-robin over the concatenated tiles
    [(512, 256, 256, 0), (512, 384, 256, 0), (272, 400, 256, 0)],
    # two K extents: the list schedule
    [(512, 512, 1024, 0), (512, 256, 256, 1), (384, 128, 1024, 0), (256, 256, 256, 0)],
    # three K extents over six problems: several launches
    [(512, 256, 128, 0), (256, 512, 512, 1), (512, 128, 1024, 0), (256, 256, 128, 0),
     (512, 384, 512, 0), (272, 144, 1024, 1)],
    # problems for both kernels (M < 256: single-CTA)
    [(128, 256, 256, 0), (512, 256, 256, 0), (48, 96, 512, 0)],
])
@pytest.mark.parametrize("mode", ["auto", "always"])
def test_gemm_grouped_matches_single_launches(f8, specs, mode, monkeypatch):
    if mode == "always":
        monkeypatch.setenv("F8_GEMM_GROUP", "2")
    probs = _problems(specs, 7)
    outs = f8.f8_gemm_grouped([(qa, qb, sa, sb, None, fa) for qa, qb, sa, sb, M, N, K, fa in probs])
    monkeypatch.delenv("F8_GEMM_GROUP", raising=False)
    singles = [f8.f8_gemm(qa, qb, sa, sb, fmt_a=fa) for qa, qb, sa, sb, M, N, K, fa in probs]
    assert f8.f8_last_device_status() == 0
    for o, s in zip(outs, singles):
        assert _eq(o, s)
    # and the oracle, for the first two problems in full
    for (qa, qb, sa, sb, M, N, K, fa), o in list(zip(probs, outs))[:2]:
        ref = oracle.gemm_rows_fmt(qa.cpu().numpy(), fa, qb.cpu().numpy(), 0, sa.item(), sb.item())
        check_close(o, ref, what=f"C {M}x{N}x{K}")


def test_gemm_grouped_forced_launch_of_eight(f8, monkeypatch):
    """Eight problems with two K extents forced into shared launches
    (launches take at most four): outputs still bit-identical."""
    specs = [(256 + 16 * i, 128 + 32 * i, 256 if i % 2 else 512, 0) for i in range(8)]
    probs = _problems(specs, 11)
    monkeypatch.setenv("F8_GEMM_GROUP", "2")
    outs = f8.f8_gemm_grouped([(qa, qb, sa, sb) for qa, qb, sa, sb, *_ in probs])
    monkeypatch.delenv("F8_GEMM_GROUP", raising=False)
    singles = [f8.f8_gemm(qa, qb, sa, sb) for qa, qb, sa, sb, *_ in probs]
    assert f8.f8_last_device_status() == 0
    for o, s in zip(outs, singles):
        assert _eq(o, s)


def _group_inputs(M, K, Ns, seed, x_std=1.0):
    x = _bf((M, K), x_std, seed)
    ws = [_bf((N, K), 0.02 * (i + 1), seed + 1 + i) for i, N in enumerate(Ns)]
    dys = [_bf((M, N), 0.01, seed + 10 + i) for i, N in enumerate(Ns)]
    return x, ws, dys


@pytest.mark.parametrize("M,K,Ns", [(256, 256, [384, 128, 128]), (512, 384, [256, 512]),
                                    (272, 528, [400, 144, 96, 272]), (128, 256, [256, 128])])
@pytest.mark.parametrize("dy_fmt", [0, 1])
def test_linear_group_matches_members(f8, M, K, Ns, dy_fmt):
    x, ws, dys = _group_inputs(M, K, Ns, M + K)
    xd = x.to(DEV)
    ys, saved = f8.f8_linear_fwd_group(xd, [w.to(DEV) for w in ws])
    dxs, dws = f8.f8_linear_bwd_group([d.to(DEV) for d in dys], saved, K, fmt=dy_fmt)
    assert f8.f8_last_device_status() == 0
    assert saved[0].x_t is saved[1].x_t
    for i, (w, dy) in enumerate(zip(ws, dys)):
        y1, s1 = f8.f8_linear_fwd(xd, w.to(DEV))
        dx1, dw1 = f8.f8_linear_bwd(dy.to(DEV), s1, dy_fmt=dy_fmt)
        assert _eq(ys[i], y1) and _eq(dxs[i], dx1) and _eq(dws[i], dw1)
        assert _eq(saved[i].x_t, s1.x_t) and _eq(saved[i].w_t, s1.w_t)
        assert saved[i].scale_x.item() == s1.scale_x.item()
        assert saved[i].scale_w.item() == s1.scale_w.item()
        fwd = oracle.linear_fwd(wl.bits(x), wl.bits(w))
        bwd = oracle.linear_bwd(wl.bits(dy), fwd, dy_fmt=dy_fmt)
        assert saved[i].scale_w.item() == float(fwd["w"]["scale"])
        assert np.array_equal(saved[i].w_t.cpu().numpy(), fwd["w"]["qt"])
        check_close(ys[i], fwd["y"], what=f"Y_{i}")
        check_close(dxs[i], bwd["dx"], what=f"dX_{i}")
        check_close(dws[i], bwd["dw"], what=f"dW_{i}")
    assert np.array_equal(saved[0].x_t.cpu().numpy(), oracle.quantize(wl.bits(x))["qt"])
    assert f8.f8_last_device_status() == 0


def test_linear_group_one_output_only(f8):
    M, K, Ns = 256, 256, [256, 128]
    x, ws, dys = _group_inputs(M, K, Ns, 3)
    ys, saved = f8.f8_linear_fwd_group(x.to(DEV), [w.to(DEV) for w in ws])
    dxs, dws = f8.f8_linear_bwd_group([d.to(DEV) for d in dys], saved, K)
    dx_only, none = f8.f8_linear_bwd_group([d.to(DEV) for d in dys], saved, K, want_dw=False)
    none2, dw_only = f8.f8_linear_bwd_group([d.to(DEV) for d in dys], saved, K, want_dx=False)
    assert none is None and none2 is None and f8.f8_last_device_status() == 0
    for i in range(len(Ns)):
        assert _eq(dx_only[i], dxs[i]) and _eq(dw_only[i], dws[i])


def test_llama8b_qkv_group(f8):
    """The q, k, v projections of the Llama-3.1-8B block at full size (M =
    8192, K = 4096, N = 4096, 1024, 1024) with the outlier workload's
    activations: the forward as three launches (two quantisation, one GEMM),
    the backward as four (two quantisation, two GEMM); every output
    bit-identical to the per-member calls and, on one sampled row per
    128-row band, within the GEMM bar of the oracle."""
    c = 5
    lins = wl.workload(c)[1][:3]
    M, K = lins[0].M, lins[0].K
    x = wl.linear_inputs(c, 0)["x"]
    ins = [wl.linear_inputs(c, i) for i in range(3)]
    xd = x.to(DEV)
    wds = [d["w"].to(DEV) for d in ins]
    dyds = [d["dy"].to(DEV) for d in ins]
    f8.f8_linear_fwd_group(xd, wds)       # first call: per-device set-up
    torch.cuda.synchronize()
    n0 = f8.f8_kernel_launches()
    ys, saved = f8.f8_linear_fwd_group(xd, wds)
    n1 = f8.f8_kernel_launches()
    dxs, dws = f8.f8_linear_bwd_group(dyds, saved, K)
    n2 = f8.f8_kernel_launches()
    assert f8.f8_last_device_status() == 0
    assert n1 - n0 == 3 and n2 - n1 == 4, (n1 - n0, n2 - n1)
    qx = oracle.quantize(wl.bits(x))
    assert saved[0].scale_x.item() == float(qx["scale"])
    rng = np.random.default_rng(5)
    rows = np.array([r * 128 + rng.integers(0, 128) for r in range(M // 128)], np.int64)
    ridx = torch.from_numpy(rows).to(DEV)
    for i, d in enumerate(ins):
        y1, s1 = f8.f8_linear_fwd(xd, wds[i])
        dx1, dw1 = f8.f8_linear_bwd(dyds[i], s1)
        assert _eq(ys[i], y1) and _eq(dxs[i], dx1) and _eq(dws[i], dw1)
        qw = oracle.quantize(wl.bits(d["w"]))
        qdy = oracle.quantize(wl.bits(d["dy"]))
        assert saved[i].scale_w.item() == float(qw["scale"])
        check_close(ys[i][ridx], oracle.gemm_rows(qx["q"], qw["q"], qx["scale"], qw["scale"], rows),
                    what=f"Y_{i} rows")
        check_close(dxs[i][ridx], oracle.gemm_rows(qdy["q"], qw["qt"], qdy["scale"], qw["scale"],
                                                   rows), what=f"dX_{i} rows")
        N = lins[i].N
        rows_n = np.array([r * 128 + rng.integers(0, 128) for r in range(N // 128)], np.int64)
        check_close(dws[i][torch.from_numpy(rows_n).to(DEV)],
                    oracle.gemm_rows(qdy["qt"], qx["qt"], qdy["scale"], qx["scale"], rows_n),
                    what=f"dW_{i} rows")
    assert f8.f8_last_device_status() == 0


def test_group_in_cuda_graph_matches_eager(f8):
    """The group forward and backward captured in a CUDA graph and replayed
    give the eager bits."""
    M, K, Ns = 512, 512, [512, 256, 256]
    x, ws, dys = _group_inputs(M, K, Ns, 21)
    xd, wds, dyds = x.to(DEV), [w.to(DEV) for w in ws], [d.to(DEV) for d in dys]
    ys, saved = f8.f8_linear_fwd_group(xd, wds)
    dxs, dws = f8.f8_linear_bwd_group(dyds, saved, K)
    torch.cuda.synchronize()
    ys2 = [torch.empty_like(y) for y in ys]
    dxs2 = [torch.empty_like(d) for d in dxs]
    dws2 = [torch.empty_like(d) for d in dws]
    saved2 = f8.group_saved(M, K, Ns, xd.device)
    wsp = f8.group_workspace(M, K, Ns, xd.device)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            f8.f8_linear_fwd_group(xd, wds, ys=ys2, saved=saved2, ws=wsp)
            f8.f8_linear_bwd_group(dyds, saved2, K, dxs=dxs2, dws=dws2, ws=wsp)
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    assert f8.f8_last_device_status() == 0
    for a, b in zip(ys + dxs + dws, ys2 + dxs2 + dws2):
        assert _eq(a, b)


def test_llama8b_w13_group(f8):
    """w1 and w3 of the Llama-3.1-8B block at full size (M = 8192, K = 4096,
    N = 14336 each; the outlier workload's activations), as the default
    bench step runs them: every output bit-identical to the per-member
    calls, and w1's Y, dX and dW within the GEMM bar of the oracle on one
    sampled row per 128-row band."""
    c = 5
    lins = wl.workload(c)[1]
    i1, i3 = 4, 5
    assert lins[i1].name == "w1" and lins[i3].name == "w3"
    M, K = lins[i1].M, lins[i1].K
    ins = [wl.linear_inputs(c, i) for i in (i1, i3)]
    x = ins[0]["x"]
    xd = x.to(DEV)
    wds = [d["w"].to(DEV) for d in ins]
    dyds = [d["dy"].to(DEV) for d in ins]
    ys, saved = f8.f8_linear_fwd_group(xd, wds)
    dxs, dws = f8.f8_linear_bwd_group(dyds, saved, K)
    assert f8.f8_last_device_status() == 0
    for i in range(2):
        y1, s1 = f8.f8_linear_fwd(xd, wds[i])
        dx1, dw1 = f8.f8_linear_bwd(dyds[i], s1)
        assert _eq(ys[i], y1) and _eq(dxs[i], dx1) and _eq(dws[i], dw1)
        del y1, s1, dx1, dw1
    qx = oracle.quantize(wl.bits(x))
    qw = oracle.quantize(wl.bits(ins[0]["w"]))
    qdy = oracle.quantize(wl.bits(ins[0]["dy"]))
    assert saved[0].scale_x.item() == float(qx["scale"])
    assert saved[0].scale_w.item() == float(qw["scale"])
    rng = np.random.default_rng(17)
    rows = np.array([r * 128 + rng.integers(0, 128) for r in range(M // 128)], np.int64)
    ridx = torch.from_numpy(rows).to(DEV)
    check_close(ys[0][ridx], oracle.gemm_rows(qx["q"], qw["q"], qx["scale"], qw["scale"], rows),
                what="Y_w1 rows")
    check_close(dxs[0][ridx], oracle.gemm_rows(qdy["q"], qw["qt"], qdy["scale"], qw["scale"], rows),
                what="dX_w1 rows")
    N = lins[i1].N
    rows_n = np.array([r * 128 + rng.integers(0, 128) for r in range(N // 128)], np.int64)
    check_close(dws[0][torch.from_numpy(rows_n).to(DEV)],
                oracle.gemm_rows(qdy["qt"], qx["qt"], qdy["scale"], qx["scale"], rows_n),
                what="dW_w1 rows")


def test_gemm_grouped_from_two_host_threads(f8):
    """Two host threads call f8_gemm_grouped at the same time, each on its
    own stream, alternating between two problem sets of their own, so the
    planner's cache of launch plans is read and filled from both threads at
    once.  The threads make no context-bound CUDA call of their own before
    the library's first call, so the library binds the device's primary
    context for them (its tensor-map encoder needs one).  Every output is
    bit-identical to f8_gemm on its problem."""
    import threading
    sets = [
        [[(512, 512, 1024, 0), (512, 256, 256, 0), (384, 128, 1024, 0)],
         [(512, 256, 128, 0), (256, 512, 512, 0), (512, 128, 1024, 0), (256, 256, 128, 0)]],
        [[(512, 384, 512, 0), (256, 256, 256, 1), (512, 640, 512, 0)],
         [(768, 256, 256, 0), (512, 512, 768, 0), (256, 384, 256, 0)]],
    ]
    probs = [[_problems(s, 300 + 40 * t + 20 * j) for j, s in enumerate(ts)]
             for t, ts in enumerate(sets)]
    singles = [[[f8.f8_gemm(qa, qb, sa, sb, fmt_a=fa) for qa, qb, sa, sb, M, N, K, fa in p]
                for p in tp] for tp in probs]
    outs = [[[torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
              for _, _, _, _, M, N, _, _ in p] for p in tp] for tp in probs]
    torch.cuda.synchronize()
    errors = []

    def work(t):
        try:
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                for it in range(40):
                    j = it % 2
                    f8.f8_gemm_grouped([(qa, qb, sa, sb, o, fa) for (qa, qb, sa, sb, M, N, K, fa), o
                                        in zip(probs[t][j], outs[t][j])])
            stream.synchronize()
        except Exception as e:  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(t,)) for t in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=120)
    assert not errors, errors
    torch.cuda.synchronize()
    assert f8.f8_last_device_status() == 0
    for t in range(2):
        for j in range(2):
            for o, s in zip(outs[t][j], singles[t][j]):
                assert _eq(o, s)


def test_planner_cache_past_its_bound(f8):
    """More distinct problem sets than the planner keeps plans for (1,100
    against 1,024): the cache is emptied and refilled on the way, and the
    outputs still equal single launches (checked on the first, the
    1,030th and the last set)."""
    K0, K1 = 256, 512
    a0 = _bf((256, K0), 1.0, 501).to(DEV)
    a1 = _bf((256, K1), 1.0, 502).to(DEV)
    b0 = _bf((16 * 1100, K0), 0.05, 503).to(DEV)
    b1 = _bf((64, K1), 0.05, 504).to(DEV)
    qa0, _, sa0, _ = _quant(a0, 0)
    qa1, _, sa1, _ = _quant(a1, 0)
    qb0, _, sb0, _ = _quant(b0, 0)
    qb1, _, sb1, _ = _quant(b1, 0)
    checked = {0: None, 1029: None, 1099: None}
    for i in range(1100):
        N = 16 * (i + 1)
        outs = f8.f8_gemm_grouped([(qa0, qb0[:N], sa0, sb0), (qa1, qb1, sa1, sb1)])
        if i in checked:
            checked[i] = (N, outs)
    for i, (N, outs) in checked.items():
        assert _eq(outs[0], f8.f8_gemm(qa0, qb0[:N], sa0, sb0)), i
        assert _eq(outs[1], f8.f8_gemm(qa1, qb1, sa1, sb1)), i
    assert f8.f8_last_device_status() == 0
