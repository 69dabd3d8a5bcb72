"""Parity bars.

GEMM outputs: elementwise |y - y_oracle| <= 2 ulp_bf16(y_oracle) + 1e-5 rms(Y_oracle)
and ||Y - Y_oracle||_F <= 1e-3 ||Y_oracle||_F, where ulp_bf16(y) = 2^(floor(log2|y|) - 7) for
normal |y| and 2^-133 below the normal range.  Both sides are bf16 outputs.

SwiGLU outputs (h = silu(a) b and its gradient): the oracle is the definition evaluated in fp64
and rounded once to bf16; the GPU evaluates it in fp32 (a few fp32 ulp from exact), so its bf16
result equals the oracle's except where the exact value lies within a few fp32 ulp of a bf16
rounding boundary, and then is one of the two neighbours: |h - h_oracle| <= 1 ulp_bf16(h_oracle),
NaN exactly where the oracle has NaN, infinities equal.  The fraction of elements that differ
at all is asserted too (a fault that moved many values by one ulp would fail it)."""
import numpy as np
import torch

ULPS = 2.0
RMS_FRAC = 1e-5
FRO = 1e-3


def bits_to_f64(b) -> np.ndarray:
    if isinstance(b, torch.Tensor):
        t = b.detach().cpu()
        if t.dtype == torch.bfloat16:
            return t.to(torch.float64).numpy()
        b = t.numpy()
    b = np.ascontiguousarray(np.asarray(b, np.uint16))
    return torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def ulp_bf16(y: np.ndarray) -> np.ndarray:
    a = np.abs(y)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a >= 2.0 ** -126, 2.0 ** (e - 7), 2.0 ** -133)


def check_close(got, ref, rms_of=None, what=""):
    """Assert the parity bar; ``rms_of`` is the full oracle output when ``ref`` is a sample."""
    g = bits_to_f64(got)
    r = bits_to_f64(ref)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    rr = r if rms_of is None else bits_to_f64(rms_of)
    rms = float(np.sqrt(np.mean(rr ** 2))) if rr.size else 0.0
    err = np.abs(g - r)
    bound = ULPS * ulp_bf16(r) + RMS_FRAC * rms
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside the bound; first at "
                             f"{tuple(i)}: got {g[tuple(i)]!r} want {r[tuple(i)]!r} "
                             f"bound {bound[tuple(i)]!r}")
    nr = np.linalg.norm(r)
    if nr > 0:
        rel = np.linalg.norm(g - r) / nr
        assert rel <= FRO, f"{what}: relative Frobenius error {rel:.3e} > {FRO}"
    return {"max_err_ulps": float((err / ulp_bf16(r)).max()) if r.size else 0.0}


SWIGLU_ULPS = 1.0
# Fraction of SwiGLU outputs allowed to differ (by at most SWIGLU_ULPS) from the oracle:
# ordinary inputs (|a| of order 1), where a CPU emulation of the kernel's fp32 steps differs
# on 2e-5 of the elements; and sweeps over every bf16 value of a, where the emulation
# differs on 1.0e-3 (mostly large |a|, where sigma(a) rounds to 1 in fp32 and a b is an
# exact bf16 midpoint that the fp64 value lies just below).
SWIGLU_MISMATCH_ORDINARY = 1e-3
SWIGLU_MISMATCH_SWEEP = 2e-3


def check_swiglu_ulp(got, ref, max_frac, what=""):
    """Assert the SwiGLU bar on two bf16 tensors (bit patterns or bf16 torch tensors);
    returns the fraction of elements that differ."""
    def _bits(x):
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous().view(torch.int16).numpy()
        return np.ascontiguousarray(np.asarray(x)).view(np.uint16).ravel()

    g, r = _bits(got), _bits(ref)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    nan_g = (g & 0x7FFF) > 0x7F80
    nan_r = (r & 0x7FFF) > 0x7F80
    assert np.array_equal(nan_g, nan_r), f"{what}: NaN in {int((nan_g != nan_r).sum())} places only on one side"
    g, r = g[~nan_r], r[~nan_r]
    diff = g != r
    if diff.any():
        gv, rv = bits_to_f64(g[diff]), bits_to_f64(r[diff])
        assert np.isfinite(gv).all() and np.isfinite(rv).all(), f"{what}: infinities differ"
        err = np.abs(gv - rv)
        bad = err > SWIGLU_ULPS * ulp_bf16(rv)
        if bad.any():
            i = int(np.argmax(bad))
            raise AssertionError(f"{what}: {int(bad.sum())} elements more than {SWIGLU_ULPS} ulp "
                                 f"off; e.g. got {gv[i]!r} want {rv[i]!r}")
    frac = float(diff.mean()) if diff.size else 0.0
    assert frac <= max_frac, f"{what}: {frac:.2e} of the elements differ (bar {max_frac:.0e})"
    return frac
