"""The GEMM parity bar: elementwise |y - y_oracle| <= 2 ulp_bf16(y_oracle) + 1e-5 rms(Y_oracle)
and ||Y - Y_oracle||_F <= 1e-3 ||Y_oracle||_F, where ulp_bf16(y) = 2^(floor(log2|y|) - 7) for
normal |y| and 2^-133 below the normal range.  Both sides are bf16 outputs."""
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
