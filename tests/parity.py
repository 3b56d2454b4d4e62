"""Comparison helpers for the GPU parity tests (element by element against the oracle)."""
import numpy as np

# Tolerances (max-abs over every element): bf16 path O 1e-2, fp8 per-token-scale path
# O 3e-2 (against the oracle run on the dequantised fp8 values), LSE 1e-3 for both.
TOL_O_BF16 = 1e-2
TOL_O_FP8 = 3e-2
TOL_LSE = 1e-3


def half_ulp_bf16(x):
    """Half a bf16 unit in the last place of |x| (the rounding error of storing x in bf16)."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, 2.0 ** (e - 8), 0.0)


def check(o_gpu, o_ref, lse_gpu, lse_ref, tol_o, tol_lse=TOL_LSE, bf16_out=True, what=""):
    """Assert |O - O_ref| <= max(tol_o, half-ulp of O_ref in bf16) elementwise and LSE within
    tol_lse (rows with no visible key: LSE = -inf and O = 0 on both sides)."""
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    lse_gpu = np.asarray(lse_gpu, dtype=np.float64)
    assert o_gpu.shape == o_ref.shape, (o_gpu.shape, o_ref.shape)
    assert np.isfinite(o_gpu).all(), "%s: non-finite output" % what
    tol = np.maximum(tol_o, half_ulp_bf16(o_ref)) if bf16_out else tol_o
    err = np.abs(o_gpu - o_ref)
    worst = np.unravel_index(np.argmax(err - tol), err.shape)
    assert (err <= tol).all(), "%s: O max-abs err %.3e at %s (ref %.4f, got %.4f)" % (
        what, err.max(), worst, o_ref[worst], o_gpu[worst])
    fin = np.isfinite(lse_ref)
    assert (np.isneginf(lse_gpu[~fin])).all(), "%s: empty rows must have LSE=-inf" % what
    if fin.any():
        lerr = np.abs(lse_gpu[fin] - lse_ref[fin]).max()
        assert lerr <= tol_lse, "%s: LSE max-abs err %.3e" % (what, lerr)
    return float(err.max()), float(np.abs(lse_gpu[fin] - lse_ref[fin]).max()) if fin.any() else 0.0
