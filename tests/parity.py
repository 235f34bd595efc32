"""Comparison helpers for the CUDA path against the float64 oracle.

Tolerances (stated for bf16 inputs/outputs with fp32 accumulation): O, dQ, dK,
dV max-abs error <= 2e-2 and relative L2 error <= 5e-3; lse max-abs <= 1e-3.
All errors are computed in float64 after upcasting the GPU's bf16/fp32 output.
"""
import numpy as np
import torch

TOL_MAXABS = 2e-2
TOL_RELL2 = 5e-3
TOL_LSE = 1e-3


def to64(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu").to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def errors(got, ref):
    g, r = to64(got), to64(ref)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.isfinite(g).all(), "non-finite values in GPU output"
    maxabs = float(np.abs(g - r).max()) if g.size else 0.0
    denom = float(np.linalg.norm(r.ravel()))
    rell2 = float(np.linalg.norm((g - r).ravel()) / denom) if denom > 0 else maxabs
    return maxabs, rell2


def assert_close(got, ref, name):
    maxabs, rell2 = errors(got, ref)
    assert maxabs <= TOL_MAXABS and rell2 <= TOL_RELL2, \
        f"{name}: max-abs {maxabs:.3e} (tol {TOL_MAXABS}), rel-L2 {rell2:.3e} (tol {TOL_RELL2})"
    return maxabs, rell2


def assert_lse_close(got, ref, name="lse"):
    g, r = to64(got), to64(ref)
    assert np.isfinite(g).all(), f"{name}: non-finite values"
    err = float(np.abs(g - r).max()) if g.size else 0.0
    assert err <= TOL_LSE, f"{name}: max-abs {err:.3e} (tol {TOL_LSE})"
    return err
