"""Shared parity checks: GPU results (up-cast) against the fp64 oracle.

Tolerances (from the stated correctness bar of this library):
* bf16 outputs: max-abs error <= 2e-2 and relative Frobenius error <= 5e-3;
* gradients and dsink: relative Frobenius error <= 1e-2;
* LSE (fp32): abs error <= 2e-3 -- the inputs are identical bf16 values, so the
  only differences are the fp32 dot products (~1e-6 relative) and the
  hardware exp2/log2 approximations (~1e-6 relative), far inside this bound;
* index and selection outputs: bit-exact.
"""
import numpy as np
import torch

O_MAX_ABS = 2e-2
O_REL_FRO = 5e-3
GRAD_REL_FRO = 1e-2
LSE_ABS = 2e-3


def _np(x):
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def rel_fro(got, want):
    got, want = _np(got), _np(want)
    den = np.linalg.norm(want)
    return np.linalg.norm(got - want) / (den if den > 0 else 1.0)


def assert_out_close(got, want, what="out"):
    got, want = _np(got), _np(want)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - want).max() if got.size else 0.0
    rf = rel_fro(got, want)
    assert err <= O_MAX_ABS, f"{what}: max-abs {err:.3e} > {O_MAX_ABS}"
    assert rf <= O_REL_FRO, f"{what}: rel-Frobenius {rf:.3e} > {O_REL_FRO}"
    return err, rf


def assert_lse_close(got, want, what="lse"):
    got, want = _np(got), _np(want)
    same_inf = np.isinf(want) & (got == want)
    fin = ~same_inf
    assert np.all(np.isfinite(got[fin])), f"{what}: unexpected non-finite"
    err = np.abs(got[fin] - want[fin]).max() if fin.any() else 0.0
    assert err <= LSE_ABS, f"{what}: max-abs {err:.3e} > {LSE_ABS}"
    return err


def assert_grad_close(got, want, what="grad"):
    got, want = _np(got), _np(want)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    rf = rel_fro(got, want)
    assert rf <= GRAD_REL_FRO, f"{what}: rel-Frobenius {rf:.3e} > {GRAD_REL_FRO}"
    return rf
