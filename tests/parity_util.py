"""Comparison helpers for GPU-vs-oracle parity tests.

The tolerances and both elementwise figures (flat 2e-2, and the widened bound
that adds the bf16 half-ulp of the reference and, for gradients, 3 u e) are
defined in ``oracle/parity.py``.  ``check`` asserts the relative Frobenius
bound and the widened elementwise bound, and records every figure -- the flat
excess included -- in the JSON-lines file named by GQA_PARITY_RECORD, keyed by
the running test, so a run leaves a record of which bound each output meets.
"""
import os

import numpy as np
import torch

from oracle import parity as P

TOL_REL_O = P.TOL_REL_O
TOL_REL_GRAD = P.TOL_REL_GRAD
TOL_ABS = P.TOL_ABS
TOL_LSE = P.TOL_LSE
rel_fro = P.rel_fro
bf16_half_ulp = P.bf16_half_ulp


def _case():
    return os.environ.get("PYTEST_CURRENT_TEST", "?").split(" (")[0]


def abs_excess(x, ref, err=None):
    """max(|x - ref| - (2e-2 + bf16 half-ulp of ref [+ 3 u err])); <= 0 passes."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float((np.abs(x - ref) - P.rounding_bound(ref, err)).max()) if x.size else -1.0


def to64(t):
    return t.detach().float().cpu().double().numpy()


def check(name, x, ref, rel_tol, err=None):
    """Relative Frobenius <= rel_tol and the widened elementwise bound; returns
    (relative Frobenius error, flat elementwise excess)."""
    x = to64(x) if isinstance(x, torch.Tensor) else np.asarray(x, dtype=np.float64)
    r = P.compare(name, x, ref, rel_tol, err)
    P.record(_case(), r)
    assert r["finite"], f"{name}: non-finite values"
    assert r["rel_fro"] <= rel_tol, f"{name}: relative Frobenius error {r['rel_fro']:.3e} > {rel_tol}"
    assert r["widened_excess"] <= 0, (f"{name}: elementwise error exceeds bound by {r['widened_excess']:.3e} "
                                      f"(flat excess {r['flat_excess']:.3e})")
    print(f"{name}: rel_fro {r['rel_fro']:.2e}, max abs {r['max_abs']:.2e} (flat excess {r['flat_excess']:+.2e}, "
          f"meets {r['meets']})")
    return r["rel_fro"], r["flat_excess"]


def check_lse(x, ref):
    x = to64(x) if isinstance(x, torch.Tensor) else np.asarray(x, dtype=np.float64)
    r = P.compare_lse(x, ref)
    P.record(_case(), r)
    assert r["ok"], f"lse: max abs error {r['max_abs']:.3e} > {TOL_LSE}"
    return r["max_abs"]
