"""Parity measures between a GPU result and the fp64 oracle.

TEST INFRASTRUCTURE ONLY (like the rest of ``oracle/``): used by the test
suite and by the benchmark's parity leg, which runs outside the timed region.

The tolerances are the ones the method is held to, for bf16 inputs and f32
accumulation:
  - relative Frobenius error ||x - ref||_F / ||ref||_F: O <= 5e-3, dQ/dK/dV <= 1e-2;
  - elementwise absolute error max |x - ref| <= 2e-2 (the "flat" bound);
  - LSE absolute error max |lse - ref| <= 1e-3.
The outputs are stored in bf16.  Rounding an exact value to bf16 moves it by
up to half a unit in its last place, 2^-9 |x| relative, which is already more
than 2e-2 once |x| > 8.  So every comparison reports two elementwise
figures:
  - the flat excess  max(|x - ref|) - 2e-2;
  - the widened excess max(|x - ref| - (2e-2 + halfulp_bf16(ref) [+ 3 u e])),
    where, for the gradients only, e is the oracle's root-sum-square
    rounding-error scale of the element when P, dS and the stored O enter the
    products as bf16 operands, and u = 2^-8 (see ``rounding_bound``).
An output "meets flat" when its flat excess is <= 0, "meets half-ulp" when
|x - ref| <= 2e-2 + halfulp_bf16(ref) everywhere (the most a correctly
rounded bf16 store of the exact value can be held to), and "meets widened"
when only the bound with the 3 u e term holds.
"""
from __future__ import annotations

import json
import os

import numpy as np

TOL_REL_O = 5e-3
TOL_REL_GRAD = 1e-2
TOL_ABS = 2e-2
TOL_LSE = 1e-3

U_BF16 = 2.0 ** -8      # unit of the bf16 operand rounding in the error scale e
LAMBDA = 3.0            # e is a root-sum-square scale; three of it bounds the sum


def rel_fro(x, ref) -> float:
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / (den if den > 0 else 1.0))


def bf16_half_ulp(ref):
    """Half a bf16 unit in the last place at |ref| (8 significant bits)."""
    a = np.abs(np.asarray(ref, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 8.0), 0.0)


def rounding_bound(ref, err=None):
    """The widened elementwise bound: 2e-2 + bf16 half-ulp of ref [+ 3 u e]."""
    bound = TOL_ABS + bf16_half_ulp(ref)
    if err is not None:
        bound = bound + LAMBDA * U_BF16 * np.asarray(err, dtype=np.float64)
    return bound


def compare(name: str, x, ref, rel_tol: float, err=None) -> dict:
    """Every parity figure of one output (x and ref float64 arrays)."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    finite = bool(np.isfinite(x).all())
    if x.size == 0:
        return dict(name=name, finite=True, rel_fro=0.0, rel_tol=rel_tol, max_abs=0.0, flat_excess=-TOL_ABS,
                    ulp_excess=-TOL_ABS, widened_excess=-TOL_ABS, max_ref=0.0, meets="flat", ok=True)
    diff = np.abs(x - ref)
    rf = rel_fro(x, ref)
    max_abs = float(diff.max())
    widened = float((diff - rounding_bound(ref, err)).max())
    ulp = float((diff - rounding_bound(ref)).max())
    flat = max_abs - TOL_ABS
    if flat <= 0:
        meets = "flat"
    elif ulp <= 0:
        meets = "half-ulp"
    else:
        meets = "widened" if widened <= 0 else "none"
    ok = finite and rf <= rel_tol and widened <= 0
    return dict(name=name, finite=finite, rel_fro=rf, rel_tol=rel_tol, max_abs=max_abs, flat_excess=flat,
                ulp_excess=ulp, widened_excess=widened, max_ref=float(np.abs(ref).max()), meets=meets, ok=ok)


def compare_lse(x, ref) -> dict:
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = float(np.abs(x - ref).max()) if x.size else 0.0
    return dict(name="lse", finite=bool(np.isfinite(x).all()), max_abs=err, tol=TOL_LSE,
                ok=bool(np.isfinite(x).all()) and err <= TOL_LSE)


def record(case: str, entry: dict) -> None:
    """Append one comparison to the JSON-lines file named by GQA_PARITY_RECORD
    (nothing when the variable is unset)."""
    path = os.environ.get("GQA_PARITY_RECORD")
    if not path:
        return
    with open(path, "a") as f:
        f.write(json.dumps(dict(case=case, **entry)) + "\n")
