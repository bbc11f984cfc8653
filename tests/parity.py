"""Shared helpers of the GPU parity tests: tolerances, cached workloads and
oracle results.  The tolerance for bf16 caches is max|d| <= 1e-2 * max|ref| +
1e-3 on out and on lse; for the fp32 cache it is 1e-4 relative to max|ref|.
"""
from __future__ import annotations

import functools
import os

import numpy as np

import oracle
from mla_tree_verify_absorbed_gb300 import inputs as I


def tol_ok(got: np.ndarray, ref: np.ndarray, dtype: str):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin), "non-finite pattern differs"
    d = np.abs(got[fin] - ref[fin])
    mx = float(np.abs(ref[fin]).max()) if fin.any() else 0.0
    dmax = float(d.max()) if d.size else 0.0
    bound = (1e-4 * mx) if dtype == "fp32" else (1e-2 * mx + 1e-3)
    return dmax <= bound, dmax, bound, mx


# Achieved margins of every comparison in this session: (test, what, max|d|,
# max|ref|, bound).  conftest.py writes them out when MLA_PARITY_MARGINS
# names a file.
MARGINS = []


def assert_close(got, ref, dtype, what=""):
    ok, dmax, bound, mx = tol_ok(got, ref, dtype)
    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
    MARGINS.append(dict(test=test, what=what, dtype=dtype, max_abs_diff=dmax, max_abs_ref=mx, bound=bound,
                        rel=dmax / max(mx, 1e-30), passed=bool(ok)))
    assert ok, f"{what}: max|d|={dmax:.3e} > bound {bound:.3e} (max|ref|={mx:.3e})"
    return dmax / max(mx, 1e-30)


@functools.lru_cache(maxsize=None)
def workload(name: str, needles: bool = False) -> I.Problem:
    p = I.make_config(name)
    if needles:
        I.plant_needles(p)
    return p


def oracle_rows(p: I.Problem, rows: np.ndarray):
    out, lse, nvis = oracle.get().verify_rows(p, rows)
    return out, lse


def gather_rows(out_t, lse_t, rows: np.ndarray):
    """GPU results at rows (b, i, h) as float64 numpy."""
    import torch
    b = torch.as_tensor(rows[:, 0], device=out_t.device, dtype=torch.long)
    i = torch.as_tensor(rows[:, 1], device=out_t.device, dtype=torch.long)
    h = torch.as_tensor(rows[:, 2], device=out_t.device, dtype=torch.long)
    o = out_t[b, i, h].float().cpu().numpy().astype(np.float64)
    l = lse_t[b, i, h].float().cpu().numpy().astype(np.float64)
    return o, l
