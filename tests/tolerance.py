"""Comparison of GPU outputs with the fp64 oracle.

Reading of the stated tolerances (forward and dx within 1 ulp of a 16-bit
output type or 1e-6 relative for fp32; grad_w / dw within 1e-5 relative):

* clause 1 — 16-bit outputs: ordered-bit distance <= 1 from the oracle's
  value rounded once to the output type; fp32 outputs: |g − r| <= tol·|r|.
* clause 2 — for results whose terms cancel (every reduction, and the SiLU
  derivative s + x·s·(1−s)), a relative bound cannot hold near zero; there
  |g − r| <= tol·S/√K, with S the sum of the terms' magnitudes and K their
  count (S/√K is the natural size of a K-term random-sign sum).  For the
  two-term SiLU derivative the scale is tol·S.
tol is 2^-10 for binary16, 2^-7 for bfloat16 (one unit in the last place at
the bottom of a binade) and 1e-6 for binary32 elementwise outputs; 1e-5 for
grad_w and dw.  A binary32 result also passes clause 1 within 2^-149 (the
subnormal quantum: values below the binary32 range, e.g. exp(-160), round to
zero or a subnormal).  Each check reports how many elements passed only by
clause 2.
"""
from __future__ import annotations

import numpy as np
import torch

TOL = {torch.float16: 2.0 ** -10, torch.bfloat16: 2.0 ** -7, torch.float32: 1e-6}
GRAD_TOL = 1e-5
F32_QUANTUM = 2.0 ** -149


def ordered(t: torch.Tensor) -> np.ndarray:
    """Map 16-bit patterns to integers ordered like the values."""
    i = t.contiguous().view(torch.int16).numpy().astype(np.int64)
    return np.where(i < 0, -(i & 0x7FFF), i)


def ulp_dist16(a: torch.Tensor, b: torch.Tensor) -> np.ndarray:
    return np.abs(ordered(a) - ordered(b))


class Result:
    def __init__(self, ok, clause2, max_rel, n):
        self.ok, self.clause2, self.max_rel, self.n = ok, clause2, max_rel, n

    def __bool__(self):
        return bool(self.ok)

    def __repr__(self):
        return f"Result(ok={self.ok}, clause2={self.clause2}, max_rel={self.max_rel:.3g}, n={self.n})"


def check_elementwise(got: torch.Tensor, ref_rounded: torch.Tensor, exact: np.ndarray,
                      scale: np.ndarray | None = None) -> Result:
    """got / ref_rounded: host tensors of the output type; exact: fp64
    values; scale: fp64 magnitude of the cancelling terms (or None)."""
    got = got.reshape(-1)
    ref_rounded = ref_rounded.reshape(-1)
    exact = np.asarray(exact, dtype=np.float64).reshape(-1)
    g = got.double().numpy()
    tol = TOL[got.dtype]
    err = np.abs(g - exact)
    with np.errstate(divide="ignore", invalid="ignore"):
        rel = np.where(exact != 0, err / np.abs(exact), np.where(err == 0, 0.0, np.inf))
    if got.dtype == torch.float32:
        c1 = err <= tol * np.abs(exact) + F32_QUANTUM
    else:
        c1 = ulp_dist16(got, ref_rounded) <= 1
    both_nan = np.isnan(g) & np.isnan(exact)
    c1 = c1 | both_nan
    c2 = np.zeros_like(c1)
    if scale is not None:
        c2 = err <= tol * np.asarray(scale, dtype=np.float64).reshape(-1)
    ok = c1 | c2
    fin = np.isfinite(rel)
    return Result(bool(ok.all()), int((~c1 & c2).sum()), float(rel[fin].max()) if fin.any() else 0.0,
                  int(ok.size))


def check_reduction(got, exact: np.ndarray, abs_sum: np.ndarray, K: int, tol: float,
                    ref_rounded: torch.Tensor | None = None) -> Result:
    """Reductions: clause 1 (relative, or 1 ulp for a 16-bit output when
    ref_rounded is given) or clause 2 with scale S/√K."""
    if isinstance(got, torch.Tensor):
        g = got.reshape(-1).double().numpy()
    else:
        g = np.asarray(got, dtype=np.float64).reshape(-1)
    exact = np.asarray(exact, dtype=np.float64).reshape(-1)
    S = np.asarray(abs_sum, dtype=np.float64).reshape(-1)
    err = np.abs(g - exact)
    if ref_rounded is not None and got.dtype != torch.float32:
        c1 = ulp_dist16(got.reshape(-1), ref_rounded.reshape(-1)) <= 1
    else:
        c1 = err <= tol * np.abs(exact)
    c2 = err <= tol * S / np.sqrt(max(K, 1))
    ok = c1 | c2
    with np.errstate(divide="ignore", invalid="ignore"):
        rel = np.where(exact != 0, err / np.abs(exact), 0.0)
    return Result(bool(ok.all()), int((~c1 & c2).sum()), float(rel.max()) if rel.size else 0.0,
                  int(ok.size))
