"""Tolerance for sums taken in another order than the fixed rank order.

The fixed rank order is the reference, and rank-order results are compared bit for bit.
A datapath that adds in another order (a pairwise tree, an in-memory reduction) is checked
against the exact sum s = sum_i x_i (fp64 here, which is exact for up to 2^29 bf16 terms and
for the sizes used with fp32 terms) with the first-order error bound of floating-point
summation in any order: |s_hat - s| <= (n - 1) * u * sum_i |x_i| with u = 2^-24 for binary32
accumulation (Higham, Accuracy and Stability of Numerical Algorithms, ch. 4), plus the final
rounding of the output: relative 2^-8 for bf16 (round to nearest, 7 stored significand bits),
inside the required 4e-3; for fp32 outputs the accumulation bound already covers it and
1e-6 relative is allowed on top.
"""

from __future__ import annotations

import numpy as np

from .arith import bf16_to_f32, to_f32

RTOL = {"bf16": 4e-3, "f32": 1e-6}


def exact_sum(terms, dtype):
    return np.sum([to_f32(t, dtype).astype(np.float64) for t in terms], axis=0)


def within_tolerance(got, terms, dtype):
    """Boolean per element: is `got` (bf16 patterns or float32) an acceptable sum?"""
    n = len(terms)
    s = exact_sum(terms, dtype)
    S = np.sum([np.abs(to_f32(t, dtype).astype(np.float64)) for t in terms], axis=0)
    g = (bf16_to_f32(got) if dtype == "bf16" else np.asarray(got, np.float32)).astype(np.float64)
    bound = RTOL[dtype] * np.abs(s) + (n - 1) * 2.0 ** -24 * S * (1 + RTOL[dtype])
    return np.abs(g - s) <= bound
