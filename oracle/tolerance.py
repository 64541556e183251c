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


def _gemv_terms(wt, x):
    """Products wt[i, j] * x[i] in binary64 ([k, n]); exact, since bf16 significands have 8
    bits and binary64 holds every product of two of them."""
    w = bf16_to_f32(wt).astype(np.float64)
    xv = bf16_to_f32(x).astype(np.float64)
    return w * xv[:, None]


def _gemv_bound(p):
    """(exact sum s, error bound B) of one payload taken in any order: the summation bound
    above over k products, plus k * 2^-53 * sum|p| for the binary64 sum standing in for
    the exact one and k * 2^-149 for products that round to binary32's subnormals."""
    k = p.shape[0]
    s = p.sum(axis=0)
    S = np.abs(p).sum(axis=0)
    acc = (k - 1) * 2.0 ** -24 * S + k * 2.0 ** -53 * S + k * 2.0 ** -149
    return s, RTOL["bf16"] * np.abs(s) + acc * (1 + RTOL["bf16"])


def _same_special(got, ref):
    """Where the plain-order result is an infinity or a NaN, another order must give the
    same class (an infinite product absorbs every finite term in any order)."""
    g = bf16_to_f32(got)
    r = bf16_to_f32(ref)
    return (np.isnan(g) & np.isnan(r)) | (np.isinf(r) & (g == r))


def gemv_within_tolerance(got, wt, x):
    """Boolean per output: is `got` (bf16 patterns) an acceptable payload y = W x for
    W given transposed as wt [k, n] and x [k] (all bf16), when a datapath adds the k
    products in another order than the plain one of ``collectives.gemv_payloads``? Each
    product is exact in binary32 when it stays in range, so only the order of the additions
    and the final rounding can move the result."""
    from .collectives import gemv_payloads
    s, B = _gemv_bound(_gemv_terms(wt, x))
    g = bf16_to_f32(got).astype(np.float64)
    ref = gemv_payloads([wt], [x])[0]
    special = ~np.isfinite(bf16_to_f32(ref))
    with np.errstate(invalid="ignore"):
        ok = np.abs(g - s) <= B
    return np.where(special, _same_special(got, ref), ok)


def gemv_sum_interval(wts, xs):
    """(t, bound, ref) for a rank-order sum over ranks r of payloads y_r = W_r x_r, each
    computed in another order than the plain one: an acceptable output g satisfies
    |g - t| <= bound where ref (the plain-order result, bf16 patterns) is finite, and has
    ref's class where ref is an infinity or a NaN.

    Payload r lies within B_r of its exact value s_r (``gemv_within_tolerance``); the
    datapath then adds the R payloads in rank order in binary32 (error at most
    (R-1) 2^-24 sum_r |y_r| <= (R-1) 2^-24 sum_r (|s_r| + B_r)) and rounds once to bf16
    (relative RTOL). With t = sum_r s_r and D the sum of those two error terms,
    |g - t| <= RTOL |t| + (1 + RTOL) D."""
    from .collectives import allreduce, gemv_payloads
    R = len(wts)
    ss, Bs = zip(*[_gemv_bound(_gemv_terms(w, x)) for w, x in zip(wts, xs)])
    t = np.sum(ss, axis=0)
    D = np.sum(Bs, axis=0) + (R - 1) * 2.0 ** -24 * np.sum(
        [np.abs(s) + b for s, b in zip(ss, Bs)], axis=0)
    ref = allreduce(gemv_payloads(wts, xs), "bf16")[0]
    return t, RTOL["bf16"] * np.abs(t) + (1 + RTOL["bf16"]) * D, ref


def gemv_sum_within_tolerance(got, wts, xs):
    """Boolean per output: is `got` (bf16 patterns) an acceptable rank-order sum of the
    payloads W_r x_r, each taken in another order (``gemv_sum_interval``)?"""
    t, bound, ref = gemv_sum_interval(wts, xs)
    g = bf16_to_f32(got).astype(np.float64)
    special = ~np.isfinite(bf16_to_f32(ref))
    with np.errstate(invalid="ignore"):
        ok = np.abs(g - t) <= bound
    return np.where(special, _same_special(got, ref), ok)
