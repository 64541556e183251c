"""Element arithmetic of the reduce primitive, written out plainly (numpy, no fusion).

The Atom datapath has two primitives, copy and reduce (Purlin article, "The Purlin PDF
describes a three-layer design"; figure "Purlin separates the collective stack").
The pages fix neither the precision nor the summation order; the reading used here:

* bf16 values widen to binary32 exactly (append 16 zero bits);
* the sum is a left-to-right chain in binary32, acc = x_0, acc = acc + x_k, each add
  rounded to nearest even (numpy float32 add is IEEE 754 binary32 addition, no FMA);
* a bf16 result is rounded once from the binary32 sum, to nearest, ties to even; a NaN
  stays a (quiet) NaN.
"""

from __future__ import annotations

import numpy as np

ESIZE = {"bf16": 2, "f32": 4, "bytes": 1}
NPTYPE = {"bf16": np.uint16, "f32": np.float32, "bytes": np.uint8}


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to binary32 values, exactly."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def f32_to_bf16_rne(x: np.ndarray) -> np.ndarray:
    """Round binary32 values to bf16 bit patterns, nearest, ties to even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).copy()
    is_nan = (u & np.uint32(0x7FFFFFFF)) > np.uint32(0x7F800000)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    with np.errstate(over="ignore"):
        r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    r = r.astype(np.uint16)
    if is_nan.any():
        r[is_nan] = ((u[is_nan] >> np.uint32(16)) | np.uint32(0x0040)).astype(np.uint16)
    return r


def to_f32(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return bf16_to_f32(x)
    if dtype == "f32":
        return np.asarray(x, dtype=np.float32)
    raise ValueError("sum is defined for bf16 and f32 only")


def ordered_sum(terms, dtype: str) -> np.ndarray:
    """Sum equally long arrays in the given order; returns the output dtype's array."""
    acc = to_f32(terms[0], dtype).copy()
    with np.errstate(over="ignore", invalid="ignore"):
        for t in terms[1:]:
            acc = acc + to_f32(t, dtype)
    if dtype == "bf16":
        return f32_to_bf16_rne(acc)
    return acc.astype(np.float32)
