"""Independent per-element evaluator with exact rational arithmetic (tiny cases only).

It shares nothing with ``oracle.naming``/``oracle.arith`` beyond the reading it
implements: binary32 values are decoded to exact rationals, each addition is carried out
exactly and rounded by the textbook rule (nearest representable value, ties to the even
significand, overflow to infinity), and bf16 is the same rule with an 8-bit significand.
Signed zero follows IEEE 754: an exact zero sum is +0 unless both addends are -0.
Used by the tests to pin the numpy oracle, never on large inputs.
"""

from __future__ import annotations

from fractions import Fraction
import struct

INF = "inf"


class Val:
    """A finite float as an exact rational plus the sign of zero, or an infinity."""

    __slots__ = ("q", "neg", "inf")

    def __init__(self, q=Fraction(0), neg=False, inf=0):
        self.q, self.neg, self.inf = Fraction(q), bool(neg), inf

    def key(self):
        if self.inf:
            return ("inf", self.inf)
        if self.q == 0:
            return ("zero", self.neg)
        return ("num", self.q)


def _decode(bits: int, ebits: int, mbits: int) -> Val:
    sign = (bits >> (ebits + mbits)) & 1
    e = (bits >> mbits) & ((1 << ebits) - 1)
    m = bits & ((1 << mbits) - 1)
    bias = (1 << (ebits - 1)) - 1
    if e == (1 << ebits) - 1:
        if m:
            raise ValueError("NaN is outside the brute-force evaluator")
        return Val(inf=-1 if sign else 1)
    if e == 0:
        q = Fraction(m, 1) * Fraction(2) ** (1 - bias - mbits)
    else:
        q = Fraction((1 << mbits) + m) * Fraction(2) ** (e - bias - mbits)
    return Val(-q if sign else q, neg=bool(sign))


def decode_f32(bits: int) -> Val:
    return _decode(bits, 8, 23)


def decode_bf16(bits: int) -> Val:
    return _decode(bits, 8, 7)


def f32_bits(x: float) -> int:
    return struct.unpack("<I", struct.pack("<f", x))[0]


def _round(v: Val, p: int, emin: int, emax: int) -> Val:
    """Round to a binary format with p significand bits (implicit bit included)."""
    if v.inf or v.q == 0:
        return v
    a = abs(v.q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    # now 2^e <= a < 2^(e+1)
    e = max(e, emin)
    ulp = Fraction(2) ** (e - p + 1)
    m = a / ulp
    n = m.numerator // m.denominator
    rem = m - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    r = n * ulp
    if r >= Fraction(2) ** (emax + 1):
        return Val(inf=-1 if v.q < 0 else 1)
    if r == 0:
        return Val(0, neg=v.q < 0)
    return Val(-r if v.q < 0 else r)


def round_f32(v: Val) -> Val:
    return _round(v, 24, -126, 127)


def round_bf16(v: Val) -> Val:
    return _round(v, 8, -126, 127)


def add(a: Val, b: Val, rounder) -> Val:
    if a.inf or b.inf:
        if a.inf and b.inf and a.inf != b.inf:
            raise ValueError("inf - inf is outside the brute-force evaluator")
        return Val(inf=a.inf or b.inf)
    s = a.q + b.q
    if s == 0:
        both_neg = (a.q == 0 and a.neg) and (b.q == 0 and b.neg)
        return Val(0, neg=both_neg)
    return rounder(Val(s))


def element_sum(vals, out_dtype: str) -> Val:
    """Left-to-right binary32 chain, then one bf16 rounding for bf16 outputs."""
    acc = vals[0]
    for v in vals[1:]:
        acc = add(acc, v, round_f32)
    if out_dtype == "bf16":
        acc = round_bf16(acc)
    return acc


def evaluate(op, dtype, in_segs, out_segs, inputs, out_len):
    """Per-element evaluation of a (valid) naming.

    inputs: list of per-rank lists of raw element bit patterns (ints).
    Returns per-rank dicts {element index: Val or raw int (copy)} for named elements.
    """
    by_name = {}
    for (r, off, cnt, name) in in_segs:
        by_name.setdefault(name, []).append((r, off))
    outs = [dict() for _ in out_len]
    dec = decode_bf16 if dtype == "bf16" else decode_f32
    for (d, off, cnt, name) in out_segs:
        prods = sorted(by_name[name])
        for i in range(cnt):
            if op == "copy":
                (s, so) = prods[0]
                outs[d][off + i] = inputs[s][so + i]
            else:
                vals = [dec(inputs[s][so + i]) for (s, so) in prods]
                outs[d][off + i] = element_sum(vals, dtype)
    return outs
