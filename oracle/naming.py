"""Evaluate a collective stated as a naming of input and output layouts.

Source: Purlin article, "The Purlin PDF describes a three-layer design" — the top layer
states a collective as a naming of an input layout and an output layout plus a copy or a
reduction. The pages give no formalism; the reading used here:

* a segment is (rank, offset, count, name), offset and count in elements of the dtype;
* every output segment receives the value of its name: for copy, the bytes of the single
  input segment carrying that name; for sum, the fixed-order sum of all input segments
  carrying that name, ordered by (rank, offset) ascending;
* output elements that no segment names are left as they were.

Error codes are the library's published numeric values; the precedence of checks is
fixed: arguments, then per-segment rank/count, bounds, lengths per name, producers per
name, overlap of outputs on one rank.
"""

from __future__ import annotations

import numpy as np

from .arith import ESIZE, ordered_sum

ERR = {
    "OK": 0,
    "EINVAL": -1,
    "ENAME": -2,
    "ELEN": -3,
    "EBOUNDS": -4,
    "EOVERLAP": -5,
}

MAX_RANKS = 64


def validate(R, op, dtype, in_len, in_segs, out_len, out_segs) -> int:
    if not (1 <= R <= MAX_RANKS) or op not in ("copy", "sum") or dtype not in ESIZE:
        return ERR["EINVAL"]
    if op == "sum" and dtype == "bytes":
        return ERR["EINVAL"]
    if len(in_len) != R or len(out_len) != R:
        return ERR["EINVAL"]
    segs = list(in_segs) + list(out_segs)
    for (r, off, cnt, name) in segs:
        if not (0 <= r < R) or cnt <= 0 or off < 0 or name < 0:
            return ERR["EINVAL"]
    for (r, off, cnt, _n) in in_segs:
        if off + cnt > in_len[r]:
            return ERR["EBOUNDS"]
    for (r, off, cnt, _n) in out_segs:
        if off + cnt > out_len[r]:
            return ERR["EBOUNDS"]
    count_of = {}
    for (_r, _o, cnt, name) in segs:
        if count_of.setdefault(name, cnt) != cnt:
            return ERR["ELEN"]
    producers = {}
    for (r, off, cnt, name) in in_segs:
        producers.setdefault(name, []).append((r, off))
    for (_r, _o, _c, name) in out_segs:
        p = producers.get(name, [])
        if len(p) == 0 or (op == "copy" and len(p) != 1):
            return ERR["ENAME"]
    for r in range(R):
        mine = sorted((off, cnt) for (rr, off, cnt, _n) in out_segs if rr == r)
        for (o0, c0), (o1, _c1) in zip(mine, mine[1:]):
            if o0 + c0 > o1:
                return ERR["EOVERLAP"]
    return ERR["OK"]


def run_naming(R, op, dtype, in_len, in_segs, out_len, out_segs, inputs, outputs) -> int:
    """Write every named output segment; `outputs` (list of R arrays) is updated in place.

    `inputs`/`outputs` hold uint16 (bf16 patterns), float32 or uint8 arrays per dtype.
    Returns the validation code; nothing is written unless it is 0.
    """
    code = validate(R, op, dtype, in_len, in_segs, out_len, out_segs)
    if code != 0:
        return code
    producers = {}
    for (r, off, cnt, name) in in_segs:
        producers.setdefault(name, []).append((r, off, cnt))
    for name in producers:
        producers[name].sort(key=lambda t: (t[0], t[1]))
    for (d, off, cnt, name) in out_segs:
        prods = producers[name]
        if op == "copy":
            (s, soff, _c) = prods[0]
            outputs[d][off:off + cnt] = inputs[s][soff:soff + cnt]
        else:
            terms = [inputs[s][soff:soff + cnt] for (s, soff, _c) in prods]
            outputs[d][off:off + cnt] = ordered_sum(terms, dtype)
    return 0


def run_epochs(R, op, dtype, in_len, in_segs, out_len, out_segs, pool_inputs, n_epochs,
               outputs_init):
    """Epoch semantics: epoch i reads input set i mod len(pool_inputs) and writes its own
    copy of the outputs (initialised from `outputs_init`); the result of an epoch does not
    depend on protocol, timing or retries. Returns a list of per-epoch output lists."""
    res = []
    for i in range(n_epochs):
        ins = pool_inputs[i % len(pool_inputs)]
        outs = [o.copy() for o in outputs_init]
        code = run_naming(R, op, dtype, in_len, in_segs, out_len, out_segs, ins, outs)
        if code != 0:
            raise ValueError(f"invalid naming: {code}")
        res.append(outs)
    return res
