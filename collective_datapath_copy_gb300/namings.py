"""Namings of the standard collectives (host-side helpers; no data is touched here).

A naming cuts each rank's input and output buffer into named segments; the operation says
what an output segment receives from the input segments with its name (Purlin article,
"The Purlin PDF describes a three-layer design"). Sizes are in elements.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from ._lib import SEG_DTYPE


def segs(rows) -> np.ndarray:
    """(rank, offset, count, name) rows -> coll_seg_t array."""
    rows = list(rows)
    a = np.zeros(len(rows), dtype=SEG_DTYPE)
    if rows:
        r = np.asarray(rows, dtype=np.int64).reshape(-1, 4)
        a["rank"], a["offset"], a["count"], a["name"] = r[:, 0], r[:, 1], r[:, 2], r[:, 3]
    return a


def _segs_cols(rank, offset, count, name) -> np.ndarray:
    a = np.zeros(len(rank), dtype=SEG_DTYPE)
    a["rank"], a["offset"], a["count"], a["name"] = rank, offset, count, name
    return a


@dataclass
class Naming:
    R: int
    op: str
    dtype: str
    in_len: list
    in_segs: np.ndarray
    out_len: list
    out_segs: np.ndarray
    meta: dict = field(default_factory=dict)

    def rows(self, which="in"):
        s = self.in_segs if which == "in" else self.out_segs
        return [(int(x["rank"]), int(x["offset"]), int(x["count"]), int(x["name"])) for x in s]


def allreduce(R: int, n: int, dtype: str = "bf16") -> Naming:
    """Every rank's whole buffer carries one name; every output receives its sum."""
    i = _segs_cols(np.arange(R), np.zeros(R), np.full(R, n), np.zeros(R))
    return Naming(R, "sum", dtype, [n] * R, i, [n] * R, i.copy())


def reduce_scatter(R: int, n: int, dtype: str = "bf16") -> Naming:
    """Input block j (of n/R) on every rank is name j; rank r's output is name r."""
    assert n % R == 0
    b = n // R
    rr, jj = np.meshgrid(np.arange(R), np.arange(R), indexing="ij")
    i = _segs_cols(rr.ravel(), (jj * b).ravel(), np.full(R * R, b), jj.ravel())
    o = _segs_cols(np.arange(R), np.zeros(R), np.full(R, b), np.arange(R))
    return Naming(R, "sum", dtype, [n] * R, i, [b] * R, o)


def allgather(R: int, n: int, dtype: str = "bf16") -> Naming:
    """Input r is name r; output block j of every rank is name j."""
    i = _segs_cols(np.arange(R), np.zeros(R), np.full(R, n), np.arange(R))
    dd, jj = np.meshgrid(np.arange(R), np.arange(R), indexing="ij")
    o = _segs_cols(dd.ravel(), (jj * n).ravel(), np.full(R * R, n), jj.ravel())
    return Naming(R, "copy", dtype, [n] * R, i, [R * n] * R, o)


def broadcast(R: int, n: int, dtype: str = "bf16", root: int = 0) -> Naming:
    """The root's input is name 0; every rank's output (the root's too) is name 0."""
    i = _segs_cols([root], [0], [n], [0])
    o = _segs_cols(np.arange(R), np.zeros(R), np.full(R, n), np.zeros(R))
    return Naming(R, "copy", dtype, [n] * R, i, [n] * R, o)


def alltoall(R: int, n: int, dtype: str = "bf16") -> Naming:
    """Block d of rank s's input is name s*R+d and lands in block s of rank d's output."""
    assert n % R == 0
    b = n // R
    ss, dd = np.meshgrid(np.arange(R), np.arange(R), indexing="ij")
    name = (ss * R + dd).ravel()
    i = _segs_cols(ss.ravel(), (dd * b).ravel(), np.full(R * R, b), name)
    o = _segs_cols(dd.ravel(), (ss * b).ravel(), np.full(R * R, b), name)
    return Naming(R, "copy", dtype, [n] * R, i, [n] * R, o)


def moe_dispatch(routing: np.ndarray, experts_per_rank: int, hidden: int,
                 dtype: str = "bf16") -> Naming:
    """All-to-all with uneven splits from a routing table [R, T, k] of expert ids.

    Token (s, t) is name s*T+t (its row of `hidden` elements on rank s). It is copied once
    to every rank hosting one of its experts (expert e lives on rank e // experts_per_rank);
    at a destination, rows are ordered by (source rank, source token). meta["counts"] holds
    the rows each rank receives.
    """
    R, T, k = routing.shape
    dest = np.zeros((R, T, R), dtype=bool)
    tok = np.arange(T)
    for s in range(R):
        for j in range(k):
            dest[s, tok, routing[s, :, j] // experts_per_rank] = True
    names = np.arange(R * T)
    i = _segs_cols(np.repeat(np.arange(R), T), np.tile(tok, R) * hidden, np.full(R * T, hidden),
                   names)
    ranks, offs, nms, counts = [], [], [], []
    flat = dest.reshape(R * T, R)  # row = s*T+t in (s, t) order
    for d in range(R):
        rows = np.nonzero(flat[:, d])[0]
        counts.append(len(rows))
        ranks.append(np.full(len(rows), d))
        offs.append(np.arange(len(rows)) * hidden)
        nms.append(rows)
    o = _segs_cols(np.concatenate(ranks), np.concatenate(offs), np.full(sum(counts), hidden),
                   np.concatenate(nms))
    out_len = [max(c, 1) * hidden for c in counts]
    return Naming(R, "copy", dtype, [T * hidden] * R, i, out_len, o,
                  meta={"counts": counts, "dest": dest})


def alltoallv_from_routing(routing: np.ndarray, experts_per_rank: int, hidden: int,
                           dtype: str = "bf16") -> Naming:
    """All-to-all with uneven splits derived from a routing table: the same naming as
    moe_dispatch (one copy of each token row per destination rank)."""
    return moe_dispatch(routing, experts_per_rank, hidden, dtype)


def reduce_to_root(R: int, n: int, dtype: str = "bf16", root: int = 0) -> Naming:
    """Every rank's whole buffer is name 0; only the root's output receives the sum."""
    i = _segs_cols(np.arange(R), np.zeros(R), np.full(R, n), np.zeros(R))
    o = _segs_cols([root], [0], [n], [0])
    return Naming(R, "sum", dtype, [n] * R, i, [n] * R, o)


def gather(R: int, n: int, dtype: str = "bf16", root: int = 0) -> Naming:
    """Input r is name r; block j of the root's output is name j."""
    i = _segs_cols(np.arange(R), np.zeros(R), np.full(R, n), np.arange(R))
    o = _segs_cols(np.full(R, root), np.arange(R) * n, np.full(R, n), np.arange(R))
    return Naming(R, "copy", dtype, [n] * R, i, [R * n] * R, o)


def scatter(R: int, n: int, dtype: str = "bf16", root: int = 0) -> Naming:
    """Block d (of n/R) of the root's input is name d; rank d's output is name d."""
    assert n % R == 0
    b = n // R
    i = _segs_cols(np.full(R, root), np.arange(R) * b, np.full(R, b), np.arange(R))
    o = _segs_cols(np.arange(R), np.zeros(R), np.full(R, b), np.arange(R))
    return Naming(R, "copy", dtype, [n] * R, i, [b] * R, o)


def moe_combine(routing: np.ndarray, experts_per_rank: int, hidden: int,
                dtype: str = "bf16") -> Naming:
    """Reverse of moe_dispatch with a sum: rank d's input holds, in dispatch order, one row
    per token routed to it; token (s, t) (name s*T+t) receives at rank s the sum of its rows
    over the destination ranks, which the fixed (rank, offset) order visits ascending.
    meta["counts"] holds the rows each rank's input has."""
    R, T, k = routing.shape
    disp = moe_dispatch(routing, experts_per_rank, hidden, dtype)
    counts = disp.meta["counts"]
    o_in = disp.out_segs  # dispatch outputs are the combine inputs
    names = np.arange(R * T)
    o = _segs_cols(np.repeat(np.arange(R), T), np.tile(np.arange(T), R) * hidden,
                   np.full(R * T, hidden), names)
    return Naming(R, "sum", dtype, list(disp.out_len), o_in.copy(), [T * hidden] * R, o,
                  meta={"counts": counts, "dest": disp.meta["dest"]})
