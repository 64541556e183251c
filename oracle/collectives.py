"""The collectives written out directly from their definitions (no naming involved).

Each function takes the R per-rank input arrays (uint16 bf16 patterns, float32 or uint8)
and returns the R per-rank output arrays.

* all-reduce: every rank receives the full sum (SiFAR review, Fig. 5 "Oneshot All-Reduce":
  each GPU pulls the whole payload from every peer and reduces it);
* reduce-scatter: rank r receives block r of that sum (SiFAR review, Fig. 6, the first
  step of twoshot, and Fig. 9);
* all-gather: every rank receives the concatenation of all inputs (Fig. 6, second step);
* broadcast: every rank receives the root's input, out of place;
* all-to-all: block d of rank s's input goes to block s of rank d's output;
* MoE dispatch: each token row goes to every rank that hosts one of its experts
  (feed abstracts on expert-parallel routing), one copy per (token, destination rank),
  rows at a destination ordered by (source rank, source token); MoE combine is its reverse
  with a sum over the destinations, in destination-rank order;
* reduce-to-root, gather and scatter: the rooted forms of all-reduce, all-gather and
  all-to-all (the Purlin article counts seven collectives without listing them; these are
  read as the three besides the five named in the workloads).

Sums are the fixed-order binary32 chain of ``oracle.arith.ordered_sum``.
"""

from __future__ import annotations

import numpy as np

from .arith import ordered_sum


def allreduce(xs, dtype):
    s = ordered_sum(list(xs), dtype)
    return [s.copy() for _ in xs]


def reduce_scatter(xs, dtype):
    R = len(xs)
    n = len(xs[0])
    assert n % R == 0
    b = n // R
    return [ordered_sum([x[r * b:(r + 1) * b] for x in xs], dtype) for r in range(R)]


def allgather(xs):
    cat = np.concatenate(list(xs))
    return [cat.copy() for _ in xs]


def broadcast(xs, root=0):
    return [xs[root].copy() for _ in xs]


def alltoall(xs):
    R = len(xs)
    n = len(xs[0])
    assert n % R == 0
    b = n // R
    return [np.concatenate([xs[s][d * b:(d + 1) * b] for s in range(R)]) for d in range(R)]


def reduce_to_root(xs, dtype, root=0):
    """Only the root receives the full sum (the other ranks' outputs are not written:
    returned as None)."""
    s = ordered_sum(list(xs), dtype)
    return [s.copy() if r == root else None for r in range(len(xs))]


def gather(xs, root=0):
    """The root receives the concatenation of all inputs in rank order."""
    cat = np.concatenate(list(xs))
    return [cat.copy() if r == root else None for r in range(len(xs))]


def scatter(xs, root=0):
    """Block d of the root's input goes to rank d."""
    R = len(xs)
    n = len(xs[root])
    assert n % R == 0
    b = n // R
    return [xs[root][d * b:(d + 1) * b].copy() for d in range(R)]


def gemv_payloads(wts, xs):
    """Row-parallel linear layer shards, the payloads of a fused producer: rank r's payload
    is y_r = W_r x_r, with W_r given transposed as wt[r] = [k, n] bf16 and x_r as [k] bf16.

    The pages say only that the all-reduces run inside megakernels, after each layer's
    computation (SiFAR review, Summary); they leave the layer's arithmetic open. The plain
    reading of y = W x is taken: for output j, the k products wt[i, j] * x[i] are each
    rounded to binary32 (exact unless a product leaves binary32's range), then added as ONE
    binary32 chain in row order i = 0..k-1, starting from the first product (round to
    nearest even at every add, no fused multiply-add), and the chain is rounded once to
    bf16. A datapath that adds the products in another order is held to the tolerance of
    ``oracle.tolerance.gemv_within_tolerance``."""
    from .arith import bf16_to_f32, f32_to_bf16_rne
    out = []
    for wt, x in zip(wts, xs):
        w = bf16_to_f32(wt)
        xv = bf16_to_f32(x)
        k = w.shape[0]
        with np.errstate(over="ignore", invalid="ignore"):
            acc = w[0] * xv[0]
            for i in range(1, k):
                acc = acc + w[i] * xv[i]
        out.append(f32_to_bf16_rne(acc))
    return out


def moe_dest_ranks(routing, experts_per_rank):
    """routing [R, T, k] expert ids -> boolean [R, T, R]: token (s,t) goes to rank d."""
    R = routing.shape[0]
    dest = np.zeros((R, routing.shape[1], R), dtype=bool)
    for s in range(R):
        for j in range(routing.shape[2]):
            d = routing[s, :, j] // experts_per_rank
            dest[s, np.arange(routing.shape[1]), d] = True
    return dest


def moe_dispatch(xs, routing, experts_per_rank):
    """xs: R arrays [T, H]. Returns (outputs, counts): outputs[d] is [count_d, H]."""
    R = len(xs)
    dest = moe_dest_ranks(routing, experts_per_rank)
    outs, counts = [], []
    for d in range(R):
        rows = [xs[s][t] for s in range(R) for t in range(xs[s].shape[0]) if dest[s, t, d]]
        counts.append(len(rows))
        H = xs[0].shape[1]
        outs.append(np.stack(rows) if rows else np.zeros((0, H), dtype=xs[0].dtype))
    return outs, counts


def moe_combine_sum(ys, routing, experts_per_rank, dtype):
    """Reverse of dispatch with summation: token (s,t) of rank s receives the fixed-order
    sum, over its destination ranks d ascending, of the row rank d holds for it.
    ys[d] is [count_d, H] in dispatch order."""
    R = len(ys)
    dest = moe_dest_ranks(routing, experts_per_rank)
    T = routing.shape[1]
    pos = [0] * R
    where = {}
    for s in range(R):
        for t in range(T):
            for d in range(R):
                if dest[s, t, d]:
                    where[(s, t, d)] = pos[d]
                    pos[d] += 1
    H = ys[0].shape[1]
    outs = []
    for s in range(R):
        o = np.zeros((T, H), dtype=ys[0].dtype)
        for t in range(T):
            terms = [ys[d][where[(s, t, d)]] for d in range(R) if dest[s, t, d]]
            o[t] = ordered_sum(terms, dtype)
        outs.append(o)
    return outs
