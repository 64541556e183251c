"""Pins for the CPU oracle: closed forms, invariants, hand-worked fixtures, brute force.

Nothing here touches the CUDA library. Each test fixes a property that the pages or plain
mathematics determine, so that a plausible slip in the oracle (a dropped term, a reversed
order, a transposed block, a wrong rounding) fails at least one of them.
"""

import os
import struct
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import arith, brute, collectives, naming
import synth

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden")


# ---------------------------------------------------------------- element arithmetic

def test_bf16_widening_is_exact_for_every_pattern():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    f = arith.bf16_to_f32(bits)
    for b in range(0, 1 << 16, 97):
        e = (b >> 7) & 0xFF
        if e == 0xFF:
            continue
        v = brute.decode_bf16(b)
        got = Fraction(float(f[b]))
        assert got == v.q, hex(b)
        if v.q == 0:
            assert (struct.pack("<f", float(f[b]))[3] >> 7) == v.neg


def test_bf16_rounding_matches_exact_rule_including_ties():
    rng = synth.seeded_rng(11)
    hi = rng.integers(0, 0x7F7F, size=4000, dtype=np.uint32)
    lo = rng.integers(0, 1 << 16, size=4000, dtype=np.uint32)
    lo[:1000] = 0x8000  # exact ties
    lo[1000:1500] = 0x7FFF
    lo[1500:2000] = 0x8001
    sign = rng.integers(0, 2, size=4000, dtype=np.uint32) << np.uint32(31)
    u = sign | (hi << np.uint32(16)) | lo
    x = u.view(np.float32)
    got = arith.f32_to_bf16_rne(x)
    for i in range(0, 4000, 3):
        want = brute.round_bf16(brute.decode_f32(int(u[i])))
        gotv = brute.decode_bf16(int(got[i]))
        assert gotv.key() == want.key(), (hex(int(u[i])), hex(int(got[i])))


def test_bf16_rounding_nan_stays_nan():
    x = np.array([np.nan, -np.nan], dtype=np.float32)
    r = arith.f32_to_bf16_rne(x)
    assert np.all(np.isnan(arith.bf16_to_f32(r)))


def test_two_term_f32_sum_equals_host_fpu():
    # fl32(a+b) through binary64 is exact (53 >= 2*24+2: double rounding is innocuous)
    rng = synth.seeded_rng(12)
    a = synth.uniform_f32(rng, 3000)
    b = synth.uniform_f32(rng, 3000) * np.float32(1e-3)
    got = arith.ordered_sum([a, b], "f32")
    for i in range(3000):
        want = struct.unpack("<f", struct.pack("<f", float(a[i]) + float(b[i])))[0]
        assert struct.pack("<f", want) == struct.pack("<f", float(got[i]))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("R", [2, 3, 5, 8])
def test_ordered_sum_matches_exact_sequential_rounding(dtype, R):
    rng = synth.seeded_rng(100 + R)
    n = 300
    if dtype == "bf16":
        xs = [synth.normal_bf16(rng, n) for _ in range(R)]
        dec = brute.decode_bf16
        raw = lambda x, i: int(x[i])
    else:
        # magnitudes spread over many binades so that the order of additions matters
        xs = [synth.uniform_f32(rng, n) * np.float32(2.0) ** rng.integers(-12, 12, n).astype(np.float32)
              for _ in range(R)]
        dec = brute.decode_f32
        raw = lambda x, i: int(x.view(np.uint32)[i])
    got = arith.ordered_sum(xs, dtype)
    gdec = (lambda i: brute.decode_bf16(int(got[i]))) if dtype == "bf16" else \
        (lambda i: brute.decode_f32(int(got.view(np.uint32)[i])))
    for i in range(n):
        want = brute.element_sum([dec(raw(x, i)) for x in xs], dtype)
        assert gdec(i).key() == want.key(), i


def test_fixed_order_is_observable():
    # a reversed chain must give a different answer on this data (pins the order)
    rng = synth.seeded_rng(7)
    xs = [synth.uniform_f32(rng, 2000) * np.float32(2.0) ** np.float32(k * 6) for k in range(4)]
    fwd = arith.ordered_sum(xs, "f32")
    rev = arith.ordered_sum(xs[::-1], "f32")
    assert not np.array_equal(fwd.view(np.uint32), rev.view(np.uint32))


def _read_sum_fixtures():
    rows = []
    with open(os.path.join(GOLDEN, "sum_rounding.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            dtype, ins, out, why = [p.strip() for p in line.split(";", 3)]
            rows.append((dtype, [int(h, 16) for h in ins.split()], int(out, 16), why))
    return rows


@pytest.mark.parametrize("row", _read_sum_fixtures(), ids=lambda r: r[3][:40])
def test_golden_sum_rounding(row):
    dtype, ins, out, why = row
    R = len(ins)
    npt = np.uint16 if dtype == "bf16" else np.uint32
    xs = [np.array([v], dtype=npt) for v in ins]
    if dtype == "f32":
        xs = [x.view(np.float32) for x in xs]
    outs = [np.zeros(1, dtype=xs[0].dtype) for _ in range(R)]
    code = naming.run_naming(R, "sum", dtype, [1] * R, [(r, 0, 1, 0) for r in range(R)],
                             [1] * R, [(r, 0, 1, 0) for r in range(R)], xs, outs)
    assert code == 0
    for r in range(R):
        got = int(outs[r].view(npt)[0])
        assert got == out, (why, hex(got))
    dec = brute.decode_bf16 if dtype == "bf16" else brute.decode_f32
    want = brute.element_sum([dec(v) for v in ins], dtype)
    assert dec(out).key() == want.key(), why


# ---------------------------------------------------------------- naming semantics

def _naming_case(seed, op, dtype, R):
    rng = synth.seeded_rng(seed)
    in_len, in_segs, out_len, out_segs = synth.random_naming(rng, R, 12, 4, 3, op)
    if dtype == "bf16":
        ins = [synth.normal_bf16(rng, n) for n in in_len]
        outs = [synth.normal_bf16(rng, n) for n in out_len]
    elif dtype == "f32":
        ins = [synth.uniform_f32(rng, n) * np.float32(2.0) ** rng.integers(-8, 8, n).astype(np.float32)
               for n in in_len]
        outs = [synth.uniform_f32(rng, n) for n in out_len]
    else:
        ins = [synth.random_bytes(rng, n) for n in in_len]
        outs = [synth.random_bytes(rng, n) for n in out_len]
    return in_len, in_segs, out_len, out_segs, ins, outs


def _raw(a, i):
    if a.dtype == np.float32:
        return int(a.view(np.uint32)[i])
    return int(a[i])


@pytest.mark.parametrize("seed", range(40))
@pytest.mark.parametrize("op,dtype", [("copy", "bf16"), ("copy", "bytes"), ("copy", "f32"),
                                      ("sum", "bf16"), ("sum", "f32")])
def test_naming_matches_brute_force(seed, op, dtype):
    R = 1 + seed % 3
    in_len, in_segs, out_len, out_segs, ins, outs = _naming_case(1000 + seed, op, dtype, R)
    before = [o.copy() for o in outs]
    code = naming.run_naming(R, op, dtype, in_len, in_segs, out_len, out_segs, ins, outs)
    assert code == 0
    raw_in = [[_raw(x, i) for i in range(len(x))] for x in ins]
    want = brute.evaluate(op, dtype, in_segs, out_segs, raw_in, out_len)
    dec = brute.decode_bf16 if dtype == "bf16" else brute.decode_f32
    for d in range(R):
        for i in range(out_len[d]):
            if i in want[d]:
                w = want[d][i]
                if op == "copy":
                    assert _raw(outs[d], i) == w
                else:
                    assert dec(_raw(outs[d], i)).key() == w.key()
            else:
                assert _raw(outs[d], i) == _raw(before[d], i), "unnamed element touched"


def test_validation_codes():
    E = naming.ERR
    ok_in = [(0, 0, 4, 7), (1, 0, 4, 7)]
    ok_out = [(0, 0, 4, 7), (1, 0, 4, 7)]
    v = lambda R=2, op="sum", dt="bf16", il=(4, 4), i=ok_in, ol=(4, 4), o=ok_out: \
        naming.validate(R, op, dt, list(il), i, list(ol), o)
    assert v() == E["OK"]
    assert v(R=0, il=(), ol=(), i=[], o=[]) == E["EINVAL"]
    assert v(R=65, il=[4] * 65, ol=[4] * 65) == E["EINVAL"]
    assert v(op="max") == E["EINVAL"]
    assert v(dt="bytes") == E["EINVAL"]
    assert v(i=[(2, 0, 4, 7)]) == E["EINVAL"]
    assert v(i=[(0, 0, 0, 7)], o=[]) == E["EINVAL"]
    assert v(i=[(0, 1, 4, 7), (1, 0, 4, 7)]) == E["EBOUNDS"]
    assert v(o=[(1, 2, 4, 7)]) == E["EBOUNDS"]
    assert v(i=[(0, 0, 4, 7), (1, 0, 3, 7)]) == E["ELEN"]
    assert v(o=[(0, 0, 4, 8)]) == E["ENAME"]
    assert v(op="copy") == E["ENAME"]
    assert v(op="copy", i=[(0, 0, 4, 7)]) == E["OK"]
    assert v(ol=(8, 4), o=[(0, 0, 4, 7), (0, 3, 4, 7)]) == E["EOVERLAP"]
    assert v(ol=(8, 4), o=[(0, 0, 4, 7), (0, 4, 4, 7)]) == E["OK"]
    # an input name nobody consumes is allowed
    assert v(i=ok_in + [(0, 0, 2, 9)]) == E["OK"]
    # empty naming is valid and writes nothing
    assert v(i=[], o=[]) == E["OK"]


# ---------------------------------------------------------------- collectives

def _ar_naming(R, n):
    return [(r, 0, n, 0) for r in range(R)], [(r, 0, n, 0) for r in range(R)]


def _run(R, op, dtype, in_len, in_segs, out_len, out_segs, ins):
    npt = arith.NPTYPE[dtype]
    outs = [np.zeros(n, dtype=npt) for n in out_len]
    assert naming.run_naming(R, op, dtype, in_len, in_segs, out_len, out_segs, ins, outs) == 0
    return outs


def _eq(a, b):
    return np.array_equal(np.asarray(a).view(np.uint8), np.asarray(b).view(np.uint8))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_allreduce_direct_equals_naming_and_rs_then_ag(dtype):
    R, n = 8, 64
    rng = synth.seeded_rng(21)
    xs = [synth.normal_bf16(rng, n) if dtype == "bf16" else synth.normal_f32(rng, n) for _ in range(R)]
    direct = collectives.allreduce(xs, dtype)
    i, o = _ar_naming(R, n)
    named = _run(R, "sum", dtype, [n] * R, i, [n] * R, o, xs)
    rs = collectives.reduce_scatter(xs, dtype)
    ag = collectives.allgather(rs)
    for r in range(R):
        assert _eq(direct[r], named[r])
        assert _eq(direct[r], ag[r])


def test_reduce_scatter_alltoall_allgather_broadcast_by_naming():
    R, n = 4, 16
    b = n // R
    rng = synth.seeded_rng(22)
    xs = [synth.normal_bf16(rng, n) for _ in range(R)]
    # reduce-scatter: input block j on every rank is name j; rank r's output is name r
    rs = _run(R, "sum", "bf16", [n] * R, [(r, j * b, b, j) for r in range(R) for j in range(R)],
              [b] * R, [(r, 0, b, r) for r in range(R)], xs)
    for r, (x, y) in enumerate(zip(rs, collectives.reduce_scatter(xs, "bf16"))):
        assert _eq(x, y)
    # all-gather: input r is name r; output block j is name j
    ag = _run(R, "copy", "bf16", [n] * R, [(r, 0, n, r) for r in range(R)],
              [R * n] * R, [(d, j * n, n, j) for d in range(R) for j in range(R)], xs)
    for x, y in zip(ag, collectives.allgather(xs)):
        assert _eq(x, y)
    # broadcast from root 2
    bc = _run(R, "copy", "bf16", [n] * R, [(2, 0, n, 0)], [n] * R, [(d, 0, n, 0) for d in range(R)], xs)
    for x, y in zip(bc, collectives.broadcast(xs, 2)):
        assert _eq(x, y)
    # all-to-all: (source s, block d) is name s*R+d; it lands at (rank d, block s)
    a2a = _run(R, "copy", "bf16", [n] * R, [(s, d * b, b, s * R + d) for s in range(R) for d in range(R)],
               [n] * R, [(d, s * b, b, s * R + d) for s in range(R) for d in range(R)], xs)
    for x, y in zip(a2a, collectives.alltoall(xs)):
        assert _eq(x, y)


def test_alltoall_twice_is_identity_and_conserves_bytes():
    R, n = 8, 64
    rng = synth.seeded_rng(23)
    xs = [synth.random_bytes(rng, n) for _ in range(R)]
    once = collectives.alltoall(xs)
    twice = collectives.alltoall(once)
    for x, y in zip(xs, twice):
        assert _eq(x, y)
    assert sorted(np.concatenate(xs).tolist()) == sorted(np.concatenate(once).tolist())
    # a2a is a transpose of the (source, block) grid: the block grid must move
    assert not all(_eq(x, y) for x, y in zip(xs, once))


def test_broadcast_single_rank_is_memcpy_and_allgather_conserves():
    rng = synth.seeded_rng(24)
    x = synth.random_bytes(rng, 33)
    assert _eq(collectives.broadcast([x])[0], x)
    xs = [synth.random_bytes(rng, 5) for _ in range(3)]
    ag = collectives.allgather(xs)
    for out in ag:
        for r in range(3):
            assert _eq(out[r * 5:(r + 1) * 5], xs[r])


def test_single_producer_sum_is_copy():
    rng = synth.seeded_rng(25)
    x = synth.normal_bf16(rng, 50)
    assert _eq(collectives.allreduce([x], "bf16")[0], x)
    y = synth.normal_f32(rng, 50)
    assert _eq(collectives.allreduce([y], "f32")[0], y)


@pytest.mark.parametrize("k", [1, 2, 3, 5, 8])
def test_identical_inputs_closed_form(k):
    # k copies of a bf16 value x: the binary32 chain is exact (8+3 significand bits), so the
    # result is k*x rounded once to bf16 -- computed here with exact rationals
    rng = synth.seeded_rng(26)
    x = synth.normal_bf16(rng, 200)
    out = collectives.allreduce([x] * k, "bf16")[0]
    for i in range(200):
        v = brute.decode_bf16(int(x[i]))
        want = brute.round_bf16(brute.Val(v.q * k, neg=v.neg))
        assert brute.decode_bf16(int(out[i])).key() == want.key()


def test_small_integer_sums_are_exact():
    R, n = 8, 500
    rng = synth.seeded_rng(27)
    xs = [synth.small_int_bf16(rng, n) for _ in range(R)]
    out = collectives.allreduce(xs, "bf16")[0]
    ints = sum(arith.bf16_to_f32(x).astype(np.int64) for x in xs)
    assert np.array_equal(arith.bf16_to_f32(out).astype(np.int64), ints)
    # sums within +-128 are exact in bf16 too, and independent of order
    rev = collectives.allreduce(xs[::-1], "bf16")[0]
    assert _eq(out, rev)


def test_moe_dispatch_golden_fixture():
    routing = np.zeros((2, 2, 2), dtype=np.int32)
    expect = {}
    with open(os.path.join(GOLDEN, "moe_dispatch_tiny.txt")) as f:
        for line in f:
            line = line.strip()
            if line.startswith("routing"):
                lhs, rhs = line.split(":")
                s = int(lhs.split("s=")[1].split()[0])
                t = int(lhs.split("t=")[1].split()[0])
                routing[s, t] = [int(v) for v in rhs.split()]
            elif line.startswith("expect"):
                lhs, rhs = line.split(":")
                expect[int(lhs.split("d=")[1])] = [int(v) for v in rhs.split()]
    xs = [np.array([[100 * s + t] for t in range(2)], dtype=np.int64) for s in range(2)]
    outs, counts = collectives.moe_dispatch(xs, routing, 2)
    for d in range(2):
        assert outs[d][:, 0].tolist() == expect[d]
        assert counts[d] == len(expect[d])


def test_moe_dispatch_counts_and_rows():
    R, T, H, E, k = 4, 64, 8, 32, 4
    routing = synth.zipf_topk_routing(5, R, T, E, k, 1.1)
    assert routing.shape == (R, T, k)
    for s in range(R):
        for t in range(T):
            assert len(set(routing[s, t].tolist())) == k
    rng = synth.seeded_rng(5)
    xs = [synth.random_bytes(rng, (T, H)) for _ in range(R)]
    outs, counts = collectives.moe_dispatch(xs, routing, E // R)
    dests = collectives.moe_dest_ranks(routing, E // R)
    assert sum(counts) == int(dests.sum())
    for d in range(R):
        want = [xs[s][t] for s in range(R) for t in range(T) if set(routing[s, t] // (E // R)) & {d}]
        assert len(want) == counts[d]
        for a, b in zip(outs[d], want):
            assert _eq(a, b)


def test_moe_combine_inverts_dispatch_for_single_destination_tokens():
    R, T, H, E, k = 2, 8, 4, 4, 1
    routing = synth.zipf_topk_routing(9, R, T, E, k, 1.1)
    rng = synth.seeded_rng(9)
    xs = [synth.normal_bf16(rng, (T, H)) for _ in range(R)]
    ys, _ = collectives.moe_dispatch(xs, routing, E // R)
    back = collectives.moe_combine_sum(ys, routing, E // R, "bf16")
    for s in range(R):
        assert _eq(back[s], xs[s])


def test_epoch_semantics_cycle_through_pool():
    R, n = 2, 8
    rng = synth.seeded_rng(31)
    pool = [[synth.normal_bf16(rng, n) for _ in range(R)] for _ in range(3)]
    i, o = _ar_naming(R, n)
    res = naming.run_epochs(R, "sum", "bf16", [n] * R, i, [n] * R, o, pool, 7,
                            [np.zeros(n, np.uint16)] * R)
    for e in range(7):
        want = collectives.allreduce(pool[e % 3], "bf16")
        for r in range(R):
            assert _eq(res[e][r], want[r])


def test_rooted_collectives_against_their_all_forms():
    R, n = 4, 32
    rng = synth.seeded_rng(60)
    xs = [synth.normal_bf16(rng, n) for _ in range(R)]
    for root in range(R):
        red = collectives.reduce_to_root(xs, "bf16", root)
        assert _eq(red[root], collectives.allreduce(xs, "bf16")[0])
        assert all(red[r] is None for r in range(R) if r != root)
        g = collectives.gather(xs, root)
        assert _eq(g[root], collectives.allgather(xs)[0])
        sc = collectives.scatter(xs, root)
        # scatter then gather at the same root is the identity on the root's input
        assert _eq(collectives.gather(sc, root)[root], xs[root])
        # scatter is the root's row of an all-to-all
        a2a = collectives.alltoall(xs)
        for d in range(R):
            assert _eq(sc[d], a2a[d][root * (n // R):(root + 1) * (n // R)])


def test_rooted_collectives_by_naming():
    R, n = 3, 12
    b = n // R
    rng = synth.seeded_rng(61)
    xs = [synth.normal_bf16(rng, n) for _ in range(R)]
    root = 1
    red = _run(R, "sum", "bf16", [n] * R, [(r, 0, n, 0) for r in range(R)], [n] * R,
               [(root, 0, n, 0)], xs)
    assert _eq(red[root], collectives.reduce_to_root(xs, "bf16", root)[root])
    g = _run(R, "copy", "bf16", [n] * R, [(r, 0, n, r) for r in range(R)], [R * n] * R,
             [(root, j * n, n, j) for j in range(R)], xs)
    assert _eq(g[root], collectives.gather(xs, root)[root])
    sc = _run(R, "copy", "bf16", [n] * R, [(root, d * b, b, d) for d in range(R)], [b] * R,
              [(d, 0, b, d) for d in range(R)], xs)
    for d in range(R):
        assert _eq(sc[d], collectives.scatter(xs, root)[d])


def test_moe_combine_is_the_ordered_sum_over_destinations():
    R, T, H, E, k = 4, 16, 4, 16, 3
    routing = synth.zipf_topk_routing(12, R, T, E, k, 1.1)
    rng = synth.seeded_rng(12)
    # destination buffers hold arbitrary rows (as after an expert computation)
    dests = collectives.moe_dest_ranks(routing, E // R)
    counts = [int(dests[:, :, d].sum()) for d in range(R)]
    ys = [synth.normal_bf16(rng, (c, H)) for c in counts]
    out = collectives.moe_combine_sum(ys, routing, E // R, "bf16")
    # brute force: walk the dispatch order and sum by hand in destination order
    pos = [0] * R
    rowsof = {}
    for s_ in range(R):
        for t in range(T):
            for d in range(R):
                if dests[s_, t, d]:
                    rowsof.setdefault((s_, t), []).append(ys[d][pos[d]])
                    pos[d] += 1
    for s_ in range(R):
        for t in range(T):
            rows = rowsof[(s_, t)]
            for h in range(H):
                want = brute.element_sum([brute.decode_bf16(int(r[h])) for r in rows], "bf16")
                assert brute.decode_bf16(int(out[s_][t, h])).key() == want.key()


# ---------------------------------------------------------------- tolerance (other orders)

def _other_order_sum(terms, dtype, order):
    """A fp32 sum in another order, written out here to exercise the tolerance."""
    vals = [arith.to_f32(t, dtype) for t in terms]
    if order == "reversed":
        vals = vals[::-1]
    if order == "tree":
        while len(vals) > 1:
            vals = [vals[i] + vals[i + 1] if i + 1 < len(vals) else vals[i]
                    for i in range(0, len(vals), 2)]
        acc = vals[0]
    else:
        acc = vals[0].copy()
        for v in vals[1:]:
            acc = acc + v
    return arith.f32_to_bf16_rne(acc) if dtype == "bf16" else acc


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("order", ["rank", "reversed", "tree"])
def test_any_summation_order_is_within_tolerance(dtype, order):
    from oracle import tolerance
    rng = synth.seeded_rng(300)
    for R in (2, 3, 8, 17):
        xs = [synth.normal_bf16(rng, 4000) if dtype == "bf16" else
              synth.normal_f32(rng, 4000) * np.float32(2.0) ** rng.integers(-20, 20, 4000).astype(np.float32)
              for _ in range(R)]
        got = _other_order_sum(xs, dtype, order) if order != "rank" else arith.ordered_sum(xs, dtype)
        assert tolerance.within_tolerance(got, xs, dtype).all(), (R, order)


def test_tolerance_rejects_real_errors():
    from oracle import tolerance
    rng = synth.seeded_rng(301)
    xs = [synth.normal_bf16(rng, 4000) for _ in range(8)]
    good = arith.ordered_sum(xs, "bf16")
    # two bf16 ulps off: rejected wherever the exact sum is not tiny against sum |x|
    bad = (good.astype(np.int32) + 2).astype(np.uint16)
    ok = tolerance.within_tolerance(bad, xs, "bf16")
    s = np.abs(tolerance.exact_sum(xs, "bf16"))
    S = np.sum([np.abs(arith.bf16_to_f32(x)) for x in xs], axis=0)
    assert not ok[s > S / 8].any()
    # a dropped term is rejected almost everywhere
    dropped = arith.ordered_sum(xs[:-1], "bf16")
    assert tolerance.within_tolerance(dropped, xs, "bf16").mean() < 0.1
    # fp32: one part in 1e5 is far outside
    ys = [synth.normal_f32(rng, 4000) for _ in range(8)]
    g32 = arith.ordered_sum(ys, "f32")
    assert not tolerance.within_tolerance(g32 * np.float32(1 + 1e-5), ys, "f32")[
        np.abs(g32) > 1.0].any()


# ---------------------------------------------------------------- fused producer (GEMV)

def _brute_gemv_chain(wt, x, j, order):
    """Output j of y = W x by exact rational arithmetic: products exact, then the binary32
    chain over the rows in the given order, from the first product; one bf16 rounding."""
    prods = [brute.Val(brute.decode_bf16(int(wt[i, j])).q * brute.decode_bf16(int(x[i])).q,
                       neg=brute.decode_bf16(int(wt[i, j])).neg != brute.decode_bf16(int(x[i])).neg)
             for i in order]
    acc = prods[0]
    for p in prods[1:]:
        acc = brute.add(acc, p, brute.round_f32)
    return brute.round_bf16(acc)


GEMV_PIN_SHAPES = ((8, 8), (16, 16), (24, 8), (5, 8), (64, 24), (32, 32))


def _order_sensitive_gemv():
    """k = 16 rows against x = 1: column j holds 2^24 at row a_j, -2^24 at row b_j and ones
    elsewhere. In binary32, 2^24 + 1 rounds back to 2^24 (a tie, to even) while -2^24 + 1 is
    exact, so the result depends on where the large terms fall in the adding order: the
    plain chain, its reverse and an eight-block order all give different values."""
    k = 16
    pos = [(0, 15), (15, 0), (0, 1), (7, 8), (3, 12), (14, 2)]
    wt = np.full((k, len(pos)), 0x3F80, dtype=np.uint16)        # 1.0
    for j, (a, b) in enumerate(pos):
        wt[a, j], wt[b, j] = 0x4B80, 0xCB80                     # 2^24, -2^24
    return wt, np.full(k, 0x3F80, dtype=np.uint16)


def _gemv_pin_cases():
    rng = synth.seeded_rng(400)
    cases = [(synth.normal_bf16(rng, (k, n)), synth.normal_bf16(rng, k)) for k, n in GEMV_PIN_SHAPES]
    return cases + [_order_sensitive_gemv()]


def test_gemv_payload_matches_exact_rational_evaluation():
    # the plain definition of y = W x, evaluated independently: k products, one chain in row
    # order; square shapes make a transposed operand visible too
    for wt, x in _gemv_pin_cases():
        k, n = wt.shape
        y = collectives.gemv_payloads([wt], [x])[0]
        for j in range(n):
            want = _brute_gemv_chain(wt, x, j, range(k))
            assert brute.decode_bf16(int(y[j])).key() == want.key(), (k, n, j)


def test_gemv_row_order_is_observable():
    # On the pins' data, the row order decides bits: the reversed chain and a chain taken in
    # eight consecutive blocks (then the block sums in order) each differ from the plain chain
    # somewhere, so the exact-rational pin above fixes the order, not only the value.
    diff_rev = diff_blk = False
    for wt, x in _gemv_pin_cases():
        k, n = wt.shape
        if k % 8:
            continue
        kb = k // 8
        for j in range(n):
            plain = _brute_gemv_chain(wt, x, j, range(k)).key()
            diff_rev |= _brute_gemv_chain(wt, x, j, range(k - 1, -1, -1)).key() != plain
            prods = [brute.Val(brute.decode_bf16(int(wt[i, j])).q * brute.decode_bf16(int(x[i])).q)
                     for i in range(k)]
            tot = None
            for b in range(8):
                acc = prods[b * kb]
                for p in prods[b * kb + 1:(b + 1) * kb]:
                    acc = brute.add(acc, p, brute.round_f32)
                tot = acc if tot is None else brute.add(tot, acc, brute.round_f32)
            diff_blk |= brute.round_bf16(tot).key() != plain
    assert diff_rev and diff_blk


def test_gemv_payload_closed_forms():
    rng = synth.seeded_rng(401)
    k = n = 32
    x = synth.normal_bf16(rng, k)
    perm = rng.permutation(n)
    one = np.uint16(0x3F80)
    wt = np.zeros((k, n), dtype=np.uint16)
    wt[np.arange(k), perm] = one           # column perm[i] picks x[i]
    y = collectives.gemv_payloads([wt], [x])[0]
    # zero products add exactly; a product's sign of zero can differ only for zero inputs
    nz = (x & 0x7FFF) != 0
    assert np.array_equal(y[perm][nz], x[nz])
    # scaling every weight by 2 doubles every output exactly (no overflow at these sizes)
    wt2 = synth.small_int_bf16(rng, (k, n), lim=3)
    y1 = collectives.gemv_payloads([wt2], [x])[0]
    wt3 = arith.f32_to_bf16_rne(arith.bf16_to_f32(wt2) * np.float32(2))
    y2 = collectives.gemv_payloads([wt3], [x])[0]
    assert np.array_equal(arith.bf16_to_f32(y2), arith.bf16_to_f32(y1) * np.float32(2))
    # small integers: every product and partial sum is exact, so y is the integer dot
    # product (rounded to bf16 once), whatever the order
    wi = synth.small_int_bf16(rng, (k, n), lim=4)
    xi = synth.small_int_bf16(rng, k, lim=4)
    dot = arith.bf16_to_f32(wi).astype(np.int64).T @ arith.bf16_to_f32(xi).astype(np.int64)
    yi = collectives.gemv_payloads([wi], [xi])[0]
    assert np.array_equal(yi, arith.f32_to_bf16_rne(dot.astype(np.float32)))
    # every product -0 (weights -0, x >= +0): the chain starts from its first product, so
    # -0 + -0 + ... stays -0 (a chain from +0.0 would give +0)
    wz = np.full((k, n), 0x8000, dtype=np.uint16)
    xp = (x & np.uint16(0x7FFF)).astype(np.uint16)
    assert np.all(collectives.gemv_payloads([wz], [xp])[0] == 0x8000)


def _blocked_gemv(wt, x, blocks):
    """y = W x with the k products added in `blocks` consecutive blocks (each a binary32
    chain from its first product), the block sums then added in block order: an alternative
    order, written out here to exercise the tolerance."""
    w, xv = arith.bf16_to_f32(wt), arith.bf16_to_f32(x)
    kb = w.shape[0] // blocks
    tot = None
    for b in range(blocks):
        acc = w[b * kb] * xv[b * kb]
        for i in range(b * kb + 1, (b + 1) * kb):
            acc = acc + w[i] * xv[i]
        tot = acc if tot is None else tot + acc
    return arith.f32_to_bf16_rne(tot)


@pytest.mark.parametrize("blocks", [1, 8, 64])
def test_gemv_other_orders_are_within_tolerance(blocks):
    from oracle import tolerance
    rng = synth.seeded_rng(403)
    k, n, R = 512, 700, 4
    wts = [synth.normal_bf16(rng, (k, n)) for _ in range(R)]
    xs = [synth.normal_bf16(rng, k) for _ in range(R)]
    ys = [_blocked_gemv(w, x, blocks) for w, x in zip(wts, xs)]
    for w, x, y in zip(wts, xs, ys):
        assert tolerance.gemv_within_tolerance(y, w, x).all()
    s = arith.ordered_sum(ys, "bf16")
    assert tolerance.gemv_sum_within_tolerance(s, wts, xs).all()
    # under heavy cancellation (2^24 - 2^24 plus small terms) the orders give values far
    # apart in relative terms, all within the accumulation term of the bound
    w, x = _order_sensitive_gemv()
    for y in (collectives.gemv_payloads([w], [x])[0], _blocked_gemv(w, x, min(blocks, 16)),
              collectives.gemv_payloads([w[::-1].copy()], [x[::-1].copy()])[0]):
        assert tolerance.gemv_within_tolerance(y, w, x).all()


def test_gemv_tolerance_rejects_real_errors():
    from oracle import tolerance
    rng = synth.seeded_rng(404)
    k, n, R = 256, 600, 4
    wts = [synth.normal_bf16(rng, (k, n)) for _ in range(R)]
    xs = [synth.normal_bf16(rng, k) for _ in range(R)]
    ys = collectives.gemv_payloads(wts, xs)
    w, x, y = wts[0], xs[0], ys[0]
    p = arith.bf16_to_f32(w).astype(np.float64) * arith.bf16_to_f32(x).astype(np.float64)[:, None]
    big = np.abs(p.sum(axis=0)) > np.abs(p).sum(axis=0) / 8
    # three bf16 ulps off: rejected wherever the exact value is not tiny against sum |p|
    bad = (y.astype(np.int32) + 3).astype(np.uint16)
    assert not tolerance.gemv_within_tolerance(bad, w, x)[big].any()
    # the last row dropped, the weights transposed (square), a sign flipped: rejected
    # almost everywhere
    dropped = collectives.gemv_payloads([w[:-1]], [x[:-1]])[0]
    assert tolerance.gemv_within_tolerance(dropped, w, x).mean() < 0.2
    ws = synth.normal_bf16(rng, (k, k))
    yt = collectives.gemv_payloads([np.ascontiguousarray(ws.T)], [x])[0]
    assert tolerance.gemv_within_tolerance(yt, ws, x).mean() < 0.05
    assert tolerance.gemv_within_tolerance(y ^ np.uint16(0x8000), w, x).mean() < 0.05
    # over ranks: a rank dropped, or the sum three ulps off, is rejected
    s = arith.ordered_sum(ys, "bf16")
    assert tolerance.gemv_sum_within_tolerance(s, wts, xs).all()
    assert tolerance.gemv_sum_within_tolerance(arith.ordered_sum(ys[:-1], "bf16"),
                                               wts, xs).mean() < 0.2
    t = np.sum([(arith.bf16_to_f32(a).astype(np.float64) *
                 arith.bf16_to_f32(b).astype(np.float64)[:, None]).sum(axis=0)
                for a, b in zip(wts, xs)], axis=0)
    Sy = np.sum([np.abs(arith.bf16_to_f32(v)) for v in ys], axis=0)
    # (each payload may sit one rounding away from the plain one, so the sum over four
    # ranks may move by a few ulps; eight is outside)
    bad_s = (s.astype(np.int32) + 8).astype(np.uint16)
    assert not tolerance.gemv_sum_within_tolerance(bad_s, wts, xs)[np.abs(t) > Sy / 2].any()


def test_gemv_tolerance_compares_special_values_by_class():
    # a product that overflows binary32 makes the payload infinite in any order
    from oracle import tolerance
    rng = synth.seeded_rng(405)
    k, n = 16, 8
    w = synth.normal_bf16(rng, (k, n))
    x = synth.normal_bf16(rng, k)
    w[3, 2], x[3] = 0x7F00, 0x7F00            # 2^127 * 2^127 overflows
    y = collectives.gemv_payloads([w], [x])[0]
    assert y[2] == 0x7F80
    ok = tolerance.gemv_within_tolerance(y, w, x)
    assert ok.all()
    assert not tolerance.gemv_within_tolerance(np.where(np.arange(n) == 2, 0x7F7F, y)
                                               .astype(np.uint16), w, x)[2]
