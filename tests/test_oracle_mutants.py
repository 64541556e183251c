"""Plant plausible mistakes in the oracle (on the CPU) and check the pins catch each one.

Each mutant replaces one piece of the oracle's arithmetic or layout logic with a subtly
wrong version; at least one pin (hand-worked fixtures, exact-rational brute force, direct
definitions, closed forms) must then fail. This shows the pins constrain the oracle rather
than merely agreeing with it.
"""

import numpy as np
import pytest

from oracle import arith, brute, collectives, naming
import synth

import test_oracle as pins


def _golden_ok():
    try:
        for row in pins._read_sum_fixtures():
            pins.test_golden_sum_rounding(row)
    except AssertionError:
        return False
    return True


def _brute_ok():
    try:
        for seed in range(12):
            for op, dt in (("sum", "bf16"), ("sum", "f32"), ("copy", "bf16")):
                pins.test_naming_matches_brute_force(seed, op, dt)
        for dt in ("bf16", "f32"):
            for R in (3, 8):
                pins.test_ordered_sum_matches_exact_sequential_rounding(dt, R)
    except AssertionError:
        return False
    return True


def _collectives_ok():
    try:
        pins.test_allreduce_direct_equals_naming_and_rs_then_ag("bf16")
        pins.test_reduce_scatter_alltoall_allgather_broadcast_by_naming()
        pins.test_alltoall_twice_is_identity_and_conserves_bytes()
        for k in (3, 8):
            pins.test_identical_inputs_closed_form(k)
        pins.test_small_integer_sums_are_exact()
        pins.test_moe_dispatch_golden_fixture()
    except AssertionError:
        return False
    return True


def _all_pins_pass():
    return _golden_ok() and _brute_ok() and _collectives_ok()


def test_unmutated_oracle_passes_every_pin():
    assert _all_pins_pass()


def _reversed_sum(terms, dtype):
    return ORIG_SUM(list(terms)[::-1], dtype)


def _dropped_last(terms, dtype):
    t = list(terms)
    return ORIG_SUM(t[:-1] if len(t) > 1 else t, dtype)


def _bf16_each_step(terms, dtype):
    if dtype != "bf16":
        return ORIG_SUM(terms, dtype)
    acc = arith.bf16_to_f32(terms[0]).copy()
    for t in terms[1:]:
        acc = arith.bf16_to_f32(arith.f32_to_bf16_rne(acc + arith.bf16_to_f32(t)))
    return arith.f32_to_bf16_rne(acc)


def _start_from_plus_zero(terms, dtype):
    acc = np.zeros(len(terms[0]), dtype=np.float32)
    for t in terms:
        acc = acc + arith.to_f32(t, dtype)
    return arith.f32_to_bf16_rne(acc) if dtype == "bf16" else acc


def _truncate_bf16(x):
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return (u >> np.uint32(16)).astype(np.uint16)


def _round_half_up_bf16(x):
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    with np.errstate(over="ignore"):
        return ((u + np.uint32(0x8000)) >> np.uint32(16)).astype(np.uint16)


ORIG_SUM = arith.ordered_sum
ORIG_RNE = arith.f32_to_bf16_rne

SUM_MUTANTS = {"reversed order": _reversed_sum, "dropped term": _dropped_last,
               "bf16 rounding after every add": _bf16_each_step,
               "accumulator starts at +0.0": _start_from_plus_zero}
RNE_MUTANTS = {"truncation": _truncate_bf16, "round half up": _round_half_up_bf16}


@pytest.mark.parametrize("name", sorted(SUM_MUTANTS))
def test_pins_catch_summation_mutants(name, monkeypatch):
    fn = SUM_MUTANTS[name]
    monkeypatch.setattr(arith, "ordered_sum", fn)
    monkeypatch.setattr(naming, "ordered_sum", fn)
    monkeypatch.setattr(collectives, "ordered_sum", fn)
    assert not _all_pins_pass(), name


@pytest.mark.parametrize("name", sorted(RNE_MUTANTS))
def test_pins_catch_rounding_mutants(name, monkeypatch):
    monkeypatch.setattr(arith, "f32_to_bf16_rne", RNE_MUTANTS[name])
    assert not _all_pins_pass(), name


def test_pins_catch_a_transposed_alltoall(monkeypatch):
    def wrong(xs):
        R = len(xs)
        b = len(xs[0]) // R
        # block s of source d instead of block d of source s
        return [np.concatenate([xs[d][s * b:(s + 1) * b] for s in range(R)]) for d in range(R)]
    monkeypatch.setattr(collectives, "alltoall", wrong)
    assert not _collectives_ok()


def test_pins_catch_copy_from_the_wrong_producer(monkeypatch):
    orig = naming.run_naming

    def wrong(R, op, dtype, in_len, in_segs, out_len, out_segs, inputs, outputs):
        if op == "copy" and in_segs:
            # shift every producer's offset by one element where that stays in bounds
            in_segs = [(r, off + 1 if off + c < in_len[r] else off, c, nm)
                       for (r, off, c, nm) in in_segs]
        return orig(R, op, dtype, in_len, in_segs, out_len, out_segs, inputs, outputs)
    monkeypatch.setattr(naming, "run_naming", wrong)
    assert not _all_pins_pass()


# ---------------------------------------------------------------- fused producer, tolerance

def _gemv_ok():
    try:
        pins.test_gemv_payload_matches_exact_rational_evaluation()
        pins.test_gemv_row_order_is_observable()
        pins.test_gemv_payload_closed_forms()
    except AssertionError:
        return False
    return True


def _gemv_mutant(kind):
    from oracle.arith import bf16_to_f32, f32_to_bf16_rne

    def gemv(wts, xs):
        out = []
        for wt, x in zip(wts, xs):
            if kind == "weights transposed" and wt.shape[0] == wt.shape[1]:
                wt = np.ascontiguousarray(wt.T)
            w, xv = bf16_to_f32(wt), bf16_to_f32(x)
            k = w.shape[0]
            rows = list(range(k))
            if kind == "rows in reverse":
                rows = rows[::-1]
            if kind == "last row dropped" and k > 1:
                rows = rows[:-1]
            prod = lambda i: w[i] * xv[i]
            if kind == "products rounded to bf16":
                prod = lambda i: bf16_to_f32(f32_to_bf16_rne(w[i] * xv[i]))
            if kind == "eight k-blocks" and k % 8 == 0:
                kb = k // 8
                acc = None
                for b in range(8):
                    part = prod(b * kb)
                    for i in range(b * kb + 1, (b + 1) * kb):
                        part = part + prod(i)
                    acc = part if acc is None else acc + part
            elif kind == "accumulator starts at +0.0":
                acc = np.zeros(w.shape[1], np.float32)
                for i in rows:
                    acc = acc + prod(i)
            else:
                acc = prod(rows[0])
                for i in rows[1:]:
                    acc = acc + prod(i)
            out.append(f32_to_bf16_rne(acc))
        return out
    return gemv


GEMV_MUTANTS = ["accumulator starts at +0.0", "products rounded to bf16", "eight k-blocks",
                "rows in reverse", "last row dropped", "weights transposed"]


def test_unmutated_gemv_oracle_passes_its_pins():
    assert _gemv_ok()


@pytest.mark.parametrize("kind", GEMV_MUTANTS)
def test_pins_catch_gemv_mutants(kind, monkeypatch):
    monkeypatch.setattr(collectives, "gemv_payloads", _gemv_mutant(kind))
    assert not _gemv_ok(), kind


def _tolerance_ok():
    try:
        for dt in ("bf16", "f32"):
            for order in ("rank", "reversed", "tree"):
                pins.test_any_summation_order_is_within_tolerance(dt, order)
        pins.test_tolerance_rejects_real_errors()
    except AssertionError:
        return False
    return True


@pytest.mark.parametrize("kind", ["ten times looser", "no accumulation term",
                                  "absolute instead of relative"])
def test_pins_catch_tolerance_mutants(kind, monkeypatch):
    from oracle import tolerance
    orig = tolerance.within_tolerance

    def wrong(got, terms, dtype):
        n = len(terms)
        s = tolerance.exact_sum(terms, dtype)
        S = np.sum([np.abs(arith.to_f32(t, dtype).astype(np.float64)) for t in terms], axis=0)
        g = (arith.bf16_to_f32(got) if dtype == "bf16"
             else np.asarray(got, np.float32)).astype(np.float64)
        rt = tolerance.RTOL[dtype]
        if kind == "ten times looser":
            bound = 10 * rt * np.abs(s) + (n - 1) * 2.0 ** -24 * S * (1 + rt)
        elif kind == "no accumulation term":
            bound = rt * np.abs(s)
        else:
            bound = np.full_like(s, rt)
        return np.abs(g - s) <= bound
    assert _tolerance_ok()
    monkeypatch.setattr(tolerance, "within_tolerance", wrong)
    assert not _tolerance_ok(), kind
    monkeypatch.setattr(tolerance, "within_tolerance", orig)


def _gemv_tolerance_ok():
    try:
        for blocks in (1, 8, 64):
            pins.test_gemv_other_orders_are_within_tolerance(blocks)
        pins.test_gemv_tolerance_rejects_real_errors()
        pins.test_gemv_tolerance_compares_special_values_by_class()
    except AssertionError:
        return False
    return True


@pytest.mark.parametrize("kind", ["ten times looser", "no accumulation term",
                                  "special values compared as numbers"])
def test_pins_catch_gemv_tolerance_mutants(kind, monkeypatch):
    from oracle import tolerance
    assert _gemv_tolerance_ok()
    if kind == "special values compared as numbers":
        monkeypatch.setattr(tolerance, "_same_special", lambda got, ref: np.zeros(got.shape, bool))
    else:
        def wrong(p):
            s = p.sum(axis=0)
            S = np.abs(p).sum(axis=0)
            rt = tolerance.RTOL["bf16"]
            if kind == "ten times looser":
                return s, 10 * (rt * np.abs(s) + (p.shape[0] - 1) * 2.0 ** -24 * S)
            return s, rt * np.abs(s)
        monkeypatch.setattr(tolerance, "_gemv_bound", wrong)
    assert not _gemv_tolerance_ok(), kind
