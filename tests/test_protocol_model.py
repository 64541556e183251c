"""Exhaustive interleavings of one speculative exchange (CPU model, no GPU).

One producer P and one consumer C share a dual-buffer slot for epoch E. Before the epoch the
slot holds the epoch E-2 payload and a flag {E-2, tag(E-2 payload)}. P writes the new payload
then the flag {E, tag}; C speculatively loads the payload, then the flag, and validates.

Every interleaving of P's two writes and C's two loads is enumerated (with P's writes in
program order, as a release store gives; and in either order, as a relaxed flag store
allows). The pages' literal check (flag epoch == E) accepts a stale payload in at least one
interleaving — the falsifier of the monotonicity premise in the SiFAR review ("What would
settle it"). The content-tagged check never accepts a payload other than the epoch-E one.
"""

import itertools

import pytest

OLD, NEW = ("payload of epoch E-2", 11), ("payload of epoch E", 22)
E = 8


def tag(payload):
    # any injective stand-in for the content hash (collisions are the 2^-32 case)
    return hash(payload) & 0xFFFFFFFF


def run(order):
    """order: sequence of 'Pd' (write payload), 'Pf' (write flag), 'Cd' (load payload),
    'Cf' (load flag). Returns (loaded payload, loaded flag)."""
    slot = OLD
    flag = (E - 2, tag(OLD))
    seen_d = seen_f = None
    for step in order:
        if step == "Pd":
            slot = NEW
        elif step == "Pf":
            flag = (E, tag(NEW))
        elif step == "Cd":
            seen_d = slot
        elif step == "Cf":
            seen_f = flag
    return seen_d, seen_f


def interleavings(release):
    steps = ["Pd", "Pf", "Cd", "Cf"]
    for perm in itertools.permutations(steps):
        if perm.index("Cd") > perm.index("Cf"):
            continue  # the consumer loads the payload first (program order)
        if release and perm.index("Pd") > perm.index("Pf"):
            continue  # a release flag store is ordered after the payload write
        yield perm


def literal_accepts(d, f):
    return f[0] == E


def tagged_accepts(d, f):
    return f[0] == E and f[1] == tag(d)


@pytest.mark.parametrize("release", [True, False])
def test_literal_check_accepts_a_stale_payload(release):
    stale_accepted = [o for o in interleavings(release)
                      if literal_accepts(*run(o)) and run(o)[0] != NEW]
    assert stale_accepted, "the falsifying interleaving must exist"
    assert ("Cd", "Pd", "Pf", "Cf") in stale_accepted


@pytest.mark.parametrize("release", [True, False])
def test_tagged_check_never_accepts_a_stale_payload(release):
    for o in interleavings(release):
        d, f = run(o)
        if tagged_accepts(d, f):
            assert d == NEW, o


@pytest.mark.parametrize("release", [True, False])
def test_tagged_check_accepts_when_the_exchange_is_complete(release):
    # liveness: if both writes precede both loads, the check passes on the first try
    for o in interleavings(release):
        if max(o.index("Pd"), o.index("Pf")) < min(o.index("Cd"), o.index("Cf")):
            assert tagged_accepts(*run(o)), o


def _states(release):
    """Every (payload, flag) state reachable by a prefix of the producer's writes."""
    orders = [("Pd", "Pf")] if release else [("Pd", "Pf"), ("Pf", "Pd")]
    for o in orders:
        for k in range(3):
            yield run(tuple(o[:k]) + ("Cd", "Cf"))


def test_with_release_a_flag_showing_E_implies_the_new_payload():
    # so after a failed check, waiting for the flag (acquire) and reloading is enough
    for d, f in _states(release=True):
        if f[0] == E:
            assert d == NEW


def test_without_release_the_retry_must_validate_again():
    # a relaxed flag may land before the payload: waiting for the flag is not enough, which
    # is why the fence-free mode re-checks the content tag on every reload
    assert any(f[0] == E and d != NEW for d, f in _states(release=False))
