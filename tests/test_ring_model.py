"""CPU model of a fused-producer compute warp's weight ring (no GPU).

Each compute warp streams its k-block of weight rows through a private ring of 3 shared-
memory slots, one 16-row tensor copy per slot, completed on the slot's mbarrier. The model
follows the kernel's steps (the prologue's first 3 fills; per block: a readiness test of
the fills already issued, a parity wait on the slot, reading it, refilling it with the fill
3 ahead when that fill belongs to the same block, else holding the refill back until the
block's results are handed over) under random landing orders of the copies, and checks:
every read finds its own fill landed; no slot is refilled before its previous fill was read;
every readiness test targets a fill already issued (a parity test of an unissued fill could
take the slot's previous phase for it); every fill carries the rows and stage item its
number stands for; every fill issued is read.
"""

import random

import pytest

SLOTS = 3


class Ring:
    def __init__(self, bs, nitems, epochs, seed):
        self.rnd = random.Random(seed)
        self.bs, self.nitems = bs, nitems
        self.total = epochs * nitems * bs
        self.issued = {}  # fill number -> (slot, row block, item)
        self.landed = set()
        self.read = set()
        self.last_in_slot = {}
        self.phase = [0] * SLOTS  # completed phases per slot

    def fill(self, slot, rj, item, t):
        assert t not in self.issued
        assert slot == t % SLOTS, ("slot", t, slot)
        assert rj == t % self.bs and item == (t // self.bs) % self.nitems, ("rows", t, rj, item)
        prev = self.last_in_slot.get(slot)
        assert prev is None or prev in self.read, ("refill before read", t, prev)
        self.issued[t] = (slot, rj, item)
        self.last_in_slot[slot] = t

    def land_some(self):
        for t in sorted(set(self.issued) - self.landed):
            # a slot's phases complete in order: its previous fill has landed already
            if self.rnd.random() < 0.5 and (t < SLOTS or t - SLOTS in self.landed):
                self.landed.add(t)
                self.phase[t % SLOTS] += 1

    def parity_done(self, slot, lap):
        # mbarrier parity test: the phase of parity lap & 1 has completed iff the current
        # phase's parity differs
        return (self.phase[slot] & 1) != (lap & 1)


def run(bs, nitems, epochs, seed):
    m = Ring(bs, nitems, epochs, seed)
    # prologue: fills 0..2; the refill cursor then points at fill 3
    j = ri = 0
    for q in range(SLOTS):
        if q < m.total:
            m.fill(q % SLOTS, j, ri, q)
        j += 1
        if j == bs:
            j, ri = 0, (ri + 1) % nitems
    q, lap, slot, rp_j, r_i = 0, 0, 0, j, ri
    for _piece in range(epochs * nitems):
        m.land_some()
        qe = q + bs
        pend = None
        npend = 0
        for jj in range(bs):
            if jj % 32 == 0:
                for lane in range(SLOTS):
                    if jj + lane < bs:
                        t = q + lane
                        assert t in m.issued, ("readiness test of an unissued fill", t)
                        o = slot + lane
                        wrap = 1 if o >= SLOTS else 0
                        s_, l_ = o - wrap * SLOTS, lap + wrap
                        assert (s_, l_) == (t % SLOTS, t // SLOTS)
                        if m.parity_done(s_, l_):
                            assert t in m.landed, ("aliased readiness", t)
            assert (slot, lap) == (q % SLOTS, q // SLOTS)
            steps = 0
            while q not in m.landed:
                m.land_some()
                steps += 1
                assert steps < 10000, "deadlock"
            m.read.add(q)
            if q + SLOTS < m.total:
                if q + SLOTS < qe:
                    m.fill(slot, rp_j, r_i, q + SLOTS)
                else:
                    if npend == 0:
                        pend = (slot, rp_j, r_i, q + SLOTS)
                    npend += 1
            q += 1
            slot += 1
            if slot == SLOTS:
                slot, lap = 0, lap + 1
            rp_j += 1
            if rp_j == bs:
                rp_j, r_i = 0, (r_i + 1) % nitems
            if m.rnd.random() < 0.3:
                m.land_some()
        if npend:  # after the block's results are handed over
            s_, rj, it, t = pend
            for d in range(npend):
                m.fill(s_, rj, it, t + d)
                s_ = (s_ + 1) % SLOTS
                rj += 1
                if rj == bs:
                    rj, it = 0, (it + 1) % nitems
    assert len(m.read) == m.total
    assert set(m.issued) == m.read


@pytest.mark.parametrize("bs", [1, 2, 3, 4, 5, 8, 31, 32, 33, 64])
@pytest.mark.parametrize("nitems", [1, 2, 3, 17])
def test_ring_reads_refills_and_readiness(bs, nitems):
    for epochs in (1, 2, 5):
        for seed in range(3):
            run(bs, nitems, epochs, seed)


def test_model_catches_a_refill_before_the_read():
    # the check is live: issuing a fill into a slot whose previous fill was not read fails
    m = Ring(4, 1, 2, 0)
    m.fill(0, 0, 0, 0)
    with pytest.raises(AssertionError):
        m.fill(0, 3, 0, 3)
