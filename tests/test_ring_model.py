"""CPU model of the fused producer's shared-memory pipeline (no GPU).

One fused CTA runs four roles that meet only through mbarriers and one shared counter:
- the weight streamer fills a ring of S slots (one tensor copy of 64 rows each) with every fill
  of the run in order, fill f into slot f % S once the compute lanes released the slot's
  previous fill (empty[s], parity of lap f // S, inverted);
- the x streamer copies piece q's x into buffer q % 2 once the engine has opened piece q
  (go > q);
- four compute warps take the pieces in order: wait for the piece's x (xfull), read the
  piece's fills in order (full[s], parity of lap), release each slot, write their part of
  result slot q % 2 and arrive on rfull;
- the engine takes piece q from its result slot (rfull) and opens piece q + 2 (go =
  min(taken + 2, pieces its chained epochs allow, total)); with chained epochs, an epoch's
  pieces are opened only when the engine reaches that epoch.
The model follows those steps with mbarriers modelled as in the PTX ISA (arrival count,
transaction bytes, phase; a parity wait passes iff the phase of that parity has completed)
under random interleavings of the roles and random landing orders of the copies, and checks:
every read finds the data its number stands for; no slot, x buffer or result slot is
overwritten before every reader has finished with its previous contents; every role ends
(no wait on a phase that can no longer complete). The go counter alone also guards the x
buffers and the result slots: piece q is opened only once piece q - 2 has been taken, so its
x and its result slot are free by then. Each wait of the protocol is shown necessary by a
variant without it that the model catches.
"""

import random

import pytest

WARPS = 4       # compute warps
LANES = 32      # arrivals per compute warp (every lane arrives)


class MBar:
    def __init__(self, count):
        self.count, self.pending, self.tx, self.phase = count, count, 0, 0

    def _check(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def arrive(self, n=1):
        assert self.pending >= n, "more arrivals than the phase expects"
        self.pending -= n
        self._check()

    def expect_tx(self, nbytes):
        self.tx += nbytes
        self.arrive()

    def complete_tx(self, nbytes):
        self.tx -= nbytes
        assert self.tx >= 0
        self._check()

    def done(self, parity):
        return (self.phase & 1) != (parity & 1)


class Pipeline:
    def __init__(self, S, kslots, nitems, epochs, chain, seed, mutant=None):
        self.rnd = random.Random(seed)
        self.mutant = mutant
        self.S, self.kslots, self.nitems, self.chain = S, kslots, nitems, chain
        self.total = epochs * nitems
        self.full = [MBar(1) for _ in range(S)]
        self.empty = [MBar(WARPS * LANES) for _ in range(S)]
        self.xfull = [MBar(1) for _ in range(2)]
        self.rfull = [MBar(WARPS * LANES) for _ in range(2)]
        self.slot = [None] * S          # fill number held by each slot
        self.slot_readers = [set(range(WARPS))] * S  # warps that read the current fill
        self.xbuf = [None, None]
        self.x_readers = [set(range(WARPS)), set(range(WARPS))]
        self.res = [[None] * WARPS for _ in range(2)]
        self.taken_from = [None, None]  # last piece the engine took from each result slot
        self.copies = []                # in flight: (kind, index, number)
        self.go = 0 if chain else min(2, self.total)
        self.taken = 0
        self.chain_open = 0 if chain else 1 << 62

    def open_pieces(self):
        ahead = 3 if self.mutant == "opens three pieces ahead" else 2
        self.go = min(self.taken + ahead, self.chain_open, self.total)

    # ------------------------------------------------------------ roles (generators)
    def weight_streamer(self):
        F = self.total * self.kslots
        for f in range(F):
            s, lap = f % self.S, f // self.S
            while self.mutant != "no empty wait" and not self.empty[s].done((lap & 1) ^ 1):
                yield
            assert self.slot_readers[s] == set(range(WARPS)), ("slot refilled before read", f)
            self.full[s].expect_tx(8192)
            self.copies.append(("w", s, f))
            yield

    def x_streamer(self):
        for q in range(self.total):
            while self.mutant != "x streamer ignores go" and self.go <= q:
                yield
            p = q % 2
            assert self.x_readers[p] == set(range(WARPS)), ("x overwritten before read", q)
            self.xfull[p].expect_tx(1024)
            self.copies.append(("x", p, q))
            yield

    def compute(self, w):
        s = lap = 0
        for q in range(self.total):
            p = q % 2
            while self.mutant != "no xfull wait" and not self.xfull[p].done((q // 2) & 1):
                yield
            assert self.xbuf[p] == q, ("wrong x", q, self.xbuf[p])
            for j in range(self.kslots):
                while self.mutant != "no full wait" and not self.full[s].done(lap & 1):
                    yield
                f = q * self.kslots + j
                assert self.slot[s] == f, ("wrong rows", f, self.slot[s])
                self.slot_readers[s] = self.slot_readers[s] | {w}
                self.empty[s].arrive(LANES)
                s += 1
                if s == self.S:
                    s, lap = 0, lap + 1
                yield
            self.x_readers[p] = self.x_readers[p] | {w}
            assert q < 2 or self.taken_from[p] == q - 2, ("result slot overwritten before taken", q)
            self.res[p][w] = q
            self.rfull[p].arrive(LANES)
            yield

    def engine(self):
        for q in range(self.total):
            if self.chain and q % self.nitems == 0:
                # the chained wait for this epoch (other CTAs' progress): some random delay
                for _ in range(self.rnd.randrange(4)):
                    yield
                self.chain_open = q + self.nitems
                self.open_pieces()
            p = q % 2
            while self.mutant != "no rfull wait" and not self.rfull[p].done((q // 2) & 1):
                yield
            assert self.res[p] == [q] * WARPS, ("wrong results", q, self.res[p])
            self.taken_from[p] = q
            self.taken = q + 1
            self.open_pieces()
            yield

    def land_one(self):
        if not self.copies:
            return
        kind, i, n = self.copies.pop(self.rnd.randrange(len(self.copies)))
        if kind == "w":
            self.slot[i] = n
            self.slot_readers[i] = set()
            self.full[i].complete_tx(8192)
        else:
            self.xbuf[i] = n
            self.x_readers[i] = set()
            self.xfull[i].complete_tx(1024)


def simulate(S, kslots, nitems, epochs, chain, seed, mutant=None):
    m = Pipeline(S, kslots, nitems, epochs, chain, seed, mutant)
    roles = [m.weight_streamer(), m.x_streamer(), m.engine()] + [m.compute(w) for w in range(WARPS)]
    live = list(roles)
    steps = 0
    while live:
        steps += 1
        assert steps < 200000, "no progress: a wait cannot complete"
        if m.copies and m.rnd.random() < 0.3:
            m.land_one()
            continue
        g = m.rnd.choice(live)
        try:
            next(g)
        except StopIteration:
            live.remove(g)
    assert not m.copies
    assert m.taken == m.total
    return m


@pytest.mark.parametrize("seed", range(60))
def test_pipeline_orders_every_buffer(seed):
    rnd = random.Random(1000 + seed)
    S = rnd.choice([2, 3, 4, 5, 22])
    kslots = rnd.choice([1, 2, 3, 5, 7, 32])
    nitems = rnd.choice([1, 1, 2, 3])
    epochs = rnd.choice([1, 2, 3, 5])
    chain = rnd.random() < 0.5
    simulate(S, kslots, nitems, epochs, chain, seed)


@pytest.mark.parametrize("mutant", ["no empty wait", "no full wait", "no xfull wait",
                                    "no rfull wait", "x streamer ignores go",
                                    "opens three pieces ahead"])
def test_the_model_catches_a_missing_wait(mutant):
    # each wait of the protocol is needed: without it, some interleaving overwrites a buffer
    # that a reader still needs, or reads the wrong data
    caught = 0
    for seed in range(60):
        for cfg in ((2, 3, 1, 4), (4, 1, 2, 4)):
            try:
                simulate(*cfg, False, seed, mutant)
            except AssertionError:
                caught += 1
    assert caught > 0, mutant


# ------------------------------------------------------------ zero-copy bulk ring

class BulkRing:
    """The zero-copy bulk ring of one CTA. Producer warp 0 resolves tiles in batches (first 32
    dealt round-robin at a time, then the tail claimed two at a time, or in the claims' sizes
    `tail_batches`, 1 to 32 tiles) into a table of `entries` slots, the tile the CTA issues
    k-th into entry k % entries, and publishes the batch; then each of the `issuers` producer
    warps issues the batch's tiles k with k % issuers == its index, each into stage k % S once
    the consumer warps released that stage's previous tile; the producer warps meet at a
    barrier after each publication and after each batch's issue. The consumers take the tiles
    in order, read the tile's entry through the stage, release the stage, and stop at the end
    marker (warp 0's plain arrival on the next stage)."""

    def __init__(self, S, nstatic, ntail, consumers, seed, entries=64, tail_batches=None,
                 issuers=2, mutant=None):
        self.rnd = random.Random(seed)
        self.S, self.C, self.entries, self.P, self.mutant = S, consumers, entries, issuers, mutant
        self.batches = [min(32, nstatic - i) for i in range(0, nstatic, 32)]
        if tail_batches is None:
            tail_batches = [min(2, ntail - i) for i in range(0, ntail, 2)]
        assert sum(tail_batches) == ntail and all(1 <= b <= 32 for b in tail_batches)
        self.batches += list(tail_batches)
        self.ntiles = nstatic + ntail
        self.full = [MBar(1) for _ in range(S)]
        self.empty = [MBar(consumers) for _ in range(S)]
        self.table = [None] * entries
        self.stile = [None] * S
        self.readers = {}       # entry -> consumers still to read its tile
        self.final = None
        self.copies = []
        self.got = [[] for _ in range(consumers)]
        self.published = None   # size of the batch published for the current round
        self.bar = [0, 0]       # arrivals at the producers' barrier, generation
        self.issued = 0

    def barrier(self):
        gen = self.bar[1]
        self.bar[0] += 1
        if self.bar[0] == self.P:
            self.bar = [0, gen + 1]
        while self.bar[1] == gen:
            yield

    def producer(self, w):
        k0 = 0
        for rnd in range(len(self.batches) + 1):
            if w == 0:
                batch = self.batches[rnd] if rnd < len(self.batches) else 0
                for i in range(batch):
                    e = (k0 + i) % self.entries
                    assert not self.readers.get(e), ("table entry rewritten while read", k0 + i)
                    self.table[e] = k0 + i
                self.published = batch
                yield
            if self.mutant != "no publish barrier":
                yield from self.barrier()
            batch = self.published
            if batch == 0:
                break
            for k in range(k0, k0 + batch):
                if k % self.P != w:
                    continue
                s, lap = k % self.S, k // self.S
                while not self.empty[s].done((lap & 1) ^ 1):
                    yield
                e = k % self.entries
                assert self.table[e] == k, ("table entry not yet written", k)
                self.stile[s] = e
                self.readers[e] = set(range(self.C))
                self.full[s].expect_tx(4096)
                self.copies.append(s)
                self.issued += 1
                yield
            k0 += batch
            if self.mutant != "no issue barrier":
                yield from self.barrier()
        if w == 0:
            s, lap = k0 % self.S, k0 // self.S
            while not self.empty[s].done((lap & 1) ^ 1):
                yield
            self.final = k0
            self.full[s].arrive()   # the end marker

    def consumer(self, c):
        k = s = lap = 0
        while True:
            while not self.full[s].done(lap & 1):
                yield
            if self.final is not None and k >= self.final:
                return
            e = self.stile[s]
            self.got[c].append(self.table[e])
            self.readers[e].discard(c)
            self.empty[s].arrive()
            k += 1
            s += 1
            if s == self.S:
                s, lap = 0, lap + 1
            yield

    def land_one(self):
        s = self.copies.pop(self.rnd.randrange(len(self.copies)))
        self.full[s].complete_tx(4096)


def simulate_bulk(S, nstatic, ntail, consumers, seed, entries=64, tail_batches=None, issuers=2,
                  mutant=None):
    m = BulkRing(S, nstatic, ntail, consumers, seed, entries, tail_batches, issuers, mutant)
    live = [m.producer(w) for w in range(issuers)] + [m.consumer(c) for c in range(consumers)]
    steps = 0
    while live:
        steps += 1
        assert steps < 400000, "no progress"
        if m.copies and m.rnd.random() < 0.3:
            m.land_one()
            continue
        g = m.rnd.choice(live)
        try:
            next(g)
        except StopIteration:
            live.remove(g)
    for c in range(consumers):
        assert m.got[c] == list(range(m.ntiles)), c


@pytest.mark.parametrize("seed", range(40))
def test_bulk_ring_table_and_end_marker(seed):
    rnd = random.Random(2000 + seed)
    simulate_bulk(rnd.choice([2, 3, 6, 8, 12]), rnd.choice([0, 1, 31, 32, 33, 64, 100]),
                  rnd.choice([0, 1, 2, 7, 40]), rnd.choice([1, 8]), seed)


def test_the_bulk_model_catches_a_table_too_small():
    # a table of 32 entries would be overwritten while the ring still holds its tiles
    caught = 0
    for seed in range(40):
        try:
            simulate_bulk(8, 100, 10, 8, seed, entries=32)
        except AssertionError:
            caught += 1
    assert caught > 0


@pytest.mark.parametrize("issuers", [1, 2])
@pytest.mark.parametrize("seed", range(20))
def test_bulk_ring_one_or_two_issuing_warps(issuers, seed):
    rnd = random.Random(5000 + seed)
    simulate_bulk(rnd.choice([2, 3, 6, 12]), rnd.choice([0, 1, 31, 33, 64, 100]),
                  rnd.choice([0, 1, 2, 7, 40]), rnd.choice([1, 8]), seed, issuers=issuers)


@pytest.mark.parametrize("mutant", ["no publish barrier", "no issue barrier"])
def test_the_bulk_model_needs_both_producer_barriers(mutant):
    # without the barrier after publication, warp 1 issues from entries not yet written;
    # without the one after the issue, warp 0 rewrites entries of tiles still in the ring
    caught = 0
    for seed in range(60):
        try:
            simulate_bulk(12, 100, 40, 8, seed, issuers=2, mutant=mutant)
        except (AssertionError, TypeError):
            caught += 1
    assert caught > 0, mutant


# ------------------------------------------------------------ claims of the bulk ring's tail

def claim_size(claimed, tail, grid, guided):
    """Tiles one claim takes: two, or (guided) about half of a CTA's fair share of the tail
    still unclaimed after `claimed`, from two to 32."""
    if not guided:
        return 2
    q = max(tail - claimed, 0) // (2 * grid)
    return min(max(q, 2), 32)


def claim_tail(tail, grid, guided, seed):
    """CTAs claiming the tail from one shared counter in a random interleaving. Each takes
    its next claim one batch ahead (size from the position after its current claim) and
    stops at the first claim that starts past the tail. Returns each CTA's batches."""
    rnd = random.Random(seed)
    counter = 0
    state = [{"cur": None, "next": None, "done": False, "batches": []} for _ in range(grid)]

    def take(n):
        nonlocal counter
        c = counter
        counter += n
        return c, n

    while not all(st["done"] for st in state):
        st = rnd.choice([x for x in state if not x["done"]])
        if st["next"] is None:
            st["cur"] = take(claim_size(0, tail, grid, guided))
        else:
            st["cur"] = st["next"]
        c, n = st["cur"]
        st["next"] = take(claim_size(c + n, tail, grid, guided))
        got = [c + i for i in range(n) if c + i < tail]
        if not got:
            st["done"] = True
        else:
            st["batches"].append(got)
    return [st["batches"] for st in state]


@pytest.mark.parametrize("guided", [False, True])
@pytest.mark.parametrize("seed", range(12))
def test_tail_claims_cover_every_tile_once(guided, seed):
    rnd = random.Random(3000 + seed)
    grid = rnd.choice([1, 2, 7, 152])
    tail = rnd.choice([0, 1, 2, 3, 63, 64 * grid, 5 * 64 * grid + 17])
    per_cta = claim_tail(tail, grid, guided, seed)
    seen = sorted(t for batches in per_cta for b in batches for t in b)
    assert seen == list(range(tail))
    for batches in per_cta:
        for b in batches:
            assert 1 <= len(b) <= 32 and b == list(range(b[0], b[0] + len(b)))
            assert guided or len(b) <= 2


def test_guided_claims_shrink_toward_the_end():
    # early claims are large (fewer claims, each covering the next one's round trips), the
    # last ones small (the tail stays balanced)
    grid, tail = 152, 64 * 152 // 5
    assert claim_size(0, tail, grid, True) == max(2, min(32, tail // (2 * grid)))
    assert claim_size(tail - 10, tail, grid, True) == 2
    sizes = [claim_size(c, 100000, 4, True) for c in list(range(0, 100000, 997)) + [99990]]
    assert sizes == sorted(sizes, reverse=True) and sizes[0] == 32 and sizes[-1] == 2


@pytest.mark.parametrize("seed", range(12))
def test_bulk_ring_with_guided_tail_batches(seed):
    # one CTA's share of a guided tail runs through the table and the stages like any batch
    rnd = random.Random(4000 + seed)
    per_cta = claim_tail(rnd.choice([40, 300, 2000]), rnd.choice([1, 3]), True, seed)
    batches = [len(b) for b in per_cta[0]]
    simulate_bulk(rnd.choice([2, 6, 8, 12]), rnd.choice([0, 33, 64]), sum(batches), 8, seed,
                  tail_batches=batches)
