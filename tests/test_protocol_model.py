"""A randomized model of the decode kernel's producer/consumer protocol.

The kernel moves K/V tiles through a ring of shared-memory stages guarded by
mbarriers (a "full" barrier armed with the expected bytes and completed by
the async copies, an "empty" barrier the consumer arrives on), and q through
a two-slot ring.  An mbarrier parity wait only tells one phase from the next,
so a waiter two phases behind would take a stale phase for the one it wants.
The kernel guards against that in two ways:

* q copies are issued in piece order (a counter in shared memory), so a
  q-ring slot never gets two copies in flight;
* a consumer first waits until the stage's round for its tile is armed (the
  issuing lane records the round after arming), then waits on the parity.

This model plays the protocol with random interleavings of the producer's
lanes, the consumer warps and the completion of in-flight copies, and checks
that every consumer reads the tile and the q it expects and that the run
finishes.  It also shows that each guard is needed: without either, some
interleaving reads stale data, double-arrives on a barrier or stalls.
No GPU is involved.
"""
import random

import pytest


class ProtocolError(Exception):
    """A consumer read stale data, a barrier got more arrivals than a phase
    expects (on the GPU: a copy landing in the wrong phase), or the actors
    stopped making progress."""


class Barrier:
    """mbarrier: a phase completes when the expected arrivals have arrived
    and the transaction count (bytes) is back to zero."""

    def __init__(self, count):
        self.count = count
        self.phase = 0
        self.pending = count
        self.tx = 0

    def _advance(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def arrive(self, tx=0):
        if self.pending == 0:
            raise ProtocolError("arrival on a completed phase")
        self.tx += tx
        self.pending -= 1
        self._advance()

    def complete_tx(self, n):
        self.tx -= n
        self._advance()

    def test_wait(self, parity):
        # true once the phase with this parity has completed
        return (self.phase & 1) != parity


def play(seed, nst, W, piece_lengths, ordered_q=True, round_guard=True, group=None):
    """One randomized run; raises ProtocolError on a stale read or an extra
    arrival."""
    rng = random.Random(seed)
    tiles = [(p, i) for p, n in enumerate(piece_lengths) for i in range(n)]
    n_local = len(tiles)
    group = group or min(32, nst)
    full = [Barrier(1) for _ in range(nst)]
    empty = [Barrier(1) for _ in range(nst)]
    qfull = [Barrier(1) for _ in range(2)]
    qempty = [Barrier(W) for _ in range(2)]
    stage = [None] * nst
    qslot = [None] * 2
    in_flight = []
    q_issued = [0]
    armed = [0] * nst                  # last armed round + 1, per stage

    def lane(k, starts_piece, qn, st, rnd):
        piece = tiles[k][0]
        if starts_piece:
            if ordered_q:
                while q_issued[0] < qn:
                    yield
            slot = qn & 1
            while not qempty[slot].test_wait(((qn >> 1) & 1) ^ 1):
                yield
            qfull[slot].arrive(tx=1)

            def land_q(slot=slot, piece=piece):
                qslot[slot] = piece
                qfull[slot].complete_tx(1)
            in_flight.append(land_q)
            q_issued[0] = qn + 1
        while not empty[st].test_wait((rnd & 1) ^ 1):
            yield
        full[st].arrive(tx=2)
        armed[st] = rnd + 1
        stage[st] = {}

        def land(part, st=st, k=k):
            stage[st][part] = k
            full[st].complete_tx(1)
        in_flight.append(lambda: land("K"))
        in_flight.append(lambda: land("V"))

    def producer():
        last_piece, qn_base, st_base, rnd_base = -1, 0, 0, 0
        for k0 in range(0, n_local, group):
            n = min(group, n_local - k0)
            starts = [tiles[k0 + j][0] != (last_piece if j == 0 else tiles[k0 + j - 1][0])
                      for j in range(n)]
            lanes = []
            for j in range(n):
                st, rnd = st_base + j, rnd_base
                if st >= nst:
                    st, rnd = st - nst, rnd + 1
                lanes.append(lane(k0 + j, starts[j], qn_base + sum(starts[:j]), st, rnd))
            while lanes:                       # the lanes poll in one loop
                ln = rng.choice(lanes)
                try:
                    next(ln)
                except StopIteration:
                    lanes.remove(ln)
                yield
            last_piece = tiles[k0 + n - 1][0]
            qn_base += sum(starts)
            st_base += n
            if st_base >= nst:
                st_base, rnd_base = st_base - nst, rnd_base + 1

    arrived = [0]

    def consumer(w):
        qn, x = 0, 0
        while x < n_local:
            piece = tiles[x][0]
            e = x
            while e < n_local and tiles[e][0] == piece:
                e += 1
            slot = qn & 1
            while not qfull[slot].test_wait((qn >> 1) & 1):
                yield
            if qslot[slot] != piece:
                raise ProtocolError("warp %d read q of piece %s for piece %s" % (w, qslot[slot], piece))
            qempty[slot].arrive()
            qn += 1
            for k in range(x + (w - x % W) % W, e, W):     # round-robin tiles
                st, rnd = k % nst, k // nst
                if round_guard:
                    while armed[st] != rnd + 1:
                        yield
                while not full[st].test_wait(rnd & 1):
                    yield
                if stage[st] != {"K": k, "V": k}:
                    raise ProtocolError("warp %d read %s for tile %d" % (w, stage[st], k))
                yield                                       # registers loaded
                empty[st].arrive()                          # stage released
            arrived[0] += 1                                 # merge barrier
            target = (arrived[0] - 1) // W * W + W
            while arrived[0] < target:
                yield
            x = e

    actors = [producer()] + [consumer(w) for w in range(W)]
    steps = 0
    while actors or in_flight:
        steps += 1
        if steps > 300_000:
            raise ProtocolError("no progress (on the GPU the bounded waits would time out)")
        if in_flight and rng.random() < 0.3:
            in_flight.pop(rng.randrange(len(in_flight)))()
            continue
        if not actors:
            continue
        a = rng.choice(actors)
        try:
            next(a)
        except StopIteration:
            actors.remove(a)


def _shape(rng):
    nst = rng.choice([2, 3, 4, 5, 8])
    W = rng.choice([1, 2, 3, 4])
    pieces = [rng.choice([1, 1, 1, 2, 3, 7, 20]) for _ in range(rng.randint(1, 25))]
    return nst, W, pieces


def _failures(trials, seed0, **kw):
    bad = 0
    for t in range(trials):
        nst, W, pieces = _shape(random.Random(seed0 + t))
        try:
            play(seed0 + t, nst, W, pieces, **kw)
        except ProtocolError:
            bad += 1
    return bad


def test_protocol_never_reads_stale_data():
    assert _failures(400, 1000) == 0


def test_protocol_with_one_tile_per_group_never_reads_stale_data():
    assert _failures(150, 5000, group=1) == 0


@pytest.mark.parametrize("guard", ["round_guard", "ordered_q"])
def test_each_guard_is_needed(guard):
    # with either guard removed, some interleaving reads a stale q or tile
    assert _failures(120, 1000, **{guard: False}) > 0
