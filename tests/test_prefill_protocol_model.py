"""A randomized model of the persistent prefill kernel's barrier protocol.

One CTA walks work items (two query halves each) with three roles that hand
work over through mbarriers: producer warps (a quarter of Q per item, then K
or V tiles into two-slot rings, tiles counted across items), one thread
issuing tensor-core operations (executed in issue order; a commit arrives
once everything issued before it is done), and one softmax warpgroup per
half (S read, P written over the same tensor-memory columns, O read out at
the end of an item).  Parity waits only tell one phase from the next, so the
protocol must keep every waiter within one phase of its barrier.

The model plays the protocol with random interleavings of the actors, the
tensor pipe and the landing of copies, and checks that every S reads the
item's Q and the right K tile, every P V reads the P of its tile and the
right V tile and never overwrites an O the softmax warps have not read out,
the softmax reads the S of its tile and O once it is complete, and that the
run finishes.  It also shows that the guards are needed: without the wait for
the last S before Q is reloaded, or for a K slot to be free, some
interleaving reads stale data; the wait for O to be read out before the next
item's first P V turns out to be implied by the softmax warps' own order.
No GPU is involved.
"""
import random

import pytest

from test_protocol_model import Barrier, ProtocolError


def play(seed, items, q_guard=True, o_guard=True, k_guard=True):
    """items: list of (tiles of half A, tiles of half B); B may be 0."""
    rng = random.Random(seed)
    k_full = [Barrier(2) for _ in range(2)]       # expect_tx arrival + 16-byte-copy arrival
    v_full = [Barrier(2) for _ in range(2)]
    k_empty = [Barrier(1) for _ in range(2)]
    v_empty = [Barrier(1) for _ in range(2)]
    s_full = [Barrier(1) for _ in range(2)]
    p_full = [Barrier(1) for _ in range(2)]       # the half's warpgroup as one arrival
    o_done = [Barrier(1) for _ in range(2)]
    o_free = [Barrier(1) for _ in range(2)]
    q_full = Barrier(4)                            # the four producer warps
    q_empty = Barrier(1)
    kslot = [None, None]                           # tile in each K / V slot
    vslot = [None, None]
    qpart = [None] * 4                             # item of each quarter of Q
    sp = [None, None]                              # S / P columns of each half
    o_acc = [None, None]                           # (item, tile) accumulated in O
    o_read = [None, None]                          # last item whose O was read out
    fifo = []                                      # tensor-core operations in issue order
    in_flight = []

    def wait(bar, parity):
        while not bar.test_wait(parity):
            yield

    def producer(kind, slot, quarter):
        full = k_full if kind == "K" else v_full
        empty = k_empty if kind == "K" else v_empty
        data = kslot if kind == "K" else vslot
        gt = qc = 0
        for it, (ta, tb) in enumerate(items):
            nt = max(ta, tb)
            if qc > 0 and q_guard:
                yield from wait(q_empty, (qc - 1) & 1)
            landed = [False]

            def land_q(it=it, landed=landed):
                qpart[quarter] = it
                landed[0] = True
            in_flight.append(land_q)
            q_sent = False
            for kt in range(nt):
                g = gt + kt
                if g % 2 != slot:
                    continue
                if g >= 2 and (kind == "V" or k_guard):
                    yield from wait(empty[slot], ((g // 2) & 1) ^ 1)
                full[slot].arrive(tx=1)

                def land(g=g):
                    data[slot] = g
                    full[slot].complete_tx(1)
                in_flight.append(land)
                yield
                full[slot].arrive()                # no 16-byte copies in the model
                if not q_sent:
                    while not landed[0]:
                        yield
                    q_full.arrive()
                    q_sent = True
            if not q_sent:
                while not landed[0]:
                    yield
                q_full.arrive()
            gt += nt
            qc += 1

    def mma():
        gt = qc = 0
        pc = [0, 0]
        ofc = [0, 0]
        o_used = [False, False]
        for it, (ta, tb) in enumerate(items):
            tiles = (ta, tb)
            nt = max(ta, tb)
            last_half = 1 if tb > 0 else 0
            s_left = [ta + tb]
            yield from wait(q_full, qc & 1)
            qc += 1
            yield from wait(k_full[gt % 2], (gt // 2) & 1)

            def issue_s(hh, g, kt):
                fifo.append(("S", hh, g, kt, it))
                if hh == last_half:
                    fifo.append(("commit", k_empty[g % 2]))
                fifo.append(("commit", s_full[hh]))
                s_left[0] -= 1
                if s_left[0] == 0:
                    fifo.append(("commit", q_empty))
            for hh in range(2):
                if tiles[hh] > 0:
                    issue_s(hh, gt, 0)
            for kt in range(nt):
                g = gt + kt
                for hh in range(2):
                    if kt >= tiles[hh]:
                        continue
                    yield from wait(p_full[hh], pc[hh] & 1)
                    yield from wait(v_full[g % 2], (g // 2) & 1)
                    pc[hh] += 1
                    if kt == 0 and o_used[hh] and o_guard:
                        yield from wait(o_free[hh], ofc[hh] & 1)
                        ofc[hh] += 1
                    fifo.append(("PV", hh, g, kt, it, o_used[hh]))
                    if hh == last_half:
                        fifo.append(("commit", v_empty[g % 2]))
                    if kt + 1 < tiles[hh]:
                        yield from wait(k_full[(g + 1) % 2], ((g + 1) // 2) & 1)
                        issue_s(hh, g + 1, kt + 1)
                    else:
                        fifo.append(("commit", o_done[hh]))
                        o_used[hh] = True
                    yield
            gt += nt

    def tensor_pipe():
        while True:
            if not fifo:
                yield
                continue
            op = fifo.pop(0)
            if op[0] == "commit":
                op[1].arrive()
            elif op[0] == "S":
                _, hh, g, kt, it = op
                if qpart != [it] * 4:
                    raise ProtocolError("S of item %d read Q %s" % (it, qpart))
                if kslot[g % 2] != g:
                    raise ProtocolError("S of tile %d read K tile %s" % (g, kslot[g % 2]))
                sp[hh] = ("S", it, kt)
            else:
                _, hh, g, kt, it, used = op
                if sp[hh] != ("P", it, kt):
                    raise ProtocolError("P V of item %d tile %d read %s" % (it, kt, sp[hh]))
                if vslot[g % 2] != g:
                    raise ProtocolError("P V of tile %d read V tile %s" % (g, vslot[g % 2]))
                if kt == 0 and used and o_read[hh] != last_item(hh, it):
                    raise ProtocolError("item %d's first P V overwrote O not read out" % it)
                o_acc[hh] = (it, kt)
            yield

    def last_item(hh, it):
        # the last earlier item with tiles in half hh
        for j in range(it - 1, -1, -1):
            if items[j][hh] > 0:
                return j
        return None

    def softmax(hh):
        sc = od = 0
        for it, tiles in enumerate(items):
            if tiles[hh] == 0:
                continue
            for kt in range(tiles[hh]):
                yield from wait(s_full[hh], sc & 1)
                sc += 1
                if sp[hh] != ("S", it, kt):
                    raise ProtocolError("softmax of item %d tile %d read %s" % (it, kt, sp[hh]))
                if any(op[0] == "PV" and op[1] == hh for op in fifo):
                    raise ProtocolError("O rescaled with a P V of its half in flight")
                yield
                sp[hh] = ("P", it, kt)
                p_full[hh].arrive()
            yield from wait(o_done[hh], od & 1)
            od += 1
            if o_acc[hh] != (it, tiles[hh] - 1):
                raise ProtocolError("item %d read O %s" % (it, o_acc[hh]))
            yield
            o_read[hh] = it
            o_free[hh].arrive()

    actors = [producer("K", 0, 0), producer("K", 1, 1), producer("V", 0, 2),
              producer("V", 1, 3), mma(), softmax(0), softmax(1)]
    pipe = tensor_pipe()
    steps = 0
    while actors or in_flight or fifo:
        steps += 1
        if steps > 400_000:
            raise ProtocolError("no progress (on the GPU the bounded waits would time out)")
        r = rng.random()
        if in_flight and r < 0.25:
            in_flight.pop(rng.randrange(len(in_flight)))()
            continue
        if fifo and r < 0.45:
            next(pipe)
            continue
        if not actors:
            if fifo:
                next(pipe)
            continue
        a = rng.choice(actors)
        try:
            next(a)
        except StopIteration:
            actors.remove(a)


def _items(rng):
    out = []
    for _ in range(rng.randint(1, 5)):
        ta = rng.randint(1, 5)
        tb = rng.choice([0, ta, ta + 1, ta + 2])
        out.append((ta, tb))
    return out


def _failures(trials, seed0, **kw):
    bad = 0
    for t in range(trials):
        try:
            play(seed0 + t, _items(random.Random(seed0 + t)), **kw)
        except ProtocolError:
            bad += 1
    return bad


def test_prefill_protocol_never_reads_stale_data():
    assert _failures(300, 2000) == 0


def test_prefill_protocol_single_items():
    for t in range(60):
        rng = random.Random(9000 + t)
        ta = rng.randint(1, 6)
        play(9000 + t, [(ta, rng.choice([0, ta, ta + 2]))])


@pytest.mark.parametrize("guard", ["q_guard", "k_guard"])
def test_each_prefill_guard_is_needed(guard):
    assert _failures(200, 2000, **{guard: False}) > 0


def test_o_free_is_implied_by_the_softmax_order():
    # The softmax warps read O out before they write the next item's first P,
    # and that P V waits for p_full: the o_free wait never decides anything
    # (the kernel keeps it so that O's hand-over does not rest on this).
    assert _failures(200, 2000, o_guard=False) == 0
