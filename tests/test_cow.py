"""Copy-on-write of shared blocks, on the CPU.

[VIS] "PagedAttention: the cache in blocks": sequences that begin with the
same tokens can reference one physical copy of those blocks, and a sharer gets
its own copy of a block only when it has to modify it.  These tests pin the oracle's block copy and the CoW semantics
(each request keeps seeing exactly its own rows), and check the library's
host bookkeeping (kv_reserve_slots_cow) against a model written here.
"""
import numpy as np
import pytest

from oracle import oracle as O
from paged_kv_cache_273_gb300 import pkv


# ------------------------------------------------------------------ oracle pins
@pytest.mark.parametrize("kind", ["f32", "u16", "i8"])
def test_oracle_block_copy_copies_whole_blocks_and_nothing_else(kind):
    rng = np.random.default_rng(21)
    NB, H, bs, D = 9, 3, 4, 8
    if kind == "f32":
        kc = rng.standard_normal((NB, H, bs, D)).astype(np.float32)
    elif kind == "u16":
        kc = rng.integers(0, 1 << 16, (NB, H, bs, D)).astype(np.uint16)
    else:
        kc = rng.integers(-127, 128, (NB, H, bs, D)).astype(np.int8)
    vc = kc[::-1].copy()
    ks = rng.integers(0, 1 << 16, (NB, H, bs)).astype(np.uint16) if kind == "i8" else None
    vs = ks[::-1].copy() if kind == "i8" else None
    src, dst = np.array([2, 7, 0], np.int32), np.array([5, 1, 8], np.int32)
    want = [a.copy() for a in (kc, vc) + ((ks, vs) if ks is not None else ())]
    for a in want:
        a[dst] = a[src]                      # numpy fancy assignment, block by block
    O.block_copy(src, dst, bs, kc, vc, ks, vs)
    got = [kc, vc] + ([ks, vs] if ks is not None else [])
    for g, w in zip(got, want):
        assert np.array_equal(g, w)


def _cow_model_step(tables, lens, refcount, free, bs):
    """One decode step of copy-on-write bookkeeping, written from the page's
    rule: a token goes to position len; a block that starts at that position
    is new; an existing block that others still hold is copied first."""
    pairs, slots = [], []
    for b in range(len(lens)):
        pos = lens[b]
        j = pos // bs
        if pos % bs == 0:
            blk = free.pop()
            refcount[blk] = 1
            tables[b][j] = blk
        elif refcount[tables[b][j]] > 1:
            old = tables[b][j]
            new = free.pop()
            refcount[new] = 1
            refcount[old] -= 1
            pairs.append((old, new))
            tables[b][j] = new
        slots.append(tables[b][j] * bs + pos % bs)
    return pairs, slots


def test_oracle_copy_on_write_keeps_every_request_private():
    rng = np.random.default_rng(22)
    NB, H, bs, D, S, prompt, steps = 40, 2, 4, 8, 4, 6, 9
    kc = np.zeros((NB, H, bs, D), np.float32)
    vc = np.zeros_like(kc)
    free = list(range(NB))[::-1]
    refcount = [0] * NB
    tables = [[0] * 8 for _ in range(S)]
    # the prompt is written once, for request 0
    for j in range(-(-prompt // bs)):
        tables[0][j] = free.pop()
        refcount[tables[0][j]] = 1
    pk = rng.standard_normal((prompt, H, D)).astype(np.float32)
    pv = rng.standard_normal((prompt, H, D)).astype(np.float32)
    O.append(pk, pv, O.F32, [tables[0][p // bs] * bs + p % bs for p in range(prompt)], bs, kc, vc)
    # the other requests fork: their tables list the same block ids
    for b in range(1, S):
        tables[b] = list(tables[0])
        for j in range(-(-prompt // bs)):
            refcount[tables[0][j]] += 1
    full_block = tables[0][0]
    full_rows = (kc[full_block].copy(), vc[full_block].copy())
    lens = [prompt] * S
    own_k = [[] for _ in range(S)]
    own_v = [[] for _ in range(S)]
    copies = 0
    for _ in range(steps):
        pairs, slots = _cow_model_step(tables, lens, refcount, free, bs)
        copies += len(pairs)
        if pairs:
            O.block_copy([p[0] for p in pairs], [p[1] for p in pairs], bs, kc, vc)
        nk = rng.standard_normal((S, H, D)).astype(np.float32)
        nv = rng.standard_normal((S, H, D)).astype(np.float32)
        O.append(nk, nv, O.F32, np.array(slots, np.int32), bs, kc, vc)
        for b in range(S):
            own_k[b].append(nk[b])
            own_v[b].append(nv[b])
            lens[b] += 1
    # the partly filled prompt block was copied for all but the last request
    assert copies == S - 1
    # the full prompt block is still shared and untouched
    assert refcount[full_block] == S
    assert np.array_equal(kc[full_block], full_rows[0])
    assert np.array_equal(vc[full_block], full_rows[1])
    q = rng.standard_normal((S, H, D)).astype(np.float32)
    tb = np.array(tables, np.int32)
    out = O.paged_decode_attention(q, O.F32, kc, vc, O.F32, tb, np.array(lens, np.int32), 0.3)
    for b in range(S):
        rk = np.concatenate([pk, np.stack(own_k[b])])
        rv = np.concatenate([pv, np.stack(own_v[b])])
        for h in range(H):
            ref = O.attend_rows(q[b, h].astype(np.float64), rk[:, h], rv[:, h], 0.3)
            assert np.array_equal(out[b, h], ref)


# ------------------------------------------------------------------ host bookkeeping
def _fork_pool(NB=24, bs=4, S=3, prompt=6, maxb=8):
    p = pkv.kv_block_pool_init(NB, bs, 1, 64, pkv.PKV_F16)
    tables = np.zeros((S, maxb), np.int32)
    pkv.kv_reserve_slots(p, [0], tables[:1], num_new=[prompt])
    nb = -(-prompt // bs)
    for b in range(1, S):
        tables[b, :nb] = tables[0, :nb]
        pkv.kv_block_share(p, tables[0, :nb])
    return p, tables


def test_reserve_slots_cow_copies_shared_partial_blocks_only():
    bs, S, prompt = 4, 3, 6
    p, tables = _fork_pool(bs=bs, S=S, prompt=prompt)
    full, part = int(tables[0, 0]), int(tables[0, 1])
    free0 = pkv.kv_num_free_blocks(p)
    lens = np.full(S, prompt, np.int32)
    slots, src, dst = pkv.kv_reserve_slots_cow(p, lens, tables)
    # requests 0 and 1 copy the incomplete last block; request 2 then holds it alone
    assert list(src) == [part, part]
    assert len(set(dst.tolist())) == 2 and part not in dst
    assert list(tables[:, 1]) == [dst[0], dst[1], part]
    assert pkv.kv_block_refcount(p, part) == 1
    for d in dst:
        assert pkv.kv_block_refcount(p, int(d)) == 1
    assert pkv.kv_block_refcount(p, full) == S
    assert pkv.kv_num_free_blocks(p) == free0 - 2
    assert list(slots) == [int(tables[b, 1]) * bs + prompt % bs for b in range(S)]
    # next step writes into private blocks: no copies
    slots, src, dst = pkv.kv_reserve_slots_cow(p, lens + 1, tables)
    assert src.size == 0 and dst.size == 0
    # a step that starts a block allocates, never copies
    p2, t2 = _fork_pool(bs=bs, S=S, prompt=8)
    s2, src2, _ = pkv.kv_reserve_slots_cow(p2, np.full(S, 8, np.int32), t2)
    assert src2.size == 0
    assert len(set(t2[:, 2].tolist())) == S


def test_reserve_slots_cow_with_prefill_and_idle_sequences():
    bs = 4
    p, tables = _fork_pool(bs=bs, S=3, prompt=6)
    part = int(tables[0, 1])
    # request 0 idle (it keeps holding the block), request 1 appends 5 tokens
    # (a copy, then one new block), request 2 one token (a copy too)
    slots, src, dst = pkv.kv_reserve_slots_cow(p, np.full(3, 6, np.int32), tables,
                                               num_new=[0, 5, 1])
    assert list(src) == [part, part]
    assert pkv.kv_block_refcount(p, part) == 1
    assert int(tables[0, 1]) == part
    assert [int(tables[1, 1]), int(tables[2, 1])] == [int(dst[0]), int(dst[1])]
    new = int(tables[1, 2])
    assert list(slots) == [int(dst[0]) * bs + 2, int(dst[0]) * bs + 3, new * bs, new * bs + 1,
                           new * bs + 2, int(dst[1]) * bs + 2]


def test_reserve_slots_cow_is_all_or_nothing():
    bs, S = 4, 3
    p, tables = _fork_pool(NB=3, bs=bs, S=S, prompt=6)   # 2 used, 1 free; needs 2 copies
    before = tables.copy()
    rc = [pkv.kv_block_refcount(p, i) for i in range(3)]
    with pytest.raises(pkv.PkvError) as e:
        pkv.kv_reserve_slots_cow(p, np.full(S, 6, np.int32), tables)
    assert e.value.status == pkv.PKV_ERR_NO_BLOCKS
    assert np.array_equal(tables, before)
    assert [pkv.kv_block_refcount(p, i) for i in range(3)] == rc
    # a written entry that is free is rejected without changes
    q, t = _fork_pool(bs=bs, S=1, prompt=6)
    t[0, 1] = 20                                         # a free block
    with pytest.raises(pkv.PkvError) as e:
        pkv.kv_reserve_slots_cow(q, [6], t)
    assert e.value.status == pkv.PKV_ERR_INVALID


def test_block_copy_argument_checks_without_a_device():
    p = pkv.kv_block_pool_init(4, 16, 1, 64, pkv.PKV_F16)
    lib = pkv.load()
    assert lib.kv_block_copy(p.handle, None, None, 0, None, None, None, None, None) == pkv.PKV_OK
    assert lib.kv_block_copy(p.handle, None, None, 1, None, None, None, None, None) == \
        pkv.PKV_ERR_INVALID
    assert lib.kv_block_copy(p.handle, None, None, -1, None, None, None, None, None) == \
        pkv.PKV_ERR_INVALID
