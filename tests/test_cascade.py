"""Shared-prefix (cascade) decode: host grouping on the CPU, GPU parity.

[VIS] "PagedAttention: the cache in blocks": sequences that begin with the
same prompt tokens can reference one stored copy of those tokens' blocks.
paged_decode_attention_cascade reads such a shared prefix once per group:
a prefix pass scores it for all members' q heads together, and the decode
pass attends each sequence over its own rows only, folding the prefix
partials in.  The result is plain attention ([NOTES] "Concept") over every
sequence's rows, so the oracle is unchanged: the fp64 paged decode oracle.
"""
import numpy as np
import pytest

from oracle import oracle as O
from paged_kv_cache_273_gb300 import pkv


# ------------------------------------------------------------------ host grouping (CPU)
def _groups_reference(tables, lens, bs, min_blocks):
    """Written separately: for every first block shared by >= 2 sequences of
    >= min_blocks whole blocks, the common run of leading entries, capped at
    the shortest member."""
    B = len(lens)
    by_first = {}
    for b in range(B):
        if lens[b] >= min_blocks * bs:
            by_first.setdefault(int(tables[b][0]), []).append(b)
    out = {}
    for first, mem in by_first.items():
        if len(mem) < 2:
            continue
        minlen = min(int(lens[b]) for b in mem)
        nb = -(-minlen // bs)
        common = 0
        while common < nb and all(tables[b][common] == tables[mem[0]][common] for b in mem):
            common += 1
        P = min(common * bs, minlen)
        if common >= min_blocks and P > 0:
            out[tuple(sorted(mem))] = P
    return out


def _as_dict(g):
    res = {}
    for i in range(g["num_groups"]):
        mem = tuple(int(x) for x in g["group_seqs"][g["group_start"][i]:g["group_start"][i + 1]])
        res[mem] = int(g["group_prefix"][i])
    return res


@pytest.mark.parametrize("seed", range(12))
def test_prefix_groups_match_a_separate_reference(seed):
    rng = np.random.default_rng(seed)
    bs = int(rng.choice([4, 16]))
    B = int(rng.integers(1, 40))
    maxb = 12
    lens = rng.integers(0, maxb * bs + 1, size=B).astype(np.int32)
    tables = rng.permutation(B * maxb + 50)[:B * maxb].reshape(B, maxb).astype(np.int32)
    # plant shared prefixes of random lengths among random subsets
    for _ in range(int(rng.integers(0, 4))):
        mem = rng.choice(B, size=int(rng.integers(2, max(3, B // 2 + 1))), replace=True)
        n = int(rng.integers(1, maxb + 1))
        donor = tables[mem[0], :n].copy()
        for b in mem:
            tables[b, :n] = donor
    min_blocks = int(rng.choice([1, 2]))
    g = pkv.kv_prefix_groups(tables, lens, bs, min_blocks)
    want = _groups_reference(tables, lens, bs, min_blocks)
    assert _as_dict(g) == want
    sp = np.zeros(B, np.int32)
    for mem, P in want.items():
        sp[list(mem)] = P
    assert np.array_equal(g["seq_prefix"], sp)
    assert g["max_prefix_len"] == max(want.values(), default=0)
    assert g["max_group_size"] == max((len(m) for m in want), default=0)


def test_prefix_groups_properties():
    # members agree on the prefix's blocks; the prefix fits every member
    rng = np.random.default_rng(7)
    bs, B, maxb = 16, 30, 20
    lens = rng.integers(1, maxb * bs + 1, size=B).astype(np.int32)
    tables = rng.permutation(B * maxb).reshape(B, maxb).astype(np.int32)
    tables[3:20, :7] = tables[3, :7]
    lens[3:20] = np.maximum(lens[3:20], 100)
    g = pkv.kv_prefix_groups(tables, lens, bs)
    assert g["num_groups"] == 1
    mem = g["group_seqs"]
    P = int(g["group_prefix"][0])
    assert list(mem) == list(range(3, 20))
    assert P == min(7 * bs, int(lens[3:20].min()))
    for b in mem:
        assert lens[b] >= P
        assert np.array_equal(tables[b, :-(-P // bs)], tables[mem[0], :-(-P // bs)])


def test_prefix_groups_rejects_bad_arguments():
    t = np.zeros((2, 2), np.int32)
    with pytest.raises(pkv.PkvError):
        pkv.kv_prefix_groups(t, np.array([1, 99], np.int32), 4)      # length beyond its row
    with pytest.raises(pkv.PkvError):
        pkv.kv_prefix_groups(t, np.array([1, 1], np.int32), 4, 0)    # min_prefix_blocks < 1


# ------------------------------------------------------------------ GPU parity
_RAW = {pkv.PKV_F16: np.float16, pkv.PKV_BF16: None}


def _bits(x, dt):
    if dt == pkv.PKV_F16:
        return x.astype(np.float16).view(np.uint16)
    return (x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _cascade_case(dt, D, Hq, Hkv, bs, lens, share, prefix_blocks, seed, min_blocks=1):
    """share: list of member lists; each group's first prefix_blocks table
    entries are made identical.  Returns (max error vs the oracle, max error
    of the plain decode path vs the oracle, status, groups)."""
    import torch
    rng = np.random.default_rng(seed)
    B = len(lens)
    maxb = max(-(-L // bs) for L in lens) + 1
    NB = B * maxb + 8
    tables = rng.permutation(NB)[:B * maxb].reshape(B, maxb).astype(np.int32)
    for mem, pb in zip(share, prefix_blocks):
        tables[mem, :pb] = tables[mem[0], :pb]
    kc = _bits(rng.standard_normal((NB, Hkv, bs, D)), dt)
    vc = _bits(rng.standard_normal((NB, Hkv, bs, D)), dt)
    q = _bits(rng.standard_normal((B, Hq, D)), dt)
    lens = np.array(lens, np.int32)
    scale = 1.0 / np.sqrt(D)
    want = O.paged_decode_attention(q, dt, kc, vc, dt, tables, lens, float(np.float32(scale)))
    tdt = torch.float16 if dt == pkv.PKV_F16 else torch.bfloat16
    dev = torch.device("cuda", 0)
    todev = lambda a: torch.from_numpy(a.view(np.int16)).to(dev).view(tdt)  # noqa: E731
    pool = pkv.kv_block_pool_init(NB, bs, Hkv, D, dt)
    kd, vd, qd = todev(kc), todev(vc), todev(q)
    td = torch.from_numpy(tables).to(dev)
    ld = torch.from_numpy(lens).to(dev)
    g = pkv.kv_prefix_groups(tables, lens, bs, min_blocks)
    gd = pkv.prefix_groups_to_device(g, dev)
    ws = pkv.alloc_cascade_workspace(pool, B, Hq, g["max_prefix_len"], dev)
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device=dev)
    max_len = int(lens.max())
    pkv.paged_decode_attention_cascade(pool, qd, kd, vd, td, ld, scale, out, ws, max_len, gd)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    status = pkv.pkv_check_error(pool)
    # the plain path on the same inputs
    ws2 = pkv.alloc_workspace(pool, B, Hq, dev)
    out2 = torch.empty_like(out)
    pkv.paged_decode_attention(pool, qd, kd, vd, td, ld, scale, out2, ws2, max_len)
    torch.cuda.synchronize()
    plain = out2.cpu().numpy()
    return (float(np.max(np.abs(got - want))), float(np.max(np.abs(plain - want))), status, g,
            bool(np.isfinite(got).all()))


@pytest.mark.gpu
@pytest.mark.parametrize("dt", [pkv.PKV_F16, pkv.PKV_BF16])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_gpu_cascade_group_sizes(dt, G):
    # one group of 5 with a 64-row prefix, one of 3 with a 23-row prefix
    # capped by its shortest member (23 < 2 blocks), one sequence alone
    lens = [200, 130, 90, 70, 65, 23, 50, 44, 300]
    share = [[0, 1, 2, 3, 4], [5, 6, 7]]
    err, plain, status, g, finite = _cascade_case(dt, 128, 4 * G, 4, 16, lens, share, [4, 3], 10 + G)
    assert g["num_groups"] == 2 and g["max_prefix_len"] == 64
    assert status == pkv.PKV_OK and finite
    assert err <= 2e-3, err
    assert plain <= 2e-3, plain


@pytest.mark.gpu
@pytest.mark.parametrize("D,bs", [(64, 16), (128, 4), (128, 32), (64, 8)])
def test_gpu_cascade_head_dims_and_block_sizes(D, bs):
    lens = [33 * bs // 4 + 5, 40 * bs // 4, 25 * bs // 4 + 1, 7]
    share = [[0, 1, 2]]
    err, plain, status, g, finite = _cascade_case(pkv.PKV_BF16, D, 16, 2, bs, lens, share,
                                                  [24 // (bs // 4) if bs >= 4 else 6], 21)
    assert g["num_groups"] == 1
    assert status == pkv.PKV_OK and finite
    assert err <= 2e-3, err


@pytest.mark.gpu
def test_gpu_cascade_many_members_and_a_member_with_no_own_rows():
    # 40 members x 8 heads = 320 query rows (two row tiles); member 3's
    # length equals the prefix, so its output is the prefix alone
    lens = [600] * 40
    lens[3] = 256
    share = [list(range(40))]
    err, plain, status, g, finite = _cascade_case(pkv.PKV_F16, 128, 64, 8, 16, lens, share, [16], 5)
    assert g["max_prefix_len"] == 256 and g["max_group_size"] == 40
    assert status == pkv.PKV_OK and finite
    assert err <= 2e-3, err


@pytest.mark.gpu
def test_gpu_cascade_long_prefix_in_several_chunks():
    # a 5000-row prefix: 40 key tiles, chunks of 3 tiles
    lens = [5100, 5007, 5600, 900]
    share = [[0, 1, 2]]
    err, plain, status, g, finite = _cascade_case(pkv.PKV_BF16, 128, 32, 8, 16, lens, share,
                                                  [313], 8)
    assert g["max_prefix_len"] == 5007 - 0 or g["max_prefix_len"] == 313 * 16
    assert status == pkv.PKV_OK and finite
    assert err <= 2e-3, err


@pytest.mark.gpu
def test_gpu_cascade_without_groups_is_plain_attention():
    lens = [100, 37, 5]
    err, plain, status, g, finite = _cascade_case(pkv.PKV_F16, 128, 8, 2, 16, lens, [], [], 3)
    assert g["num_groups"] == 0
    assert status == pkv.PKV_OK and finite
    assert err <= 2e-3


@pytest.mark.gpu
def test_gpu_cascade_llama2_70b_workload():
    """The Llama-2-70B-shaped workload (16 of 32 sequences share 64 blocks):
    cascade decode after one append step, against the oracle."""
    import torch
    from paged_kv_cache_273_gb300 import workloads as W
    from parity_harness import TOL, append_step, attend_oracle, build, to_device
    case = build(W.make_inputs("llama2_70b"))
    append_step(case, 0)
    wl = case.wl
    lens = case.inp.lens_after_step(0)
    g = pkv.kv_prefix_groups(case.inp.block_tables, lens, wl.block_size)
    assert g["num_groups"] == 1 and g["max_group_size"] == 16 and g["max_prefix_len"] == 1024
    gd = pkv.prefix_groups_to_device(g)
    ws = pkv.alloc_cascade_workspace(case.pool, wl.batch, wl.num_q_heads, g["max_prefix_len"])
    out = torch.full((wl.batch, wl.num_q_heads, wl.head_dim), float("nan"), dtype=torch.float32,
                     device="cuda")
    q = to_device(case.inp.step_q[0], wl.q_dtype)
    for _ in range(2):                      # the workspace's counters are left at zero
        pkv.paged_decode_attention_cascade(case.pool, q, case.gk.tensor, case.gv.tensor,
                                           case.tables_d, torch.from_numpy(lens).cuda(),
                                           1.0 / np.sqrt(wl.head_dim), out, ws, int(lens.max()), gd)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        want = attend_oracle(case, 0)
        assert np.max(np.abs(got - want)) <= TOL[wl.kv_dtype]
    assert pkv.pkv_check_error(case.pool) == pkv.PKV_OK
    n = wl.batch * wl.num_kv_heads
    assert not bool(ws[:n * 4].view(torch.int32).any().item())
    assert case.guards_intact()


@pytest.mark.gpu
def test_gpu_cascade_bad_prefix_length_is_reported():
    import torch
    dev = torch.device("cuda", 0)
    pool = pkv.kv_block_pool_init(8, 16, 1, 64, pkv.PKV_F16)
    kc, vc, _, _ = pool.alloc_cache(dev)
    q = torch.zeros((2, 1, 64), dtype=torch.float16, device=dev)
    tables = torch.tensor([[0, 1], [2, 3]], dtype=torch.int32, device=dev)
    lens = torch.tensor([20, 20], dtype=torch.int32, device=dev)
    g = {"group_start": np.array([0], np.int32), "group_seqs": np.zeros(0, np.int32),
         "group_prefix": np.zeros(0, np.int32), "seq_prefix": np.array([0, 30], np.int32),
         "num_groups": 0, "max_group_size": 0, "max_prefix_len": 0}
    gd = pkv.prefix_groups_to_device(g, dev)
    ws = pkv.alloc_cascade_workspace(pool, 2, 1, 0, dev)
    out = torch.zeros((2, 1, 64), dtype=torch.float32, device=dev)
    pkv.paged_decode_attention_cascade(pool, q, kc, vc, tables, lens, 0.1, out, ws, 32, gd)
    assert pkv.pkv_check_error(pool) == pkv.PKV_ERR_BAD_INDEX


def _random_cascade_shape(seed):
    rng = np.random.default_rng(8000 + seed)
    dt = int(rng.choice([pkv.PKV_F16, pkv.PKV_BF16]))
    D = int(rng.choice([64, 128]))
    Hkv = int(rng.choice([1, 2, 4]))
    G = int(rng.choice([1, 2, 4, 8]))
    bs = int(rng.choice([4, 8, 16, 32]))
    B = int(rng.integers(2, 21))
    lens = [int(rng.integers(1, 1500)) for _ in range(B)]
    # one to three groups of members sharing their first blocks (a member
    # may be shorter than the blocks it shares: the prefix is capped by it)
    share, pblocks, free = [], [], list(rng.permutation(B))
    for _ in range(int(rng.integers(1, 4))):
        if len(free) < 2:
            break
        n = int(rng.integers(2, min(len(free), 8) + 1))
        mem = sorted(int(x) for x in free[:n])
        free = free[n:]
        share.append(mem)
        pblocks.append(int(rng.integers(1, max(2, min(lens[m] for m in mem) // bs + 2))))
    return dt, D, Hkv * G, Hkv, bs, lens, share, pblocks


@pytest.mark.gpu
@pytest.mark.parametrize("seed", range(24))
def test_gpu_cascade_random_shapes(seed):
    # seeded random types, head sizes, groups, block sizes, sharing
    # patterns and lengths: the cascade and the plain path against the oracle
    dt, D, Hq, Hkv, bs, lens, share, pblocks = _random_cascade_shape(seed)
    err, plain, status, g, finite = _cascade_case(dt, D, Hq, Hkv, bs, lens, share, pblocks,
                                                  300 + seed)
    assert status == pkv.PKV_OK and finite
    assert err <= 2e-3, (err, dt, D, Hq, Hkv, bs, lens, share, pblocks)
    assert plain <= 2e-3, plain
