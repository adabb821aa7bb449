"""CPU tests of the C ABI: the library loads and exports every declared
symbol; the host pool, slot bookkeeping and argument validation behave as
the header states (no GPU needed)."""
import os
import re

import numpy as np
import pytest

from oracle import oracle as O
from paged_kv_cache_273_gb300 import pkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "pkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\**\s*([a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol():
    lib = pkv.load()
    declared = _declared_functions()
    assert len(declared) >= 16
    assert sorted(pkv.SYMBOLS) == declared
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings():
    assert pkv.status_string(0) == "ok"
    assert "free blocks" in pkv.status_string(pkv.PKV_ERR_NO_BLOCKS)


def test_pool_init_validation():
    for args in [(0, 16, 8, 128, 2), (16, 12, 8, 128, 2), (16, 512, 8, 128, 2), (16, 16, 0, 128, 2),
                 (16, 16, 8, 128, 9), (1 << 28, 16, 8, 128, 2)]:
        with pytest.raises(pkv.PkvError) as e:
            pkv.kv_block_pool_init(*args)
        assert e.value.status == pkv.PKV_ERR_INVALID, args
    for args in [(16, 16, 8, 96, 2), (16, 4, 8, 128, 3), (16, 2, 8, 128, 2)]:
        with pytest.raises(pkv.PkvError) as e:
            pkv.kv_block_pool_init(*args)
        assert e.value.status == pkv.PKV_ERR_UNSUPPORTED, args


def test_cache_sizes():
    p = pkv.kv_block_pool_init(10, 16, 8, 128, pkv.PKV_BF16)
    assert pkv.kv_cache_bytes(p) == 10 * 8 * 16 * 128 * 2
    assert pkv.kv_scales_bytes(p) == 0
    q = pkv.kv_block_pool_init(10, 16, 8, 128, pkv.PKV_I8)
    assert pkv.kv_cache_bytes(q) == 10 * 8 * 16 * 128
    assert pkv.kv_scales_bytes(q) == 10 * 8 * 16 * 2


def test_alloc_share_free_refcounts():
    p = pkv.kv_block_pool_init(6, 16, 1, 64, pkv.PKV_F16)
    a = pkv.kv_block_alloc(p, 4)
    assert a.tolist() == [0, 1, 2, 3] and pkv.kv_num_free_blocks(p) == 2
    with pytest.raises(pkv.PkvError) as e:
        pkv.kv_block_alloc(p, 3)                      # all-or-nothing
    assert e.value.status == pkv.PKV_ERR_NO_BLOCKS and pkv.kv_num_free_blocks(p) == 2
    pkv.kv_block_share(p, [1, 2])                     # a second request shares a prefix
    assert [pkv.kv_block_refcount(p, i) for i in range(6)] == [1, 2, 2, 1, 0, 0]
    pkv.kv_block_free(p, [0, 1, 2])
    assert [pkv.kv_block_refcount(p, i) for i in range(6)] == [0, 1, 1, 1, 0, 0]
    assert pkv.kv_num_free_blocks(p) == 3
    with pytest.raises(pkv.PkvError):
        pkv.kv_block_free(p, [0])                     # already free
    with pytest.raises(pkv.PkvError):
        pkv.kv_block_free(p, [3, 3])                  # repeats count
    assert pkv.kv_block_refcount(p, 3) == 1
    with pytest.raises(pkv.PkvError):
        pkv.kv_block_share(p, [4])                    # cannot share a free block
    with pytest.raises(pkv.PkvError):
        pkv.kv_block_free(p, [6])
    pkv.kv_block_free(p, [1, 2, 3])
    assert pkv.kv_num_free_blocks(p) == 6
    b = pkv.kv_block_alloc(p, 6)
    assert sorted(b.tolist()) == list(range(6))


def test_reserve_slots_matches_oracle_and_wastes_at_most_one_block():
    rng = np.random.default_rng(0)
    for bs in (4, 16, 64):
        B, maxb = 12, 40
        NB = B * maxb
        p = pkv.kv_block_pool_init(NB, bs, 2, 64, pkv.PKV_F16)
        tables = np.zeros((B, maxb), np.int32)
        lens = np.zeros(B, np.int32)
        for step in range(30):
            room = maxb * bs - lens
            n_new = np.minimum(rng.integers(0, 3 * bs, size=B), room).astype(np.int32)
            slots = pkv.kv_reserve_slots(p, lens, tables, n_new)
            want = O.slot_mapping(tables, bs, lens, n_new)
            assert np.array_equal(slots, want)
            lens = lens + n_new
            blocks = -(-lens // bs)
            # blocks are allocated on demand: each sequence ends with at
            # most one block that is not full
            waste = blocks * bs - lens
            assert np.all((waste >= 0) & (waste < bs))
            assert NB - pkv.kv_num_free_blocks(p) == int(blocks.sum())
            used = np.concatenate([tables[b, :blocks[b]] for b in range(B)])
            assert len(set(used.tolist())) == used.size     # no block given twice
        # freeing every sequence returns every block
        for b in range(B):
            pkv.kv_block_free(p, tables[b, :-(-lens[b] // bs)])
        assert pkv.kv_num_free_blocks(p) == NB


def test_reserve_slots_is_all_or_nothing():
    p = pkv.kv_block_pool_init(3, 4, 1, 64, pkv.PKV_F32)
    tables = np.zeros((2, 4), np.int32)
    with pytest.raises(pkv.PkvError) as e:
        pkv.kv_reserve_slots(p, [0, 0], tables, [8, 8])  # needs 4 blocks
    assert e.value.status == pkv.PKV_ERR_NO_BLOCKS
    assert pkv.kv_num_free_blocks(p) == 3 and not tables.any()
    with pytest.raises(pkv.PkvError) as e:
        pkv.kv_reserve_slots(p, [0, 0], tables, [17, 0])  # overflows the table row
    assert e.value.status == pkv.PKV_ERR_INVALID


def test_slot_mapping_matches_oracle():
    rng = np.random.default_rng(1)
    tables = rng.permutation(200).reshape(10, 20).astype(np.int32)
    for bs in (1, 4, 16):
        start = rng.integers(0, 20 * bs, size=10).astype(np.int32)
        n = np.array([rng.integers(0, 20 * bs - s + 1) for s in start], np.int32)
        got = pkv.kv_slot_mapping(tables, bs, start, n)
        want = O.slot_mapping(tables, bs, start, n)
        assert np.array_equal(got, want)
    with pytest.raises(pkv.PkvError):
        pkv.kv_slot_mapping(tables, 4, np.full(10, 79, np.int32), np.full(10, 2, np.int32))


def test_slot_mapping_into_a_given_array():
    # the in-place form a serving loop uses: slots written straight into a
    # slice of a staging buffer, equal to the returned form
    rng = np.random.default_rng(2)
    tables = rng.permutation(200).reshape(10, 20).astype(np.int32)
    start = rng.integers(0, 20 * 16, size=10).astype(np.int32)
    stage = np.full(64, 0x7F, np.uint8)
    out = stage[8:48].view(np.int32)
    got = pkv.kv_slot_mapping(tables, 16, start, out=out)
    assert got.ctypes.data == out.ctypes.data
    assert np.array_equal(out, O.slot_mapping(tables, 16, start, np.ones(10, np.int32)))
    assert (stage[:8] == 0x7F).all() and (stage[48:] == 0x7F).all()
    for bad in (np.zeros(9, np.int32), np.zeros(10, np.int64), np.zeros(20, np.int32)[::2]):
        with pytest.raises(ValueError):
            pkv.kv_slot_mapping(tables, 16, start, out=bad)


def test_workspace_size_formula_is_monotone():
    p = pkv.kv_block_pool_init(10, 16, 8, 128, pkv.PKV_BF16)
    a = pkv.paged_decode_workspace_bytes(p, 16, 32)
    b = pkv.paged_decode_workspace_bytes(p, 32, 32)
    c = pkv.paged_decode_workspace_bytes(p, 16, 64)
    assert 0 < a < b and a < c
    assert pkv.paged_decode_workspace_bytes(p, 16, 12) == 0      # not a multiple of Hkv


def test_device_calls_without_a_device_report_cuda_error():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    import ctypes
    lib = pkv.load()
    h = ctypes.c_void_p()
    assert lib.kv_block_pool_init(ctypes.byref(h), 4, 16, 1, 64, pkv.PKV_F16) == 0
    buf = (ctypes.c_uint8 * 4096)()
    addr = (ctypes.addressof(buf) + 15) // 16 * 16
    rc = lib.kv_append(h, addr, addr, pkv.PKV_F16, addr, 1, addr, addr, None, None, None)
    assert rc == pkv.PKV_ERR_CUDA
    assert lib.pkv_check_error(h, None) == pkv.PKV_ERR_CUDA
    lib.kv_block_pool_destroy(h)
