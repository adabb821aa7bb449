"""GPU parity: libpkv's CUDA kernels against the fp64 CPU oracle.

Slot mapping, appended cache contents and int8 codes/scales must match bit
for bit; attention output within 2e-3 (fp32/fp16/bf16 K/V) or 2e-2 (int8 K/V)
max-abs of the oracle.  Every call goes through the C ABI (ctypes binding).
"""
import dataclasses

import numpy as np
import pytest
import torch

from paged_kv_cache_273_gb300 import pkv
from paged_kv_cache_273_gb300 import workloads as W

from parity_harness import Guarded, attend_gpu, attend_oracle, build, run, to_device

pytestmark = pytest.mark.gpu


def _assert_ok(res):
    assert res["cache_equal_history"], "history append differs from the oracle"
    assert res["cache_equal"], "cache after the decode steps differs from the oracle"
    assert res["max_err"] <= res["tol"], res
    assert res["error_word"] == pkv.PKV_OK
    assert res["guards"], "a canary around a device buffer was overwritten"
    assert res["counters_zero"], "a split-merge counter was left non-zero"


# ------------------------------------------------------------------ the five workloads
def test_tiny():
    _assert_ok(run(W.make_inputs("tiny")))


def test_tiny_other_reading():
    # 7 and 3 read as the lengths before the decode step: the step fills the
    # last block of each sequence exactly.
    _assert_ok(run(W.make_inputs("tiny", lengths=(8, 4))))


def test_gpt2_small():
    _assert_ok(run(W.make_inputs("gpt2")))


def test_llama3_8b_64_steps():
    # all 64 appends are checked bit for bit through the final cache; attention
    # is checked at the first steps, across a block boundary and at the end.
    _assert_ok(run(W.make_inputs("llama3_8b"), check_steps=[0, 1, 15, 16, 17, 63]))


def test_llama2_70b_shared_prefix():
    _assert_ok(run(W.make_inputs("llama2_70b")))


def test_int8_cache():
    _assert_ok(run(W.make_inputs("int8")))


# ------------------------------------------------------------------ shapes and edges
def _custom(name, Hq, Hkv, D, bs, kv, lengths, q=None, src=None, seed=7, steps=1):
    base = W.Workload(name, Hq, Hkv, D, bs, len(lengths), kv, q if q is not None else
                      (W.F16 if kv == W.I8 else kv), src if src is not None else
                      (W.F16 if kv == W.I8 else kv), seed, "uniform", 1, 2, steps)
    return W.make_inputs(base, lengths=lengths)


EDGE_LENGTHS = [1, 2, 15, 16, 17, 31, 32, 33, 100, 0, 1000, 4097]


@pytest.mark.parametrize("kv", [W.F32, W.F16, W.BF16, W.I8])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_dtype_head_dim_group_grid(kv, D, G):
    Hkv = 2
    inp = _custom("grid", Hkv * G, Hkv, D, 16, kv, EDGE_LENGTHS, seed=100 + D + G + 7 * kv)
    _assert_ok(run(inp))


@pytest.mark.parametrize("bs", [4, 8, 16, 32, 64, 128])
def test_block_sizes(bs):
    kv = W.BF16
    inp = _custom("bs", 8, 2, 128, bs, kv, [1, bs - 1, bs, bs + 1, 3 * bs + 5, 777], seed=bs)
    _assert_ok(run(inp))


@pytest.mark.parametrize("bs", [8, 32])
def test_int8_block_sizes(bs):
    inp = _custom("bs8", 8, 2, 128, bs, W.I8, [1, bs, bs + 1, 500], seed=3 + bs)
    _assert_ok(run(inp))


# Multi-tile work units (a stage of 2 or 4 tiles gathered by rows of
# min(bs, 16, unit / 4) tokens) across block sizes: 16-bit d 64 and 8-bit
# rows at one head per KV head on the CUDA cores, 8-bit and 4-bit rows on
# the tensor cores.
UNIT_CASES = [(W.F16, 64, 1, bs) for bs in (4, 8, 32, 128)] + \
             [(W.BF16, 64, 1, 8)] + \
             [(W.I8, 128, 4, bs) for bs in (8, 64)] + \
             [(W.I8, 128, 1, bs) for bs in (8, 128)] + \
             [(W.I4, 128, 4, bs) for bs in (64, 128)] + \
             [(W.I4, 128, 1, bs) for bs in (8, 64)]


@pytest.mark.parametrize("kv,D,G,bs", UNIT_CASES)
def test_work_units_across_block_sizes(kv, D, G, bs):
    q = W.F16 if kv in (W.I8, W.I4) else kv
    lengths = [1, bs - 1 if bs > 1 else 1, 31, 32, 33, 63, 64, 65, 129, 0, 777]
    inp = _custom("units", 2 * G, 2, D, bs, kv, lengths, q=q, src=q, seed=53 + bs + kv)
    _assert_ok(run(inp))


def test_int8_with_bf16_queries_and_f32_source():
    inp = _custom("q8b", 8, 2, 128, 16, W.I8, [5, 300, 17], q=W.BF16, src=W.F32, seed=31)
    _assert_ok(run(inp))


def test_mqa_single_kv_head():
    inp = _custom("mqa", 8, 1, 128, 16, W.F16, [3000, 1, 64, 65], seed=41)
    _assert_ok(run(inp))


def test_one_long_sequence_split_over_all_ctas():
    inp = _custom("long", 8, 1, 128, 16, W.BF16, [70000], seed=43)
    _assert_ok(run(inp))


def test_fewer_tiles_than_ctas():
    inp = _custom("few", 4, 2, 64, 16, W.F16, [3, 20], seed=47)
    _assert_ok(run(inp))


@pytest.mark.parametrize("lens", [[1, 15, 16, 17, 53, 777], [33], [16, 16, 16, 40],
                                  [2000, 3, 70, 0, 129]])
def test_split_sequences_with_idle_ctas(lens):
    # fewer 16-token tiles than SMs, so some CTAs own no tile while
    # multi-tile sequences are still split across several CTAs
    inp = _custom("idle", 8, 2, 128, 16, W.BF16, lens, seed=len(lens))
    _assert_ok(run(inp))


def test_many_short_sequences():
    rng = np.random.default_rng(53)
    lens = rng.integers(1, 40, size=1500).tolist()
    inp = _custom("short", 4, 1, 64, 16, W.F16, lens, seed=53)
    _assert_ok(run(inp))


def test_all_sequences_empty():
    inp = _custom("empty", 4, 2, 64, 16, W.F16, [0, 0, 0], seed=59)
    res = run(inp)
    assert res["max_err"] == 0.0 and res["error_word"] == pkv.PKV_OK


def test_repeat_calls_are_deterministic_and_reset_counters():
    inp = W.make_inputs("llama2_70b")
    case = build(inp)
    from parity_harness import append_step
    append_step(case, 0)
    a = attend_gpu(case, 0)
    b = attend_gpu(case, 0)
    assert np.array_equal(a, b)
    ncnt = inp.workload.batch * inp.workload.num_kv_heads
    assert not case.workspace[:ncnt * 4].view(torch.int32).any().item()
    want = attend_oracle(case, 0)
    assert np.max(np.abs(a - want)) <= 2e-3


# ------------------------------------------------------------------ bad indices
def _small_pool(kv=W.F16, NB=8, bs=16, Hkv=2, D=64):
    pool = pkv.kv_block_pool_init(NB, bs, Hkv, D, kv)
    k = Guarded((NB, Hkv, bs, D), torch.float16)
    v = Guarded((NB, Hkv, bs, D), torch.float16)
    return pool, k, v


def test_append_bad_slot_sets_error_and_writes_nothing_outside():
    pool, k, v = _small_pool()
    rows = torch.ones((3, 2, 64), dtype=torch.float16, device="cuda")
    slots = torch.tensor([0, 8 * 16, -1], dtype=torch.int32, device="cuda")   # 128 = NB*bs
    pkv.kv_append(pool, rows, rows, slots, k.tensor, v.tensor)
    assert pkv.pkv_check_error(pool) == pkv.PKV_ERR_BAD_INDEX
    assert pkv.pkv_check_error(pool) == pkv.PKV_OK          # cleared
    assert k.intact() and v.intact()
    assert k.tensor[0, :, 0].float().sum().item() == 128.0
    assert k.tensor.float().sum().item() == 128.0


def test_attention_bad_block_id_and_bad_length():
    pool, k, v = _small_pool()
    q = torch.randn((2, 4, 64), dtype=torch.float16, device="cuda")
    out = torch.zeros((2, 4, 64), dtype=torch.float32, device="cuda")
    ws = pkv.alloc_workspace(pool, 2, 4)
    tables = torch.tensor([[0, 99], [1, 2]], dtype=torch.int32, device="cuda")
    lens = torch.tensor([20, 5], dtype=torch.int32, device="cuda")
    pkv.paged_decode_attention(pool, q, k.tensor, v.tensor, tables, lens, 0.125, out, ws, 20)
    assert pkv.pkv_check_error(pool) == pkv.PKV_ERR_BAD_INDEX
    lens = torch.tensor([5, 33], dtype=torch.int32, device="cuda")          # > 2 blocks * 16
    pkv.paged_decode_attention(pool, q, k.tensor, v.tensor, tables, lens, 0.125, out, ws, 40)
    assert pkv.pkv_check_error(pool) == pkv.PKV_ERR_BAD_INDEX
    assert not out[1].any().item()                           # treated as empty
    assert k.intact() and v.intact()
    # the workspace is still usable: a valid call afterwards is correct
    tables = torch.tensor([[0, 3], [1, 2]], dtype=torch.int32, device="cuda")
    lens = torch.tensor([20, 5], dtype=torch.int32, device="cuda")
    pkv.paged_decode_attention(pool, q, k.tensor, v.tensor, tables, lens, 0.125, out, ws, 20)
    assert pkv.pkv_check_error(pool) == pkv.PKV_OK


def test_host_validation_errors():
    pool, k, v = _small_pool()
    q = torch.randn((1, 4, 64), dtype=torch.bfloat16, device="cuda")      # wrong q dtype
    out = torch.zeros((1, 4, 64), dtype=torch.float32, device="cuda")
    ws = pkv.alloc_workspace(pool, 1, 4)
    tables = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    lens = torch.ones(1, dtype=torch.int32, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_attention(pool, q, k.tensor, v.tensor, tables, lens, 0.1, out, ws, 1)
    assert e.value.status == pkv.PKV_ERR_INVALID
    q = torch.randn((1, 6, 64), dtype=torch.float16, device="cuda")       # G = 3
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_attention(pool, q, k.tensor, v.tensor, tables, lens, 0.1,
                                   torch.zeros((1, 6, 64), device="cuda"), ws, 1)
    assert e.value.status == pkv.PKV_ERR_UNSUPPORTED
    small = torch.zeros(16, dtype=torch.uint8, device="cuda")
    q = torch.randn((1, 4, 64), dtype=torch.float16, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_attention(pool, q, k.tensor, v.tensor, tables, lens, 0.1, out, small, 1)
    assert e.value.status == pkv.PKV_ERR_INVALID


def test_reserve_slots_drives_a_decode_loop():
    """Host allocation (a block only when the last one is full) feeding the
    device append and attention for a few steps, checked against the oracle."""
    from oracle import oracle as O
    rng = np.random.default_rng(61)
    B, Hq, Hkv, D, bs, NB = 3, 8, 2, 128, 16, 64
    pool = pkv.kv_block_pool_init(NB, bs, Hkv, D, pkv.PKV_BF16)
    kc, vc, _, _ = pool.alloc_cache()
    ok = np.zeros((NB, Hkv, bs, D), np.uint16)
    ov = np.zeros_like(ok)
    tables = np.zeros((B, 8), np.int32)
    lens = np.zeros(B, np.int32)
    ws = pkv.alloc_workspace(pool, B, Hq)
    prompt = np.array([5, 16, 31], np.int32)
    for step in range(40):
        n_new = prompt if step == 0 else np.ones(B, np.int32)
        slots = pkv.kv_reserve_slots(pool, lens, tables, n_new)
        assert np.array_equal(slots, O.slot_mapping(tables, bs, lens, n_new))
        T = int(n_new.sum())
        bits = (rng.standard_normal((2, T, Hkv, D)).astype(np.float32).view(np.uint32) >> 16) \
            .astype(np.uint16)
        pkv.kv_append(pool, to_device(bits[0], W.BF16), to_device(bits[1], W.BF16),
                      torch.from_numpy(slots).cuda(), kc, vc)
        O.append(bits[0], bits[1], O.BF16, slots, bs, ok, ov)
        lens = lens + n_new
        used = -(-lens // bs)
        assert NB - pkv.kv_num_free_blocks(pool) == int(used.sum())
        qb = (rng.standard_normal((B, Hq, D)).astype(np.float32).view(np.uint32) >> 16) \
            .astype(np.uint16)
        out = torch.empty((B, Hq, D), dtype=torch.float32, device="cuda")
        pkv.paged_decode_attention(pool, to_device(qb, W.BF16), kc, vc,
                                   torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                                   D ** -0.5, out, ws, int(lens.max()))
        want = O.paged_decode_attention(qb, O.BF16, ok, ov, O.BF16, tables, lens, D ** -0.5)
        assert np.max(np.abs(out.cpu().numpy() - want)) <= 2e-3
    assert pkv.pkv_check_error(pool) == pkv.PKV_OK


@pytest.mark.gpu
def test_gpu_bounded_wait_reports_timeout_and_device_stays_usable():
    """A kernel waits on an mbarrier phase that nothing completes; the bounded
    wait gives up (about a second), the error word says PKV_ERR_TIMEOUT, and
    the next attention call on the same device runs and matches the oracle."""
    import time
    pool = pkv.kv_block_pool_init(4, 16, 1, 64, W.F16)
    t0 = time.perf_counter()
    pkv.pkv_selftest_wait_timeout(pool)
    assert pkv.pkv_check_error(pool) == pkv.PKV_ERR_TIMEOUT
    assert time.perf_counter() - t0 < 30.0
    assert pkv.pkv_check_error(pool) == pkv.PKV_OK     # the word was cleared
    r = run(W.make_inputs("tiny"))
    assert r["max_err"] <= r["tol"] and r["error_word"] == pkv.PKV_OK
