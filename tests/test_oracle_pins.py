"""Pins of the fp64 CPU oracle against what the pages and mathematics fix.

Each test checks the oracle against something other than itself: values the
pages print (tests/golden), library routines for the number formats, closed
forms and special cases of attention, invariances of the definition, and a
separately written brute force on tiny shapes.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- number formats
def test_half_decode_matches_numpy_for_every_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([O.half_to_double(int(b)) for b in bits])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got), np.isinf(ref))


@pytest.mark.filterwarnings("ignore::RuntimeWarning")
def test_bf16_decode_matches_float32_top_half_for_every_pattern():
    bits = np.arange(65536, dtype=np.uint32)
    ref = (bits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    got = np.array([O.bf16_to_double(int(b)) for b in bits])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


@pytest.mark.filterwarnings("ignore::RuntimeWarning")
def test_float_to_half_rne_matches_numpy():
    rng = np.random.default_rng(11)
    xs = [0.0, -0.0, 1.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6, 2.0 ** -24, 2.0 ** -25,
          3 * 2.0 ** -26, 2.0 ** -14, 2.0 ** -14 - 2.0 ** -25, 1.0 + 2.0 ** -11,
          1.0 + 3 * 2.0 ** -11, 0.0236220472]
    xs += list(rng.standard_normal(4000).astype(np.float32))
    xs += list((rng.standard_normal(4000) * 1e-5).astype(np.float32))
    xs += list((rng.standard_normal(2000) * 3e4).astype(np.float32))
    # exact ties between two halves, both parities
    for m in range(1024, 1100):
        xs.append(float(np.float32((m + 0.5) * 2.0 ** -10)))
    for x in xs:
        x32 = np.float32(x)
        want = int(np.array([x32], np.float32).astype(np.float16).view(np.uint16)[0])
        assert O.float_to_half_rne(x32) == want, x


# ---------------------------------------------------------------- slot mapping / append
def _walk_slots(table_row, block_size, length):
    """Position -> slot by walking the table: block after block, offset after offset."""
    slots = []
    for blk in table_row:
        for off in range(block_size):
            if len(slots) == length:
                return slots
            slots.append(int(blk) * block_size + off)
    return slots


@pytest.mark.parametrize("bs", [1, 4, 16])
def test_slot_mapping_matches_table_walk(bs):
    rng = np.random.default_rng(bs)
    B, maxb = 5, 7
    tables = rng.permutation(B * maxb).reshape(B, maxb).astype(np.int32)
    lens = rng.integers(0, maxb * bs + 1, size=B)
    start = np.zeros(B, np.int32)
    slots = O.slot_mapping(tables, bs, start, lens.astype(np.int32))
    want = []
    for b in range(B):
        want += _walk_slots(tables[b], bs, int(lens[b]))
    assert slots.tolist() == want


def test_append_then_gather_round_trip_and_untouched_cells():
    rng = np.random.default_rng(3)
    NB, H, bs, D = 12, 3, 4, 8
    B = 3
    lens = [5, 9, 1]
    perm = rng.permutation(NB).astype(np.int32)
    tables = np.full((B, 4), -1, np.int32)
    c = 0
    for b in range(B):
        n = -(-lens[b] // bs)
        tables[b, :n] = perm[c:c + n]
        c += n
    rows_k = rng.standard_normal((sum(lens), H, D)).astype(np.float32)
    rows_v = rng.standard_normal((sum(lens), H, D)).astype(np.float32)
    slots = O.slot_mapping(np.where(tables < 0, 0, tables), bs, np.zeros(B, np.int32),
                           np.array(lens, np.int32))
    canary = np.float32(-777.0)
    kc = np.full((NB, H, bs, D), canary, np.float32)
    vc = np.full((NB, H, bs, D), canary, np.float32)
    O.append(rows_k, rows_v, O.F32, slots, bs, kc, vc)
    off = 0
    touched = np.zeros((NB, bs), bool)
    for b in range(B):
        for h in range(H):
            got = O.gather(kc, None, O.F32, tables[b], lens[b], h, bs)
            assert np.array_equal(got, rows_k[off:off + lens[b], h].astype(np.float64))
            got = O.gather(vc, None, O.F32, tables[b], lens[b], h, bs)
            assert np.array_equal(got, rows_v[off:off + lens[b], h].astype(np.float64))
        for s in slots[off:off + lens[b]]:
            touched[s // bs, s % bs] = True
        off += lens[b]
    kt, vt = kc.transpose(0, 2, 1, 3), vc.transpose(0, 2, 1, 3)   # [NB, bs, H, D]
    assert np.all(kt[~touched] == canary) and np.all(vt[~touched] == canary)


def test_append_skips_padding_slots():
    kc = np.zeros((2, 1, 4, 8), np.float32)
    vc = np.zeros_like(kc)
    rows = np.ones((2, 1, 8), np.float32)
    O.append(rows, rows, O.F32, np.array([-1, 5], np.int32), 4, kc, vc)
    assert kc.sum() == 8 and kc[1, 0, 1].sum() == 8


def test_append_is_a_bit_copy_for_16_bit_rows():
    rng = np.random.default_rng(5)
    rows = rng.integers(0, 65536, size=(6, 2, 64)).astype(np.uint16)
    kc = np.zeros((4, 2, 4, 64), np.uint16)
    vc = np.zeros_like(kc)
    slots = np.array([3, 0, 15, 8, 9, 4], np.int32)
    O.append(rows, rows[::-1].copy(), O.BF16, slots, 4, kc, vc)
    for t, s in enumerate(slots):
        assert np.array_equal(kc[s // 4, :, s % 4], rows[t])
        assert np.array_equal(vc[s // 4, :, s % 4], rows[::-1][t])


# ---------------------------------------------------------------- int8 quantizer
def test_q8_unit_scale_rounds_half_to_even():
    # amax 127 -> scale 127/127 = 1.0 exactly (fp16 0x3C00), so codes are the
    # round-half-even integers of the inputs.
    x = np.zeros(128, np.float32)
    x[:7] = [127.0, -63.5, 0.5, -0.5, 1.5, 2.5, -2.5]
    codes, sb = O.quantize_row_q8(x)
    assert sb == 0x3C00
    assert codes[:7].tolist() == [127, -64, 0, 0, 2, 2, -2]
    assert not codes[7:].any()


def test_q8_divides_by_the_fp16_rounded_scale():
    # amax 1000: 1000/127 = 7.87401... in fp32 rounds to 7.875 in fp16 (0x47E0).
    # Divided by 7.875, 3.9375 is exactly 0.5 (-> 0), 11.8125 is 1.5 (-> 2),
    # 19.6875 is 2.5 (-> 2); divided by the unrounded scale they would round
    # the other way.  1000/7.875 = 126.98... -> 127.
    x = np.zeros(64, np.float32)
    x[:5] = [1000.0, 3.9375, 11.8125, 19.6875, -19.6875]
    codes, sb = O.quantize_row_q8(x)
    assert sb == 0x47E0
    assert codes[:5].tolist() == [127, 0, 2, 2, -2]


def test_q8_zero_row_and_single_nonzero():
    codes, sb = O.quantize_row_q8(np.zeros(128, np.float32))
    assert sb == 0 and not codes.any()
    # amax 3: 3/127 = 0.0236220... rounds to 1548 * 2^-16 = 0.0236206 (0x260C);
    # 3 / that = 127.0077 -> 127.
    x = np.zeros(128, np.float32)
    x[3] = -3.0
    codes, sb = O.quantize_row_q8(x)
    assert sb == 0x260C
    assert codes[3] == -127 and np.count_nonzero(codes) == 1


def test_q8_error_bound_symmetry_and_range():
    rng = np.random.default_rng(7)
    for trial in range(200):
        x = rng.standard_normal(128).astype(np.float32)
        mask = rng.random(128) < 0.01
        x = np.where(mask, x * 8, x).astype(np.float32)
        codes, sb = O.quantize_row_q8(x)
        s = O.half_to_double(sb)
        assert abs(s - np.abs(x).max() / 127) <= s * 2.0 ** -11 * 1.01
        assert codes.min() >= -127 and codes.max() <= 127
        assert np.abs(codes).max() == 127
        err = np.abs(x.astype(np.float64) - codes * s)
        assert np.all(err <= s / 2 * (1 + 2.0 ** -10) + 1e-12)
        neg, sb2 = O.quantize_row_q8(-x)
        assert sb2 == sb and np.array_equal(neg, -codes)


def test_q8_append_writes_codes_and_scales_at_slots():
    rng = np.random.default_rng(9)
    T, H, D, bs, NB = 5, 2, 128, 8, 4
    rows = rng.standard_normal((T, H, D)).astype(np.float16).view(np.uint16)
    kc = np.zeros((NB, H, bs, D), np.int8)
    vc = np.zeros_like(kc)
    ks = np.zeros((NB, H, bs), np.uint16)
    vs = np.zeros_like(ks)
    slots = np.array([0, 9, 31, 17, -1], np.int32)
    O.append_q8(rows, rows, O.F16, slots, bs, kc, vc, ks, vs)
    for t in range(4):
        s = slots[t]
        for h in range(H):
            x = rows[t, h].view(np.float16).astype(np.float32)
            codes, sb = O.quantize_row_q8(x)
            assert np.array_equal(kc[s // bs, h, s % bs], codes)
            assert ks[s // bs, h, s % bs] == sb
    assert not kc[1, :, 6].any() and ks[1, 0, 6] == 0


# ---------------------------------------------------------------- attention
def _brute_attention(q, kc, vc, table_row, L, h, bs, scale):
    """Written separately: walk the table, score, exponentiate, normalise."""
    keys, vals = [], []
    for blk in table_row:
        for off in range(bs):
            if len(keys) == L:
                break
            keys.append([float(v) for v in kc[blk, h, off]])
            vals.append([float(v) for v in vc[blk, h, off]])
    if L == 0:
        return [0.0] * len(q)
    scores = [scale * sum(a * b for a, b in zip(q, k)) for k in keys]
    top = max(scores)
    w = [math.exp(s - top) for s in scores]
    z = sum(w)
    return [sum(w[t] * vals[t][i] for t in range(L)) / z for i in range(len(q))]


def _tiny_case(rng, NB=10, Hkv=2, G=2, D=8, bs=4, lens=(5, 1, 8, 0)):
    B = len(lens)
    Hq = Hkv * G
    kc = rng.standard_normal((NB, Hkv, bs, D)).astype(np.float32)
    vc = rng.standard_normal((NB, Hkv, bs, D)).astype(np.float32)
    maxb = max(1, max(-(-L // bs) for L in lens))
    perm = rng.permutation(NB).astype(np.int32)
    tables = np.zeros((B, maxb), np.int32)
    c = 0
    for b, L in enumerate(lens):
        n = -(-L // bs)
        tables[b, :n] = perm[c:c + n]
        c += n
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    return kc, vc, tables, np.array(lens, np.int32), q


def test_attention_matches_brute_force_on_tiny_shapes():
    rng = np.random.default_rng(21)
    for G in (1, 2, 4):
        kc, vc, tables, lens, q = _tiny_case(rng, G=G)
        scale = 1 / math.sqrt(8)
        out = O.paged_decode_attention(q, O.F32, kc, vc, O.F32, tables, lens, scale)
        Hkv = kc.shape[1]
        for b in range(len(lens)):
            for h in range(Hkv * G):
                want = _brute_attention([float(v) for v in q[b, h]], kc, vc, tables[b],
                                        int(lens[b]), h // G, 4, scale)
                assert np.max(np.abs(out[b, h] - want)) <= 1e-12


def test_single_token_returns_its_value_exactly():
    rng = np.random.default_rng(2)
    kc, vc, tables, lens, q = _tiny_case(rng, lens=(1, 1))
    out = O.paged_decode_attention(q, O.F32, kc, vc, O.F32, tables, lens, 0.3)
    for b in range(2):
        for h in range(4):
            assert np.array_equal(out[b, h], vc[tables[b, 0], h // 2, 0].astype(np.float64))


def test_equal_keys_give_the_mean_of_values():
    rng = np.random.default_rng(4)
    kc, vc, tables, lens, q = _tiny_case(rng, lens=(7, 3))
    kc[:] = kc[0, 0, 0]                          # every key the same
    out = O.paged_decode_attention(q, O.F32, kc, vc, O.F32, tables, lens, 0.5)
    for b, L in enumerate(lens):
        for h in range(4):
            rows = O.gather(vc, None, O.F32, tables[b], int(L), h // 2, 4)
            assert np.max(np.abs(out[b, h] - rows.mean(axis=0))) <= 1e-14


def test_gqa_equals_mha_with_repeated_kv_heads():
    rng = np.random.default_rng(6)
    G = 4
    kc, vc, tables, lens, q = _tiny_case(rng, Hkv=2, G=G)
    gqa = O.paged_decode_attention(q, O.F32, kc, vc, O.F32, tables, lens, 0.35)
    kr = np.ascontiguousarray(np.repeat(kc, G, axis=1))
    vr = np.ascontiguousarray(np.repeat(vc, G, axis=1))
    mha = O.paged_decode_attention(q, O.F32, kr, vr, O.F32, tables, lens, 0.35)
    assert np.array_equal(gqa, mha)


def test_paged_equals_contiguous_and_any_block_placement():
    rng = np.random.default_rng(8)
    B, Hkv, D, bs, L = 3, 2, 16, 4, 11
    nb = -(-L // bs)
    rows_k = rng.standard_normal((B, L, Hkv, D)).astype(np.float32)
    rows_v = rng.standard_normal((B, L, Hkv, D)).astype(np.float32)
    q = rng.standard_normal((B, Hkv, D)).astype(np.float32)
    lens = np.full(B, L, np.int32)
    outs = []
    for placement in ("identity", "shuffled", "reversed"):
        NB = B * nb + 5
        if placement == "identity":
            ids = np.arange(B * nb)
        elif placement == "shuffled":
            ids = rng.permutation(NB)[:B * nb]
        else:
            ids = np.arange(NB)[::-1][:B * nb]
        tables = ids.reshape(B, nb).astype(np.int32)
        kc = np.zeros((NB, Hkv, bs, D), np.float32)
        vc = np.zeros_like(kc)
        slots = O.slot_mapping(tables, bs, np.zeros(B, np.int32), lens)
        O.append(rows_k.reshape(B * L, Hkv, D), rows_v.reshape(B * L, Hkv, D), O.F32, slots, bs,
                 kc, vc)
        outs.append(O.paged_decode_attention(q, O.F32, kc, vc, O.F32, tables, lens, 0.25))
    # contiguous: attend directly over the rows, no cache at all
    cont = np.zeros_like(outs[0])
    for b in range(B):
        for h in range(Hkv):
            cont[b, h] = O.attend_rows(q[b, h].astype(np.float64), rows_k[b, :, h], rows_v[b, :, h],
                                       0.25)
    for o in outs:
        assert np.array_equal(o, outs[0])
        assert np.array_equal(o, cont)


def test_shared_prefix_blocks_equal_private_copies():
    rng = np.random.default_rng(10)
    NB, Hkv, bs, D = 16, 1, 4, 8
    kc = rng.standard_normal((NB, Hkv, bs, D)).astype(np.float32)
    vc = rng.standard_normal((NB, Hkv, bs, D)).astype(np.float32)
    # both sequences point at blocks 3, 7 for their first 8 tokens
    shared = np.array([[3, 7, 1], [3, 7, 2]], np.int32)
    # private copies of blocks 3, 7 into 10, 11 and 12, 13
    kp, vp = kc.copy(), vc.copy()
    for src, dst in ((3, 10), (7, 11), (3, 12), (7, 13)):
        kp[dst], vp[dst] = kc[src], vc[src]
    private = np.array([[10, 11, 1], [12, 13, 2]], np.int32)
    lens = np.array([10, 12], np.int32)
    q = rng.standard_normal((2, 1, D)).astype(np.float32)
    a = O.paged_decode_attention(q, O.F32, kc, vc, O.F32, shared, lens, 0.5)
    b = O.paged_decode_attention(q, O.F32, kp, vp, O.F32, private, lens, 0.5)
    assert np.array_equal(a, b)


def test_attention_is_invariant_to_the_order_of_cached_tokens():
    rng = np.random.default_rng(12)
    L, D = 37, 16
    k = rng.standard_normal((L, D))
    v = rng.standard_normal((L, D))
    q = rng.standard_normal(D)
    a = O.attend_rows(q, k, v, 0.25)
    p = rng.permutation(L)
    b = O.attend_rows(q, k[p], v[p], 0.25)
    assert np.max(np.abs(a - b)) <= 1e-14


def test_two_token_closed_form():
    # softmax of two scores is the logistic function of their difference.
    k = np.array([[1.0, 0.0], [0.0, 2.0]])
    v = np.array([[3.0, -1.0], [5.0, 7.0]])
    q = np.array([0.7, -0.4])
    s0, s1 = 0.5 * 0.7, 0.5 * (-0.8)
    w1 = 1.0 / (1.0 + math.exp(s0 - s1))
    want = (1 - w1) * v[0] + w1 * v[1]
    assert np.max(np.abs(O.attend_rows(q, k, v, 0.5) - want)) <= 1e-15


def test_oracle_rejects_out_of_range_tables_and_lengths():
    rng = np.random.default_rng(13)
    kc, vc, tables, lens, q = _tiny_case(rng, lens=(5, 3))
    bad = tables.copy()
    bad[0, 1] = 99
    with pytest.raises(ValueError):
        O.paged_decode_attention(q, O.F32, kc, vc, O.F32, bad, lens, 0.5)
    with pytest.raises(ValueError):
        O.paged_decode_attention(q, O.F32, kc, vc, O.F32, tables, np.array([5, 99], np.int32), 0.5)


def test_int8_attention_is_attention_over_dequantized_rows():
    rng = np.random.default_rng(14)
    NB, H, bs, D = 6, 2, 8, 128
    kc = rng.integers(-127, 128, size=(NB, H, bs, D)).astype(np.int8)
    vc = rng.integers(-127, 128, size=(NB, H, bs, D)).astype(np.int8)
    ks = rng.standard_normal((NB, H, bs)).astype(np.float16).view(np.uint16)
    vs = rng.standard_normal((NB, H, bs)).astype(np.float16).view(np.uint16)
    tables = np.array([[4, 1], [0, 5]], np.int32)
    lens = np.array([13, 9], np.int32)
    q = rng.standard_normal((2, 4, D)).astype(np.float16).view(np.uint16)
    out = O.paged_decode_attention(q, O.F16, kc, vc, O.I8, tables, lens, 0.1, ks, vs)
    kd = kc.astype(np.float64) * ks.view(np.float16).astype(np.float64)[..., None]
    vd = vc.astype(np.float64) * vs.view(np.float16).astype(np.float64)[..., None]
    qd = q.view(np.float16).astype(np.float64)
    for b in range(2):
        for h in range(4):
            want = _brute_attention(list(qd[b, h]), kd, vd, tables[b], int(lens[b]), h // 2, bs, 0.1)
            assert np.max(np.abs(out[b, h] - want)) <= 1e-12


# ---------------------------------------------------------------- pages' figures
def test_toy_loop_row_counts_and_cache_changes_nothing():
    g = _golden("kv_rows_table.json")
    rng = np.random.default_rng(15)
    E, D = 12, 8
    n = g["prompt_tokens"] + g["decode_steps"]
    x = rng.standard_normal((n, E))
    Wq, Wk, Wv = (rng.standard_normal((D, E)) for _ in range(3))
    on, oc, rn, rc = O.toy_generation(x, g["prompt_tokens"], g["decode_steps"], Wq, Wk, Wv, 4)
    assert rn.tolist() == g["rows_without_cache"]
    assert rc.tolist() == g["rows_with_cache"]
    assert int(rn.sum()) == g["total_without_cache"] and int(rc.sum()) == g["total_with_cache"]
    assert np.array_equal(on, oc)            # caching saves work; the outputs stay identical


def _size(text):
    num, unit = text.split()
    mult = {"KiB": 2 ** 10, "MiB": 2 ** 20, "GiB": 2 ** 30}[unit]
    return float(num) * mult


def test_bytes_per_token_table():
    g = _golden("memory_table.json")
    for m in g["models"]:
        per_tok = O.kv_bytes_per_token(m["layers"], m["kv_heads"], m["head_dim"],
                                       g["bytes_per_number"])
        assert per_tok == _size(m["per_token"])
        total = per_tok * g["tokens"]
        printed = _size(m["per_4096"])
        if m["name"] == "Llama-2-70B":
            # exact 1,342,177,280 B = 1.25 GiB; the page prints it rounded as "1.3 GiB"
            assert total == 1342177280
            assert abs(total / 2 ** 30 - printed / 2 ** 30) <= 0.05 + 1e-12
        else:
            assert total == printed


def test_batch_gqa_and_guide_examples():
    g = _golden("memory_table.json")
    be = g["batch_example"]
    m7 = [m for m in g["models"] if m["name"] == be["model"]][0]
    cache = be["requests"] * be["tokens"] * O.kv_bytes_per_token(m7["layers"], m7["kv_heads"],
                                                                  m7["head_dim"], 2)
    assert cache == _size(be["cache"])
    assert cache > be["weights_gb_about"] * 1e9
    ge = g["gqa_example"]
    m3 = [m for m in g["models"] if m["name"] == ge["model"]][0]
    mha = O.kv_bytes_per_token(m3["layers"], ge["q_heads"], m3["head_dim"], 2)
    gqa = O.kv_bytes_per_token(m3["layers"], ge["kv_heads"], m3["head_dim"], 2)
    assert mha == ge["saving"] * gqa
    gu = g["guide_example"]
    one = gu["tokens"] * O.kv_bytes_per_token(gu["layers"], gu["kv_heads"], gu["head_dim"], 2)
    assert one == 512 * 2 ** 20 and abs(one / 1e9 - gu["about_gb"]) < 0.05
