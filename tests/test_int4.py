"""4-bit KV cache: oracle pins (CPU) and GPU parity.

[NOTES] "Quantized KV cache" stores the cache in fewer bits; [VIS] "What the
page leaves out" names 8-bit and 4-bit caches without fixing a scheme.  The
reading here is the int8 scheme with the 4-bit range: one fp16 scale per
(token, KV head) row, s = fp16_rne(amax / 7), codes round-half-even of x / s
clamped to +-7, two per byte (element 2j in the low nibble of byte j).
"""
import numpy as np
import pytest

from oracle import oracle as O


def _f16(bits):
    return float(O.decode(np.array([bits], np.uint16), O.F16)[0])


def test_q4_unit_scale_rounds_half_to_even():
    # amax 7 gives the scale 1.0 exactly
    x = np.array([0.5, 1.5, 2.5, -2.5, 3.5, -0.5, 7.0, 0.0], np.float32)
    codes, s = O.quantize_row_q4(x)
    assert s == 0x3C00
    assert list(codes) == [0, 2, 2, -2, 4, 0, 7, 0]


def test_q4_divides_by_the_fp16_rounded_scale():
    # amax 1: 1/7 rounds to the fp16 0x3092 = 0.142822265625.  3.5 * that is
    # an exact tie (-> 4); divided by the unrounded 1/7 it would give 3.
    s16 = 0x3092
    s = _f16(s16)
    assert s == 0.142822265625
    x = np.array([1.0, 3.5 * s, -3.5 * s, 2.5 * s], np.float32)
    codes, sb = O.quantize_row_q4(x)
    assert sb == s16
    assert list(codes) == [7, 4, -4, 2]


def test_q4_zero_row_and_clamp():
    codes, s = O.quantize_row_q4(np.zeros(16, np.float32))
    assert s == 0 and not codes.any()
    # the rounded scale can fall below amax / 7: the largest code clamps at 7
    x = np.array([100.0, -100.0, 50.0, 1e-3], np.float32)
    codes, sb = O.quantize_row_q4(x)
    s = _f16(sb)
    assert list(codes[:2]) == [7, -7]
    assert abs(100.0 - 7 * s) <= 7 * s * 2.0 ** -11 + 1e-12


def test_q4_error_bound_and_symmetry():
    rng = np.random.default_rng(60)
    for _ in range(50):
        x = (rng.standard_normal(128) * rng.uniform(0.01, 100)).astype(np.float32)
        codes, sb = O.quantize_row_q4(x)
        s = _f16(sb)
        assert np.all(np.abs(codes) <= 7)
        err = np.abs(x.astype(np.float64) - codes * s)
        assert np.all(err <= s / 2 + 7 * s * 2.0 ** -11 + 1e-12)
        neg, sn = O.quantize_row_q4(-x)
        assert sn == sb and np.array_equal(neg, -codes)


def test_q4_packing_low_nibble_first():
    assert list(O.pack_q4(np.array([1, -1, 7, -7, 0, -8 + 1, 3, 2], np.int8))) == \
        [0xF1, 0x97, 0x90, 0x23]


def test_q4_append_and_gather_round_trip():
    rng = np.random.default_rng(61)
    NB, H, bs, D = 6, 2, 8, 128
    kc = np.zeros((NB, H, bs, D // 2), np.uint8)
    vc = np.zeros_like(kc)
    ks = np.zeros((NB, H, bs), np.uint16)
    vs = np.zeros_like(ks)
    rows_k = rng.standard_normal((5, H, D)).astype(np.float32)
    rows_v = rng.standard_normal((5, H, D)).astype(np.float32)
    slots = np.array([3, 17, -1, 40, 9], np.int32)
    O.append_q4(rows_k, rows_v, O.F32, slots, bs, kc, vc, ks, vs)
    for t, slot in enumerate(slots):
        if slot < 0:
            continue
        blk, off = divmod(int(slot), bs)
        for h in range(H):
            codes, sb = O.quantize_row_q4(rows_k[t, h])
            assert ks[blk, h, off] == sb
            assert np.array_equal(kc[blk, h, off], O.pack_q4(codes))
            got = O.gather(kc, ks, O.I4, np.array([blk], np.int32), off + 1, h, bs)[off]
            assert np.array_equal(got, codes.astype(np.float64) * _f16(sb))
    assert not ks[2, :, 0].any()          # the padding token wrote nothing


def test_q4_attention_is_attention_over_dequantized_rows():
    rng = np.random.default_rng(62)
    NB, H, bs, D, G, L = 8, 2, 8, 128, 2, 29
    kc = np.zeros((NB, H, bs, D // 2), np.uint8)
    vc = np.zeros_like(kc)
    ks = np.zeros((NB, H, bs), np.uint16)
    vs = np.zeros_like(ks)
    rk = rng.standard_normal((L, H, D)).astype(np.float32)
    rv = rng.standard_normal((L, H, D)).astype(np.float32)
    table = rng.permutation(NB)[:4].astype(np.int32)
    slots = np.array([table[p // bs] * bs + p % bs for p in range(L)], np.int32)
    O.append_q4(rk, rv, O.F32, slots, bs, kc, vc, ks, vs)
    q = rng.standard_normal((1, H * G, D)).astype(np.float16).view(np.uint16)
    out = O.paged_decode_attention(q, O.F16, kc, vc, O.I4, table[None, :], np.array([L]), 0.09,
                                   ks, vs)
    for h in range(H * G):
        dk = np.stack([O.quantize_row_q4(rk[t, h // G])[0] *
                       _f16(O.quantize_row_q4(rk[t, h // G])[1]) for t in range(L)])
        dv = np.stack([O.quantize_row_q4(rv[t, h // G])[0] *
                       _f16(O.quantize_row_q4(rv[t, h // G])[1]) for t in range(L)])
        ref = O.attend_rows(O.decode(q[0, h], O.F16), dk, dv, 0.09)
        assert np.array_equal(out[0, h], ref)


# ------------------------------------------------------------------ GPU parity
gpu = pytest.mark.gpu


@gpu
def test_gpu_int4_workload_matches_oracle():
    import parity_harness as PH
    from paged_kv_cache_273_gb300 import pkv, workloads as W
    r = PH.run(W.make_inputs("int4"))
    assert r["cache_equal_history"] and r["cache_equal"]
    assert r["max_err"] <= r["tol"], r
    assert r["error_word"] == pkv.PKV_OK and r["guards"] and r["counters_zero"]


@gpu
@pytest.mark.parametrize("G,bs,src", [(1, 16, "f16"), (2, 8, "bf16"), (4, 32, "f32"),
                                      (8, 16, "f16")])
def test_gpu_int4_grid(G, bs, src):
    import dataclasses
    import parity_harness as PH
    from paged_kv_cache_273_gb300 import pkv, workloads as W
    code = {"f16": W.F16, "bf16": W.BF16, "f32": W.F32}[src]
    wl = dataclasses.replace(W.WORKLOADS["int4"], name="int4_grid", num_q_heads=4 * G,
                             num_kv_heads=4, block_size=bs, batch=9, src_dtype=code,
                             q_dtype=W.BF16 if code == W.BF16 else W.F16, len_lo=1,
                             len_hi=700, decode_steps=2)
    r = PH.run(W.make_inputs(wl))
    assert r["cache_equal_history"] and r["cache_equal"]
    assert r["max_err"] <= r["tol"], r
    assert r["error_word"] == pkv.PKV_OK and r["guards"] and r["counters_zero"]
