"""Prefill attention over the paged cache: oracle pins (CPU) and GPU parity.

[VIS] "Prefill and decode feel different": the prompt is processed as one
batch of tokens, not one token per step.  Each new token attends causally over the cached rows up to its own
position, with the softmax of [NOTES] "Concept"; the new tokens' K and V are
already in the cache (kv_append with T > 1).
"""
import math

import numpy as np
import pytest

from oracle import oracle as O


def _case(rng, news, cached, H=2, G=2, D=16, bs=4, dtype=np.float32):
    """Caches holding each sequence's rows; q for its last `news[b]` tokens."""
    B = len(news)
    lens = [c + n for c, n in zip(cached, news)]
    maxb = max(1, max(-(-L // bs) for L in lens))
    NB = B * maxb + 2
    perm = rng.permutation(NB).astype(np.int32)
    tables = perm[:B * maxb].reshape(B, maxb).copy()
    kc = rng.standard_normal((NB, H, bs, D)).astype(dtype)
    vc = rng.standard_normal((NB, H, bs, D)).astype(dtype)
    qs = np.zeros(B + 1, np.int32)
    qs[1:] = np.cumsum(news)
    q = rng.standard_normal((int(qs[-1]), H * G, D)).astype(dtype)
    return q, kc, vc, tables, qs, np.array(lens, np.int32)


def _brute(q, kc, vc, table, L, n, h, G, bs, scale):
    """Written separately: for every new token, walk the table up to its
    position, score, exponentiate, normalise."""
    outs = []
    for i in range(n):
        p = L - n + i
        keys, vals = [], []
        for pos in range(p + 1):
            blk, off = table[pos // bs], pos % bs
            keys.append([float(x) for x in kc[blk, h // G, off]])
            vals.append([float(x) for x in vc[blk, h // G, off]])
        qq = [float(x) for x in q[i, h]]
        sc = [scale * sum(a * b for a, b in zip(qq, k)) for k in keys]
        top = max(sc)
        w = [math.exp(s - top) for s in sc]
        z = sum(w)
        outs.append([sum(w[t] * vals[t][d] for t in range(p + 1)) / z for d in range(len(qq))])
    return np.array(outs)


def test_prefill_matches_brute_force():
    rng = np.random.default_rng(70)
    G, bs = 2, 4
    q, kc, vc, tb, qs, lens = _case(rng, news=[5, 1, 7], cached=[0, 6, 3], G=G, bs=bs)
    out = O.paged_prefill_attention(q, O.F32, kc, vc, O.F32, tb, qs, lens, 0.3)
    for b in range(3):
        n = qs[b + 1] - qs[b]
        for h in range(q.shape[1]):
            ref = _brute(q[qs[b]:qs[b + 1]], kc, vc, tb[b], lens[b], n, h, G, bs, 0.3)
            assert np.max(np.abs(out[qs[b]:qs[b + 1], h] - ref)) <= 1e-12


def test_last_new_token_is_the_decode_step():
    rng = np.random.default_rng(71)
    q, kc, vc, tb, qs, lens = _case(rng, news=[9, 4], cached=[3, 12])
    out = O.paged_prefill_attention(q, O.F32, kc, vc, O.F32, tb, qs, lens, 0.25)
    dec = O.paged_decode_attention(q[qs[1:] - 1], O.F32, kc, vc, O.F32, tb, lens, 0.25)
    assert np.array_equal(out[qs[1:] - 1], dec)


def test_first_token_of_a_fresh_prompt_returns_its_value():
    rng = np.random.default_rng(72)
    G, bs = 2, 4
    q, kc, vc, tb, qs, lens = _case(rng, news=[6], cached=[0], G=G, bs=bs)
    out = O.paged_prefill_attention(q, O.F32, kc, vc, O.F32, tb, qs, lens, 0.5)
    for h in range(q.shape[1]):
        assert np.array_equal(out[0, h], vc[tb[0, 0], h // G, 0].astype(np.float64))


def test_prefill_is_causal():
    rng = np.random.default_rng(73)
    bs = 4
    q, kc, vc, tb, qs, lens = _case(rng, news=[10], cached=[2], bs=bs)
    out = O.paged_prefill_attention(q, O.F32, kc, vc, O.F32, tb, qs, lens, 0.3)
    # rows after position 7 (the 6th new token) are rewritten
    kc2, vc2 = kc.copy(), vc.copy()
    for pos in range(8, 12):
        kc2[tb[0, pos // bs], :, pos % bs] += 3.0
        vc2[tb[0, pos // bs], :, pos % bs] -= 2.0
    out2 = O.paged_prefill_attention(q, O.F32, kc2, vc2, O.F32, tb, qs, lens, 0.3)
    assert np.array_equal(out2[:6], out[:6])          # positions 2..7 cannot see them
    assert not np.array_equal(out2[6:], out[6:])


def test_chunked_prefill_equals_prefill_at_once():
    rng = np.random.default_rng(74)
    q, kc, vc, tb, qs, lens = _case(rng, news=[40], cached=[0])
    once = O.paged_prefill_attention(q, O.F32, kc, vc, O.F32, tb, qs, lens, 0.2)
    a = O.paged_prefill_attention(q[:25], O.F32, kc, vc, O.F32, tb, [0, 25], [25], 0.2)
    b = O.paged_prefill_attention(q[25:], O.F32, kc, vc, O.F32, tb, [0, 15], [40], 0.2)
    assert np.array_equal(np.concatenate([a, b]), once)


# ------------------------------------------------------------------ GPU parity
# Tolerance: 2e-3 max-abs for fp16/bf16 K/V with fp32 accumulation, as for
# decode.  From the arithmetic: scores are exact products summed in fp32; the
# weights p enter P.V as a high and a low part of the input type (p = hi + lo
# up to the rounding of lo, ~2^-16 relative for bf16, ~2^-22 for fp16), so the
# error left is fp32 accumulation and the exp2 approximation (~2^-22 relative),
# orders of magnitude inside the bound whatever the score pattern.
PREFILL_TOL = {"f16": 2e-3, "bf16": 2e-3}


def _gpu_prefill_case(dt, D, Hq, Hkv, bs, news, cached, seed, k_growth=0.0, with_vmax=False):
    import torch
    from paged_kv_cache_273_gb300 import pkv
    import parity_harness as PH
    from paged_kv_cache_273_gb300 import workloads as W
    code = {"f16": W.F16, "bf16": W.BF16}[dt]
    rng = np.random.default_rng(seed)
    dev = torch.device("cuda", 0)
    B = len(news)
    lens = np.array([c + n for c, n in zip(cached, news)], np.int32)
    maxb = max(-(-int(L) // bs) for L in lens)
    NB = B * maxb + 5
    tables = rng.permutation(NB)[:B * maxb].astype(np.int32).reshape(B, maxb)
    pool = pkv.kv_block_pool_init(NB, bs, Hkv, D, code)
    gk = PH.Guarded((NB, Hkv, bs, D), PH._TORCH[code])
    gv = PH.Guarded((NB, Hkv, bs, D), PH._TORCH[code])
    ok = np.zeros((NB, Hkv, bs, D), np.uint16)
    ov = np.zeros_like(ok)
    total = int(lens.sum())
    rows_k = W._values(rng, (total, Hkv, D), code)
    rows_v = W._values(rng, (total, Hkv, D), code)
    if k_growth > 0.0:
        # K rows grow with their position in the sequence, so that each new
        # key tile holds larger scores than every earlier one
        pos = np.concatenate([np.arange(int(L)) for L in lens]).astype(np.float32)
        kf = rng.standard_normal((total, Hkv, D), dtype=np.float32) * \
            (1.0 + k_growth * pos)[:, None, None]
        rows_k = (kf.view(np.uint32) >> 16).astype(np.uint16) if code == W.BF16 else \
            kf.astype(np.float16).view(np.uint16)
    slots = pkv.kv_slot_mapping(tables, bs, np.zeros(B, np.int32), lens)
    pkv.kv_append(pool, PH.to_device(rows_k, code), PH.to_device(rows_v, code),
                  torch.from_numpy(slots).to(dev), gk.tensor, gv.tensor)
    O.append(rows_k, rows_v, code, slots, bs, ok, ov)
    qs = np.zeros(B + 1, np.int32)
    qs[1:] = np.cumsum(news)
    q = W._values(rng, (int(qs[-1]), Hq, D), code)
    out = torch.full((int(qs[-1]), Hq, D), float("nan"), dtype=torch.float32, device=dev)
    scale = 1.0 / np.sqrt(D)
    pkv.paged_prefill_attention(pool, PH.to_device(q, code), gk.tensor, gv.tensor,
                                torch.from_numpy(tables).to(dev), torch.from_numpy(qs).to(dev),
                                torch.from_numpy(lens).to(dev), scale, out, max(news))
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    want = O.paged_prefill_attention(q, code, ok, ov, code, tables, qs, lens,
                                     float(np.float32(scale)))
    same_cache = np.array_equal(PH.to_raw(gk.tensor, code), ok) and \
        np.array_equal(PH.to_raw(gv.tensor, code), ov)
    res = (float(np.max(np.abs(got - want))), pkv.pkv_check_error(pool), same_cache,
           gk.intact() and gv.intact())
    if with_vmax:
        res += (float(np.max(np.abs(O.decode(rows_v, code)))),)
    return res


@pytest.mark.gpu
@pytest.mark.parametrize("dt,D,Hq,Hkv,bs,news,cached", [
    ("bf16", 128, 8, 2, 16, [200, 70, 1], [0, 263, 76]),
    ("f16", 64, 4, 4, 4, [64, 33, 130], [0, 10, 5]),
    ("bf16", 128, 32, 8, 16, [1000], [0]),
    ("f16", 128, 16, 2, 32, [129, 5, 64], [0, 300, 64]),
    ("f16", 128, 8, 8, 16, [1], [1]),
    ("bf16", 64, 8, 4, 8, [300, 513, 256], [17, 0, 40]),
    ("bf16", 128, 4, 2, 256, [700, 3], [300, 509]),
    # more work items (256-query tiles x heads) than SMs: each CTA runs
    # several, some of them empty
    ("bf16", 128, 32, 8, 16, [700, 300, 900, 50], [0, 100, 0, 500]),
    ("f16", 64, 32, 4, 8, [513, 1, 260], [10, 0, 3]),
    # d 128 with the smallest blocks (4 rows: 16-byte copies) and 8-row
    # tensor copies
    ("bf16", 128, 8, 4, 4, [150, 20], [30, 7]),
    ("f16", 128, 4, 4, 8, [300], [9]),
])
def test_gpu_prefill_matches_oracle(dt, D, Hq, Hkv, bs, news, cached):
    from paged_kv_cache_273_gb300 import pkv
    err, status, same_cache, intact = _gpu_prefill_case(dt, D, Hq, Hkv, bs, news, cached, 80)
    assert same_cache and intact
    assert status == pkv.PKV_OK
    assert err <= PREFILL_TOL[dt], err


def _random_prefill_shape(seed):
    rng = np.random.default_rng(5000 + seed)
    dt = str(rng.choice(["bf16", "f16"]))
    D = int(rng.choice([64, 128]))
    Hkv = int(rng.choice([1, 2, 4]))
    Hq = Hkv * int(rng.choice([1, 2, 4, 8]))
    bs = int(rng.choice([4, 8, 16, 32, 64, 128, 256]))
    B = int(rng.integers(1, 6))
    edge = [1, 2, 127, 128, 129, 255, 256, 257, 511]
    news = [int(rng.choice(edge)) if rng.random() < 0.4 else int(rng.integers(1, 900))
            for _ in range(B)]
    cached = [0 if rng.random() < 0.4 else int(rng.integers(0, 700)) for _ in range(B)]
    return dt, D, Hq, Hkv, bs, news, cached


@pytest.mark.gpu
@pytest.mark.parametrize("seed", range(24))
def test_gpu_prefill_random_shapes(seed):
    # seeded random types, head sizes, groups, block sizes and prompt /
    # cached-length mixes (tile-boundary lengths among them)
    from paged_kv_cache_273_gb300 import pkv
    dt, D, Hq, Hkv, bs, news, cached = _random_prefill_shape(seed)
    err, status, same_cache, intact = _gpu_prefill_case(dt, D, Hq, Hkv, bs, news, cached,
                                                        600 + seed)
    assert same_cache and intact
    assert status == pkv.PKV_OK
    assert err <= PREFILL_TOL[dt], (err, dt, D, Hq, Hkv, bs, news, cached)


@pytest.mark.gpu
def test_gpu_prefill_full_size_sampled():
    """The timed prefill workload (4 prompts x 4096 new tokens, 32 q / 8 KV
    heads, d 128, bf16, block size 16, one launch as the bench makes it);
    sampled outputs checked one by one: the attention of new token i is the
    decode oracle over the first i + 1 cached rows."""
    import torch
    from paged_kv_cache_273_gb300 import pkv
    import parity_harness as PH
    from paged_kv_cache_273_gb300 import workloads as W
    code, B, n, Hq, Hkv, D, bs = W.BF16, 4, 4096, 32, 8, 128, 16
    rng = np.random.default_rng(90)
    dev = torch.device("cuda", 0)
    nb = n // bs
    NB = B * nb + 3
    tables = rng.permutation(NB)[:B * nb].astype(np.int32).reshape(B, nb)
    pool = pkv.kv_block_pool_init(NB, bs, Hkv, D, code)
    kc = torch.zeros((NB, Hkv, bs, D), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    ok = np.zeros((NB, Hkv, bs, D), np.uint16)
    ov = np.zeros_like(ok)
    lens = np.full(B, n, np.int32)
    rows_k = W._values(rng, (B * n, Hkv, D), code)
    rows_v = W._values(rng, (B * n, Hkv, D), code)
    slots = pkv.kv_slot_mapping(tables, bs, np.zeros(B, np.int32), lens)
    pkv.kv_append(pool, PH.to_device(rows_k, code), PH.to_device(rows_v, code),
                  torch.from_numpy(slots).to(dev), kc, vc)
    O.append(rows_k, rows_v, code, slots, bs, ok, ov)
    qs = np.arange(0, (B + 1) * n, n, dtype=np.int32)
    q = W._values(rng, (B * n, Hq, D), code)
    out = torch.full((B * n, Hq, D), float("nan"), dtype=torch.float32, device=dev)
    scale = 1.0 / np.sqrt(D)
    pkv.paged_prefill_attention(pool, PH.to_device(q, code), kc, vc,
                                torch.from_numpy(tables).to(dev), torch.from_numpy(qs).to(dev),
                                torch.from_numpy(lens).to(dev), scale, out, n)
    torch.cuda.synchronize()
    assert pkv.pkv_check_error(pool) == pkv.PKV_OK
    got = out.cpu().numpy()
    assert not np.isnan(got).any()                  # every output row was written
    assert np.array_equal(PH.to_raw(kc, code), ok) and np.array_equal(PH.to_raw(vc, code), ov)
    picks = [(b, i, h) for b in range(B) for i in (0, 1, 255, 256, 4095)
             for h in (0, 31)] + [tuple(x) for x in
                                  zip(rng.integers(0, B, 40), rng.integers(0, n, 40),
                                      rng.integers(0, Hq, 40))]
    err = 0.0
    for b, i, h in picks:
        qrow = q[qs[b] + i][None, :, :]
        want = O.paged_decode_attention(qrow, code, ok, ov, code, tables[b:b + 1],
                                        np.array([i + 1], np.int32), float(np.float32(scale)))
        err = max(err, float(np.max(np.abs(got[qs[b] + i, h] - want[0, h]))))
    assert err <= PREFILL_TOL["bf16"], err


def _prefill_error_case(bad: str):
    """A small bf16 prefill whose inputs are wrong in one way; returns the
    pool's status and whether the caches' canaries are intact."""
    import torch
    from paged_kv_cache_273_gb300 import pkv
    import parity_harness as PH
    from paged_kv_cache_273_gb300 import workloads as W
    code, D, Hq, Hkv, bs = W.BF16, 128, 8, 2, 16
    rng = np.random.default_rng(91)
    dev = torch.device("cuda", 0)
    news, cached = [300, 40], [20, 0]
    lens = np.array([c + n for c, n in zip(cached, news)], np.int32)
    maxb = max(-(-int(L) // bs) for L in lens)
    NB = 2 * maxb + 2
    tables = rng.permutation(NB)[:2 * maxb].astype(np.int32).reshape(2, maxb)
    pool = pkv.kv_block_pool_init(NB, bs, Hkv, D, code)
    gk = PH.Guarded((NB, Hkv, bs, D), torch.bfloat16)
    gv = PH.Guarded((NB, Hkv, bs, D), torch.bfloat16)
    qs = np.array([0, news[0], news[0] + news[1]], np.int32)
    q = W._values(rng, (int(qs[-1]), Hq, D), code)
    if bad == "block":
        tables[0, 5] = NB + 7                      # an id past the pool, inside the prefix
    elif bad == "length":
        lens[1] = news[1] - 1                      # fewer cached rows than new tokens
    out = torch.full((int(qs[-1]), Hq, D), float("nan"), dtype=torch.float32, device=dev)
    pkv.paged_prefill_attention(pool, PH.to_device(q, code), gk.tensor, gv.tensor,
                                torch.from_numpy(tables).to(dev), torch.from_numpy(qs).to(dev),
                                torch.from_numpy(lens).to(dev), 1.0 / np.sqrt(D), out, max(news))
    torch.cuda.synchronize()
    return pkv.pkv_check_error(pool), gk.intact() and gv.intact(), out


@pytest.mark.gpu
@pytest.mark.parametrize("bad", ["block", "length"])
def test_gpu_prefill_reports_bad_inputs(bad):
    from paged_kv_cache_273_gb300 import pkv
    status, intact, out = _prefill_error_case(bad)
    assert status == pkv.PKV_ERR_BAD_INDEX
    assert intact
    if bad == "length":                            # the other sequence is still computed
        assert not out[:300].isnan().any()


@pytest.mark.gpu
@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_gpu_prefill_rising_scores(dt):
    """Scores that keep rising along the keys move each row's running offset
    inside most tiles (the rare path: P already written in the tile, the sums
    and O are rescaled)."""
    from paged_kv_cache_273_gb300 import pkv
    err, status, same_cache, intact, vmax = _gpu_prefill_case(
        dt, 128, 8, 2, 16, [600, 130], [100, 0], 81, k_growth=1.0 / 32, with_vmax=True)
    assert same_cache and intact
    assert status == pkv.PKV_OK
    # With one or two keys carrying nearly all the weight rounding errors of
    # P would not average out; with P in two parts the weights' error is
    # ~2^-16 of max |v| at worst, inside the same bound as everywhere.
    assert vmax > 0
    assert err <= PREFILL_TOL[dt], (err, vmax)
