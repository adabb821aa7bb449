"""Sliding-window decode attention: oracle pins (CPU) and GPU parity.

A variant [VIS] "What the page leaves out" names: each sequence attends over
its last `window` cached rows only.  The plain reading, taken here, is the
softmax of [NOTES] "Concept" over those rows.
"""
import math

import numpy as np
import pytest

from oracle import oracle as O


def _brute_window(q, rows_k, rows_v, window, scale):
    """Written separately: keep the last `window` rows, score, normalise."""
    L = len(rows_k)
    keep = range(max(0, L - window) if window > 0 else 0, L)
    scores = [scale * sum(a * b for a, b in zip(q, rows_k[t])) for t in keep]
    top = max(scores)
    w = [math.exp(s - top) for s in scores]
    z = sum(w)
    return [sum(wi * rows_v[t][i] for wi, t in zip(w, keep)) / z for i in range(len(q))]


def _paged_case(rng, lens, bs=4, H=2, D=8, G=2):
    B = len(lens)
    maxb = max(-(-L // bs) for L in lens)
    NB = B * maxb + 3
    perm = rng.permutation(NB).astype(np.int32)
    tables = perm[:B * maxb].reshape(B, maxb).copy()
    kc = rng.standard_normal((NB, H, bs, D)).astype(np.float32)
    vc = rng.standard_normal((NB, H, bs, D)).astype(np.float32)
    q = rng.standard_normal((B, H * G, D)).astype(np.float32)
    return q, kc, vc, tables, np.array(lens, np.int32)


def _rows(kc, table_row, L, h, bs):
    return [[float(x) for x in kc[table_row[p // bs], h, p % bs]] for p in range(L)]


@pytest.mark.parametrize("window", [1, 3, 5, 8, 13])
def test_window_matches_brute_force_over_the_last_rows(window):
    rng = np.random.default_rng(40 + window)
    bs, G = 4, 2
    q, kc, vc, tables, lens = _paged_case(rng, [11, 4, 1, 9], bs=bs, G=G)
    out = O.paged_decode_attention(q, O.F32, kc, vc, O.F32, tables, lens, 0.35, window=window)
    for b, L in enumerate(lens):
        for h in range(q.shape[1]):
            ref = _brute_window([float(x) for x in q[b, h]], _rows(kc, tables[b], L, h // G, bs),
                                _rows(vc, tables[b], L, h // G, bs), window, 0.35)
            assert np.max(np.abs(out[b, h] - ref)) <= 1e-12


def test_window_covering_every_row_is_full_attention_bit_for_bit():
    rng = np.random.default_rng(50)
    q, kc, vc, tables, lens = _paged_case(rng, [11, 4, 7])
    full = O.paged_decode_attention(q, O.F32, kc, vc, O.F32, tables, lens, 0.3)
    for window in (0, 11, 12, 1000):
        got = O.paged_decode_attention(q, O.F32, kc, vc, O.F32, tables, lens, 0.3, window=window)
        assert np.array_equal(got, full)


def test_window_of_one_returns_the_last_value_exactly():
    rng = np.random.default_rng(51)
    bs = 4
    q, kc, vc, tables, lens = _paged_case(rng, [10, 3, 1], bs=bs, G=1)
    out = O.paged_decode_attention(q, O.F32, kc, vc, O.F32, tables, lens, 0.5, window=1)
    for b, L in enumerate(lens):
        last = vc[tables[b, (L - 1) // bs], :, (L - 1) % bs]
        assert np.array_equal(out[b], last.astype(np.float64))


def test_window_ignores_table_entries_before_it():
    rng = np.random.default_rng(52)
    bs = 4
    q, kc, vc, tables, lens = _paged_case(rng, [17, 9], bs=bs)
    want = O.paged_decode_attention(q, O.F32, kc, vc, O.F32, tables, lens, 0.3, window=6)
    t2 = tables.copy()
    for b, L in enumerate(lens):
        t2[b, :(L - 6) // bs] = -1                    # blocks a caller already freed
    got = O.paged_decode_attention(q, O.F32, kc, vc, O.F32, t2, lens, 0.3, window=6)
    assert np.array_equal(got, want)
    with pytest.raises(ValueError):                   # the full attention still needs them
        O.paged_decode_attention(q, O.F32, kc, vc, O.F32, t2, lens, 0.3)


# ------------------------------------------------------------------ GPU parity
gpu = pytest.mark.gpu


def _window_run(name, window, steps=1, free_before=False):
    import torch
    from paged_kv_cache_273_gb300 import pkv, workloads as W
    import parity_harness as PH
    inp = W.make_inputs(name)
    case = PH.build(inp)
    for s in range(steps):
        PH.append_step(case, s)
    s = steps - 1
    wl = case.wl
    lens = inp.lens_after_step(s)
    tables = inp.block_tables.copy()
    if free_before:
        for b, L in enumerate(lens):
            lo = max(0, int(L) - window)
            tables[b, :lo // wl.block_size] = -1
    dev = torch.device("cuda", 0)
    q = PH.to_device(inp.step_q[s], wl.q_dtype)
    out = torch.empty((wl.batch, wl.num_q_heads, wl.head_dim), dtype=torch.float32, device=dev)
    scale = 1.0 / np.sqrt(wl.head_dim)
    pkv.paged_decode_attention_window(
        case.pool, q, case.gk.tensor, case.gv.tensor, torch.from_numpy(tables).to(dev),
        torch.from_numpy(lens).to(dev), scale, out, case.workspace, int(lens.max()), window,
        None if case.gks is None else case.gks.tensor,
        None if case.gvs is None else case.gvs.tensor)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    want = O.paged_decode_attention(inp.step_q[s], wl.q_dtype, case.ok, case.ov, wl.kv_dtype,
                                    tables, lens, float(np.float32(scale)), case.oks, case.ovs,
                                    window=window)
    err = float(np.max(np.abs(got - want))) if got.size else 0.0
    return err, PH.TOL[wl.kv_dtype], pkv.pkv_check_error(case.pool), PH.counters_zero(case), \
        case, got


@gpu
@pytest.mark.parametrize("name,window", [("tiny", 3), ("tiny", 5), ("gpt2", 100),
                                         ("gpt2", 16), ("llama3_8b", 1000),
                                         ("llama2_70b", 4096), ("int8", 513), ("int4", 700),
                                         ("gpt2", 40)])
def test_gpu_window_matches_oracle(name, window):
    from paged_kv_cache_273_gb300 import pkv
    err, tol, status, zero, _, _ = _window_run(name, window)
    assert err <= tol, err
    assert status == pkv.PKV_OK
    assert zero


@gpu
def test_gpu_window_does_not_read_blocks_before_it():
    from paged_kv_cache_273_gb300 import pkv
    err, tol, status, zero, _, _ = _window_run("gpt2", 200, free_before=True)
    assert err <= tol, err
    assert status == pkv.PKV_OK          # no -1 entry was looked up
    assert zero


@gpu
def test_gpu_window_covering_everything_equals_full_attention():
    import torch
    from paged_kv_cache_273_gb300 import pkv
    import parity_harness as PH
    _, _, _, _, case, got = _window_run("gpt2", 1 << 20)
    full = PH.attend_gpu(case, 0)
    assert np.array_equal(got, full)
    assert pkv.pkv_check_error(case.pool) == pkv.PKV_OK
