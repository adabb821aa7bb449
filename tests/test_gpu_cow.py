"""Copy-on-write on the GPU, through the C ABI, against the oracle.

[VIS] "PagedAttention: the cache in blocks": sequences that begin alike may
reference one physical copy of their first blocks, and a sharer gets a private
copy of a block only when it must modify it.  kv_block_copy must be a bit copy of whole blocks; a fork of one
prompt into several requests, each appending its own tokens with
kv_reserve_slots_cow + kv_block_copy + kv_append, must leave every request
seeing exactly the prompt followed by its own rows, and attention over them
must match the oracle.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from paged_kv_cache_273_gb300 import pkv
from parity_harness import TOL, to_device, to_raw
from paged_kv_cache_273_gb300 import workloads as W

pytestmark = pytest.mark.gpu

_RAW = {W.F32: np.float32, W.F16: np.uint16, W.BF16: np.uint16, W.I8: np.int8}


def _random_raw(rng, shape, code):
    if code == W.F32:
        return rng.standard_normal(shape).astype(np.float32)
    if code == W.I8:
        return rng.integers(-127, 128, shape).astype(np.int8)
    x = rng.standard_normal(shape).astype(np.float32)
    if code == W.F16:
        return x.astype(np.float16).view(np.uint16)
    return (x.view(np.uint32) >> 16).astype(np.uint16)       # bf16 by truncation


@pytest.mark.parametrize("code,bs", [(W.F16, 16), (W.BF16, 4), (W.F32, 16), (W.I8, 16)])
def test_block_copy_is_a_bit_copy_of_whole_blocks(code, bs):
    rng = np.random.default_rng(31)
    NB, H, D = 40, 4, 128
    dev = torch.device("cuda", 0)
    pool = pkv.kv_block_pool_init(NB, bs, H, D, code)
    kc_h = _random_raw(rng, (NB, H, bs, D), code)
    vc_h = _random_raw(rng, (NB, H, bs, D), code)
    ks_h = vs_h = None
    if code == W.I8:
        ks_h = rng.integers(0, 0x7bff, (NB, H, bs)).astype(np.uint16)
        vs_h = rng.integers(0, 0x7bff, (NB, H, bs)).astype(np.uint16)
    kc, vc = to_device(kc_h, code), to_device(vc_h, code)
    ks = None if ks_h is None else to_device(ks_h, W.F16)
    vs = None if vs_h is None else to_device(vs_h, W.F16)
    src = np.array([3, 17, 0, 39, 22], np.int32)
    dst = np.array([5, 1, 38, 12, 30], np.int32)
    pkv.kv_block_copy(pool, torch.from_numpy(src).to(dev), torch.from_numpy(dst).to(dev),
                      kc, vc, ks, vs)
    torch.cuda.synchronize()
    O.block_copy(src, dst, bs, kc_h, vc_h, ks_h, vs_h)
    assert np.array_equal(to_raw(kc, code), kc_h)
    assert np.array_equal(to_raw(vc, code), vc_h)
    if code == W.I8:
        assert np.array_equal(to_raw(ks, W.F16), ks_h)
        assert np.array_equal(to_raw(vs, W.F16), vs_h)
    assert pkv.pkv_check_error(pool) == pkv.PKV_OK


def test_block_copy_skips_bad_ids_and_reports_them():
    rng = np.random.default_rng(32)
    NB, H, bs, D = 8, 2, 16, 64
    dev = torch.device("cuda", 0)
    pool = pkv.kv_block_pool_init(NB, bs, H, D, W.F16)
    kc_h = _random_raw(rng, (NB, H, bs, D), W.F16)
    vc_h = _random_raw(rng, (NB, H, bs, D), W.F16)
    kc, vc = to_device(kc_h, W.F16), to_device(vc_h, W.F16)
    src = np.array([1, 9, -1, 4], np.int32)
    dst = np.array([2, 3, 5, 100], np.int32)
    pkv.kv_block_copy(pool, torch.from_numpy(src).to(dev), torch.from_numpy(dst).to(dev), kc, vc)
    torch.cuda.synchronize()
    O.block_copy(src[:1], dst[:1], bs, kc_h, vc_h)     # only the valid pair
    assert np.array_equal(to_raw(kc, W.F16), kc_h)
    assert np.array_equal(to_raw(vc, W.F16), vc_h)
    assert pkv.pkv_check_error(pool) == pkv.PKV_ERR_BAD_INDEX
    assert pkv.pkv_check_error(pool) == pkv.PKV_OK


def _rows_as_f64(raw, code, scales=None):
    x = O.decode(raw, code) if code != W.I8 else raw.astype(np.float64)
    if scales is not None:
        x = x * O.decode(scales, W.F16)[..., None]
    return x


@pytest.mark.parametrize("code,bs,G", [(W.F16, 16, 4), (W.BF16, 4, 2), (W.I8, 16, 4)])
def test_fork_and_decode_with_copy_on_write(code, bs, G):
    rng = np.random.default_rng(33)
    dev = torch.device("cuda", 0)
    H, D, S, prompt, steps = 2, 128, 5, 21, 24
    Hq = H * G
    src_code = W.F16 if code == W.I8 else code
    q_code = W.F16 if code == W.I8 else code
    NB = 64
    maxb = -(-(prompt + steps) // bs) + 1
    pool = pkv.kv_block_pool_init(NB, bs, H, D, code)
    kc, vc, ks, vs = pool.alloc_cache(dev)
    tables = np.zeros((S, maxb), np.int32)
    # the prompt, written once for request 0
    pk = _random_raw(rng, (prompt, H, D), src_code)
    pv = _random_raw(rng, (prompt, H, D), src_code)
    slots = pkv.kv_reserve_slots(pool, [0], tables[:1], num_new=[prompt])
    pkv.kv_append(pool, to_device(pk, src_code), to_device(pv, src_code),
                  torch.from_numpy(slots).to(dev), kc, vc, ks, vs)
    # fork
    nb = -(-prompt // bs)
    for b in range(1, S):
        tables[b, :nb] = tables[0, :nb]
        pkv.kv_block_share(pool, tables[0, :nb])
    lens = np.full(S, prompt, np.int32)
    own_k = [[] for _ in range(S)]
    own_v = [[] for _ in range(S)]
    ncopies = 0
    scale = 1.0 / np.sqrt(D)
    ws = pkv.alloc_workspace(pool, S, Hq, dev)
    out = torch.empty((S, Hq, D), dtype=torch.float32, device=dev)
    max_err = 0.0
    for step in range(steps):
        slots, src, dst = pkv.kv_reserve_slots_cow(pool, lens, tables)
        ncopies += src.size
        if src.size:
            pkv.kv_block_copy(pool, torch.from_numpy(src).to(dev), torch.from_numpy(dst).to(dev),
                              kc, vc, ks, vs)
        nk = _random_raw(rng, (S, H, D), src_code)
        nv = _random_raw(rng, (S, H, D), src_code)
        pkv.kv_append(pool, to_device(nk, src_code), to_device(nv, src_code),
                      torch.from_numpy(slots).to(dev), kc, vc, ks, vs)
        for b in range(S):
            own_k[b].append(nk[b])
            own_v[b].append(nv[b])
        lens += 1
        if step % 6 == 5 or step == steps - 1:
            q = _random_raw(rng, (S, Hq, D), q_code)
            pkv.paged_decode_attention(pool, to_device(q, q_code), kc, vc,
                                       torch.from_numpy(tables).to(dev),
                                       torch.from_numpy(lens).to(dev), scale, out, ws,
                                       int(lens.max()), ks, vs)
            got = out.cpu().numpy()
            qf = O.decode(q, q_code)
            for b in range(S):
                rk = np.concatenate([pk, np.stack(own_k[b])])
                rv = np.concatenate([pv, np.stack(own_v[b])])
                if code == W.I8:
                    # the rows the cache must hold: the oracle's codes and scales
                    kq = [O.quantize_row_q8(O.decode(r, src_code)) for r in rk.reshape(-1, D)]
                    vq = [O.quantize_row_q8(O.decode(r, src_code)) for r in rv.reshape(-1, D)]
                    kf = np.stack([c.astype(np.float64) * O.decode(np.uint16(s), W.F16)
                                   for c, s in kq]).reshape(-1, H, D)
                    vf = np.stack([c.astype(np.float64) * O.decode(np.uint16(s), W.F16)
                                   for c, s in vq]).reshape(-1, H, D)
                else:
                    kf, vf = _rows_as_f64(rk, code), _rows_as_f64(rv, code)
                for h in range(Hq):
                    ref = O.attend_rows(qf[b, h], kf[:, h // G], vf[:, h // G], scale)
                    max_err = max(max_err, float(np.max(np.abs(got[b, h] - ref))))
    torch.cuda.synchronize()
    assert max_err <= TOL[code], max_err
    # every request sees exactly the prompt followed by its own rows
    kch, vch = to_raw(kc, code), to_raw(vc, code)
    for b in range(S):
        pos = np.arange(lens[b])
        blk = tables[b, pos // bs]
        gk = kch[blk, :, pos % bs]
        gv = vch[blk, :, pos % bs]
        rk = np.concatenate([pk, np.stack(own_k[b])])
        rv = np.concatenate([pv, np.stack(own_v[b])])
        if code == W.I8:
            rk = np.stack([O.quantize_row_q8(O.decode(r, src_code))[0]
                           for r in rk.reshape(-1, D)]).reshape(-1, H, D)
            rv = np.stack([O.quantize_row_q8(O.decode(r, src_code))[0]
                           for r in rv.reshape(-1, D)]).reshape(-1, H, D)
        assert np.array_equal(gk, rk), b
        assert np.array_equal(gv, rv), b
    # the partly filled prompt block was copied for all but one request; the
    # full prompt blocks are still shared by all
    assert ncopies == (S - 1 if prompt % bs else 0)
    for j in range(prompt // bs):
        assert pkv.kv_block_refcount(pool, int(tables[0, j])) == S
    assert pkv.pkv_check_error(pool) == pkv.PKV_OK
