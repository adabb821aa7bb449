"""paged_decode_step: one decode step with its inputs and result in host
memory (one host-to-device copy of a staging buffer, kv_append, decode
attention, one device-to-host copy of the output).

GPU: the step call against the same steps made by separate calls (the same
kernels on the same inputs: outputs bit-identical, caches bit-identical to
the oracle's) and against the fp64 oracle.  CPU: argument validation (every
case fails before any device work, so it runs without a GPU)."""
import ctypes

import numpy as np
import pytest

from paged_kv_cache_273_gb300 import pkv
from paged_kv_cache_273_gb300 import workloads as W


def _al(x):
    return (x + 255) // 256 * 256


def _layout(B, Hq, Hkv, D, in_bytes, q_bytes):
    kv = B * Hkv * D * in_bytes
    qb = B * Hq * D * q_bytes
    k, v = 0, _al(kv)
    q = 2 * _al(kv)
    slots = q + _al(qb)
    lens = slots + _al(B * 4)
    return pkv.StepLayout(k, v, q, slots, lens), lens + _al(B * 4)


def test_step_validation_without_device_work():
    lib = pkv.load()
    p = pkv.kv_block_pool_init(8, 16, 2, 64, pkv.PKV_F16)
    B, Hq = 2, 4
    good, total = _layout(B, Hq, 2, 64, 2, 2)
    buf = (ctypes.c_uint8 * (total + 64))()
    base = (ctypes.addressof(buf) + 15) // 16 * 16
    ptr = ctypes.c_void_p(base)

    def call(layout, in_dtype=pkv.PKV_F16, q_dtype=pkv.PKV_F16, hq=Hq, in_bytes=total,
             batch=B, ws=1 << 20):
        return lib.paged_decode_step(p.handle, ptr, ptr, in_bytes,
                                     None if layout is None else ctypes.byref(layout), in_dtype,
                                     q_dtype, hq, ptr, ptr, None, None, ptr, 4, batch, 64, 0.125,
                                     ptr, ptr, ptr, ws, None)

    def shifted(**kw):
        lay = pkv.StepLayout(good.k_new, good.v_new, good.q, good.slot_mapping, good.seq_lens)
        for k, v in kw.items():
            setattr(lay, k, v)
        return lay

    bad = [
        (None, {}),                                        # no layout
        (shifted(k_new=8), {}),                            # k_new off 16 bytes
        (shifted(q=good.q + 4), {}),                       # q off 16 bytes
        (shifted(seq_lens=good.seq_lens + 2), {}),         # lengths off 4 bytes
        (shifted(v_new=total - 16), {}),                   # v_new past the end
        (shifted(slot_mapping=total), {}),                 # slots past the end
        (shifted(seq_lens=1 << 62), {}),                   # offset overflow
        (good, {"in_bytes": good.seq_lens + 4}),           # lengths cut off
        (good, {"in_dtype": pkv.PKV_I8}),                  # not an input type
        (good, {"q_dtype": pkv.PKV_I4}),
        (good, {"hq": 3}),                                 # not a multiple of Hkv
        (good, {"batch": -1}),
        (good, {"q_dtype": pkv.PKV_BF16}),                 # the attention's check: q type
        (good, {"ws": 16}),                                # ... and its workspace size
    ]
    for lay, kw in bad:
        assert call(lay, **kw) == pkv.PKV_ERR_INVALID, (lay, kw)
    assert call(good, batch=0) == pkv.PKV_OK              # an empty batch is a no-op


@pytest.mark.gpu
@pytest.mark.parametrize("name,steps,pinned,lengths", [
    ("llama3_8b", 3, True, None), ("int8", 1, True, None), ("gpt2", 1, True, None),
    ("llama3_8b", 2, False, None),
    ("gpt2", 1, True, (0, 1, 17, 0, 300, 2048, 5, 16)),     # idle sequences: slot -1
])
def test_step_matches_separate_calls_and_oracle(name, steps, pinned, lengths):
    # pinned host buffers are copied by kernels through their device mapping
    # (over fp caches the input copy and the append are one kernel),
    # pageable ones by cudaMemcpyAsync
    import torch
    import parity_harness as PH
    inp = W.make_inputs(name, lengths=lengths)
    wl = inp.workload
    B, Hq, Hkv, D = wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    ref = PH.build(inp)      # separate kv_append / paged_decode_attention calls
    case = PH.build(inp)     # paged_decode_step
    eb = {W.F32: 4, W.F16: 2, W.BF16: 2}
    layout, total = _layout(B, Hq, Hkv, D, eb[wl.src_dtype], eb[wl.q_dtype])
    host_in = torch.empty(total, dtype=torch.uint8)
    host_out = torch.empty((B, Hq, D), dtype=torch.float32)
    if pinned:
        host_in, host_out = host_in.pin_memory(), host_out.pin_memory()
    dev_in = torch.empty(total, dtype=torch.uint8, device="cuda")
    out = torch.empty((B, Hq, D), dtype=torch.float32, device="cuda")
    step = pkv.DecodeStep(case.pool, dev_in, layout, PH._TORCH[wl.src_dtype],
                          PH._TORCH[wl.q_dtype], Hq, case.gk.tensor, case.gv.tensor,
                          case.tables_d, B, int(inp.final_lens.max()), 1.0 / np.sqrt(D), out,
                          case.workspace, None if case.gks is None else case.gks.tensor,
                          None if case.gvs is None else case.gvs.tensor)
    hn = host_in.numpy()

    def put(off, raw, code):
        t = PH.to_device(raw, code, device="cpu").contiguous().view(torch.uint8).numpy()
        hn[off:off + t.size] = t.reshape(-1)

    for s in range(steps):
        PH.append_step(ref, s)
        want = PH.attend_gpu(ref, s)
        slots = PH.step_slots(case, s)
        lens = inp.lens_after_step(s).astype(np.int32)
        put(layout.k_new, inp.step_k[s], wl.src_dtype)
        put(layout.v_new, inp.step_v[s], wl.src_dtype)
        put(layout.q, inp.step_q[s], wl.q_dtype)
        hn[layout.slot_mapping:layout.slot_mapping + 4 * B] = slots.view(np.uint8)
        hn[layout.seq_lens:layout.seq_lens + 4 * B] = lens.view(np.uint8)
        host_out.fill_(float("nan"))
        step(host_in, host_out)
        torch.cuda.synchronize()
        PH._append_oracle(case, inp.step_k[s], inp.step_v[s], slots)
        got = host_out.numpy().copy()
        # the same kernels on the same inputs: bit-identical to the separate calls
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), s
        assert np.max(np.abs(got - PH.attend_oracle(case, s))) <= PH.TOL[wl.kv_dtype]
    assert PH.caches_equal(case)
    assert PH.caches_equal(ref)
    assert pkv.pkv_check_error(case.pool) == pkv.PKV_OK
    assert case.guards_intact()
    assert PH.counters_zero(case)
