"""Randomized decode parity: seeded random shapes against the fp64 oracle.

Each case draws a cache type (fp32, fp16, bf16, int8, int4), head size, group
size G, KV head count, block size, a batch of lengths mixing empty, one-row,
block- and tile-boundary and long sequences, the query and source types and,
for some, a sliding window; appends one decode step through the C ABI and
compares the attention output element by element with the oracle, the caches
bit by bit, and checks the error word, the canaries and the counters.  This
spans the tile paths (CUDA cores and tensor cores), the work-unit sizes and
gather rows of every block size, and the split over CTAs on mixes the fixed
tests do not pin.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

CASES = 160


def _draw(seed):
    from paged_kv_cache_273_gb300 import workloads as W
    rng = np.random.default_rng(7000 + seed)
    kv = int(rng.choice([W.F32, W.F16, W.BF16, W.I8, W.I4]))
    D = 128 if kv == W.I4 else int(rng.choice([64, 128]))
    G = int(rng.choice([1, 2, 4, 8]))
    Hkv = int(rng.choice([1, 2, 3]))
    quant = kv in (W.I8, W.I4)
    bs = int(rng.choice([8, 16, 32, 64, 128] if quant else [4, 8, 16, 32, 64, 128]))
    B = int(rng.integers(1, 25))
    special = [0, 1, bs - 1, bs, bs + 1, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 129]
    lengths = [int(rng.choice(special)) if rng.random() < 0.5 else int(rng.integers(1, 3001))
               for _ in range(B)]
    lengths = [max(L, 1) if i == 0 else L for i, L in enumerate(lengths)]   # one non-empty
    if quant:
        q = int(rng.choice([W.F16, W.BF16]))
        src = int(rng.choice([W.F16, W.BF16, W.F32]))
    else:
        q = src = kv
    window = 0 if rng.random() < 0.6 else int(rng.integers(1, max(lengths) + 1))
    wl = W.Workload("fuzz%d" % seed, Hkv * G, Hkv, D, bs, B, kv, q, src, 9000 + seed,
                    "uniform", 1, 2, 1)
    return W.make_inputs(wl, lengths=lengths), window


@pytest.mark.parametrize("seed", range(CASES))
def test_gpu_decode_random_shape(seed):
    import torch
    from oracle import oracle as O
    from paged_kv_cache_273_gb300 import pkv
    import parity_harness as PH
    inp, window = _draw(seed)
    case = PH.build(inp)
    PH.append_step(case, 0)
    wl = case.wl
    lens = inp.lens_after_step(0)
    q = PH.to_device(inp.step_q[0], wl.q_dtype)
    out = torch.full((wl.batch, wl.num_q_heads, wl.head_dim), float("nan"), dtype=torch.float32,
                     device="cuda")
    scale = 1.0 / np.sqrt(wl.head_dim)
    pkv.paged_decode_attention_window(
        case.pool, q, case.gk.tensor, case.gv.tensor, case.tables_d,
        torch.from_numpy(lens).cuda(), scale, out, case.workspace, int(lens.max()), window,
        None if case.gks is None else case.gks.tensor,
        None if case.gvs is None else case.gvs.tensor)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    want = O.paged_decode_attention(inp.step_q[0], wl.q_dtype, case.ok, case.ov, wl.kv_dtype,
                                    inp.block_tables, lens, float(np.float32(scale)), case.oks,
                                    case.ovs, window=window)
    err = float(np.max(np.abs(got - want)))
    assert err <= PH.TOL[wl.kv_dtype], (err, wl, window)
    assert PH.caches_equal(case)
    assert pkv.pkv_check_error(case.pool) == pkv.PKV_OK
    assert case.guards_intact()
    assert PH.counters_zero(case)
