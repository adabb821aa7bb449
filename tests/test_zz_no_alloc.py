"""The decode-attention entry point that allocates nothing.

paged_decode_attention_noalloc serves callers that cannot allocate device
memory when they call (for example from an allocator hook, or in a serving
loop that must not allocate after start-up): instead of a caller workspace it
uses a fixed scratch array in the library's device image.  These tests call it
through the C ABI and check it against the workspace entry point.  The file
is collected last so that a failure here stops a `-x` run only after every
other test has run; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_273_gb300 import pkv
from paged_kv_cache_273_gb300 import workloads as W

from parity_harness import TOL, append_step, attend_gpu, build, to_device

pytestmark = pytest.mark.gpu


def _noalloc(case, s):
    wl = case.wl
    lens = case.inp.lens_after_step(s)
    q = to_device(case.inp.step_q[s], wl.q_dtype)
    out = torch.full((wl.batch, wl.num_q_heads, wl.head_dim), float("nan"), dtype=torch.float32,
                     device="cuda")
    pkv.paged_decode_attention_noalloc(case.pool, q, case.gk.tensor, case.gv.tensor, case.tables_d,
                                       torch.from_numpy(lens).cuda(), 1.0 / np.sqrt(wl.head_dim),
                                       out, int(lens.max()))
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("name", ["llama2_70b", "gpt2"])
def test_noalloc_matches_workspace_entry_point_on_two_calls(name):
    # llama2_70b splits long sequences over many CTAs, so the shared counters
    # and partials in the scratch array are exercised; gpt2 has many pieces.
    case = build(W.make_inputs(name))
    append_step(case, 0)
    want = attend_gpu(case, 0)
    for _ in range(2):
        got = _noalloc(case, 0)
        assert np.all(np.isfinite(got))
        assert np.max(np.abs(got - want)) <= TOL[case.wl.kv_dtype]
    assert pkv.pkv_check_error(case.pool) == pkv.PKV_OK


def test_noalloc_rejects_batches_beyond_its_scratch():
    pool = pkv.kv_block_pool_init(16, 16, 8, 128, pkv.PKV_BF16)
    kc, vc, _, _ = pool.alloc_cache()
    B = 4096                                   # 32,768 (sequence, KV head) pairs at G = 8
    q = torch.zeros((B, 64, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((B, 64, 128), dtype=torch.float32, device="cuda")
    tables = torch.zeros((B, 1), dtype=torch.int32, device="cuda")
    lens = torch.ones(B, dtype=torch.int32, device="cuda")
    assert pkv.paged_decode_workspace_bytes(pool, B, 64) > (4 << 20)
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_attention_noalloc(pool, q, kc, vc, tables, lens, 0.1, out, 16)
    assert e.value.status == pkv.PKV_ERR_UNSUPPORTED
