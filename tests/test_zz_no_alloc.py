"""The decode-attention entry point that allocates nothing.

paged_decode_attention_noalloc serves callers that cannot allocate device
memory when they call (for example from an allocator hook, or in a serving
loop that must not allocate after start-up): instead of a caller workspace it
uses a fixed scratch array in the library's device image.  These tests call it
through the C ABI and check it against the workspace entry point (the same
deterministic kernel, so the outputs must be bit-identical) and against the
fp64 oracle.  The file is collected last so that a failure here stops a `-x`
run only after every other test has run; it also passes on its own in a fresh
process.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_273_gb300 import pkv
from paged_kv_cache_273_gb300 import workloads as W

from parity_harness import TOL, append_step, attend_gpu, attend_oracle, build, to_device

pytestmark = pytest.mark.gpu


class _Call:
    """Device buffers of one no-alloc call, made once so that repeated calls
    allocate nothing on the torch side either."""

    def __init__(self, case, s):
        wl = case.wl
        self.case = case
        self.lens_h = case.inp.lens_after_step(s)
        self.q = to_device(case.inp.step_q[s], wl.q_dtype)
        self.lens = torch.from_numpy(self.lens_h).cuda()
        self.out = torch.empty((wl.batch, wl.num_q_heads, wl.head_dim), dtype=torch.float32,
                               device="cuda")

    def __call__(self):
        c, wl = self.case, self.case.wl
        self.out.fill_(float("nan"))
        pkv.paged_decode_attention_noalloc(
            c.pool, self.q, c.gk.tensor, c.gv.tensor, c.tables_d, self.lens,
            1.0 / np.sqrt(wl.head_dim), self.out, int(self.lens_h.max()),
            None if c.gks is None else c.gks.tensor, None if c.gvs is None else c.gvs.tensor)
        torch.cuda.synchronize()
        return self.out.cpu().numpy()


@pytest.mark.parametrize("name", ["llama2_70b", "gpt2", "int8"])
def test_noalloc_matches_workspace_entry_point_on_two_calls(name):
    # llama2_70b splits long sequences over many CTAs, so the shared counters
    # and partials in the scratch array are exercised; gpt2 has many pieces;
    # int8 passes the scale arrays through.
    case = build(W.make_inputs(name))
    append_step(case, 0)
    want = attend_gpu(case, 0)
    ref = attend_oracle(case, 0)
    call = _Call(case, 0)
    for _ in range(2):
        got = call()
        # the same kernel with the same inputs and merge order: bit-identical
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
        assert np.max(np.abs(got - ref)) <= TOL[case.wl.kv_dtype]
    assert pkv.pkv_check_error(case.pool) == pkv.PKV_OK


def test_noalloc_calls_leave_free_device_memory_unchanged():
    # After one warm call (which may load the library's device image, and
    # with it the scratch array), further calls must not change the device's
    # free memory: they allocate nothing.
    case = build(W.make_inputs("llama2_70b"))
    append_step(case, 0)
    call = _Call(case, 0)
    first = call()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        got = call()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert np.array_equal(got.view(np.uint32), first.view(np.uint32))


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
