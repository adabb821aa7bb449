"""Runs one workload through libpkv (CUDA) and through the CPU oracle, and
compares them: slot mapping and caches bit for bit, attention within the
tolerance of the K/V type.

Used by the GPU tests and by ``__graft_entry__.smoke()``.  Both sides get the
same seeded raw inputs from ``paged_kv_cache_273_gb300.workloads``; nothing
the CUDA path produces is fed to the oracle.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

from oracle import oracle as O
from paged_kv_cache_273_gb300 import pkv
from paged_kv_cache_273_gb300 import workloads as W

# Max-abs attention error allowed against the fp64 oracle: fp32 accumulation
# over fp32/fp16/bf16 K/V, and int8 K/V (the oracle attends over the same
# dequantized codes, so the budget covers fp32 rounding only, with margin).
TOL = {W.F32: 2e-3, W.F16: 2e-3, W.BF16: 2e-3, W.I8: 2e-2, W.I4: 2e-2}

_NP_RAW = {W.F32: np.float32, W.F16: np.uint16, W.BF16: np.uint16, W.I8: np.int8,
           W.I4: np.uint8}
_TORCH = {W.F32: torch.float32, W.F16: torch.float16, W.BF16: torch.bfloat16, W.I8: torch.int8,
          W.I4: torch.uint8}
_QUANT = (W.I8, W.I4)

GUARD = 4096  # canary bytes on each side of every guarded buffer
CANARY = 0x5A


def to_device(raw: np.ndarray, code: int, device="cuda") -> torch.Tensor:
    """Raw numpy bits -> CUDA tensor of the matching dtype (bit-identical)."""
    raw = np.ascontiguousarray(raw)
    if code in (W.F16, W.BF16):
        t = torch.from_numpy(raw.view(np.int16)).to(device).view(_TORCH[code])
    else:
        t = torch.from_numpy(raw).to(device)
    return t


def to_raw(t: torch.Tensor, code: int) -> np.ndarray:
    t = t.detach().contiguous().cpu()
    if code in (W.F16, W.BF16):
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


class Guarded:
    """A device tensor with canary bytes around it (out-of-bounds writes show up)."""

    def __init__(self, shape, dtype, device="cuda"):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.nbytes = n
        self.buf = torch.full((n + 2 * GUARD,), CANARY, dtype=torch.uint8, device=device)
        self.tensor = self.buf[GUARD:GUARD + n].view(dtype).view(shape)
        self.tensor.zero_()

    def intact(self) -> bool:
        head = self.buf[:GUARD]
        tail = self.buf[GUARD + self.nbytes:]
        return bool(torch.all(head == CANARY).item() and torch.all(tail == CANARY).item())


@dataclasses.dataclass
class Case:
    inp: W.Inputs
    pool: pkv.Pool
    gk: Guarded
    gv: Guarded
    gks: Guarded | None
    gvs: Guarded | None
    tables_d: torch.Tensor
    workspace: torch.Tensor
    # oracle state
    ok: np.ndarray
    ov: np.ndarray
    oks: np.ndarray | None
    ovs: np.ndarray | None

    @property
    def wl(self) -> W.Workload:
        return self.inp.workload

    def guards_intact(self) -> bool:
        gs = [self.gk, self.gv] + [g for g in (self.gks, self.gvs) if g is not None]
        return all(g.intact() for g in gs)


def _append_oracle(case: Case, rows_k, rows_v, slots):
    wl = case.wl
    if wl.kv_dtype == W.I8:
        O.append_q8(rows_k, rows_v, wl.src_dtype, slots, wl.block_size, case.ok, case.ov,
                    case.oks, case.ovs)
    elif wl.kv_dtype == W.I4:
        O.append_q4(rows_k, rows_v, wl.src_dtype, slots, wl.block_size, case.ok, case.ov,
                    case.oks, case.ovs)
    else:
        O.append(rows_k, rows_v, wl.kv_dtype, slots, wl.block_size, case.ok, case.ov)


def build(inp: W.Inputs, device="cuda") -> Case:
    """Create the pool and caches on both sides and write the history rows."""
    wl = inp.workload
    B, Hq, Hkv, D, bs = wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.block_size
    NB = inp.num_blocks
    pool = pkv.kv_block_pool_init(NB, bs, Hkv, D, wl.kv_dtype)
    shape = (NB, Hkv, bs, D // 2 if wl.kv_dtype == W.I4 else D)   # 4-bit: two codes a byte
    gk = Guarded(shape, _TORCH[wl.kv_dtype], device)
    gv = Guarded(shape, _TORCH[wl.kv_dtype], device)
    gks = gvs = None
    ok = np.zeros(shape, _NP_RAW[wl.kv_dtype])
    ov = np.zeros(shape, _NP_RAW[wl.kv_dtype])
    oks = ovs = None
    if wl.kv_dtype in _QUANT:
        gks = Guarded(shape[:3], torch.float16, device)
        gvs = Guarded(shape[:3], torch.float16, device)
        oks = np.zeros(shape[:3], np.uint16)
        ovs = np.zeros(shape[:3], np.uint16)
    tables_d = torch.from_numpy(inp.block_tables).to(device)
    ws = pkv.alloc_workspace(pool, B, Hq, device)
    case = Case(inp, pool, gk, gv, gks, gvs, tables_d, ws, ok, ov, oks, ovs)

    # history rows: slots from the library's host computation and from the oracle
    zeros = np.zeros(B, np.int32)
    slots = pkv.kv_slot_mapping(inp.block_tables, bs, zeros, inp.prefix_lens)
    oslots = O.slot_mapping(inp.block_tables, bs, zeros, inp.prefix_lens)
    assert np.array_equal(slots, oslots), "history slot mapping differs"
    slots = np.where(inp.hist_write, slots, -1).astype(np.int32)
    if slots.size:
        pkv.kv_append(pool, to_device(inp.hist_k, wl.src_dtype, device),
                      to_device(inp.hist_v, wl.src_dtype, device),
                      torch.from_numpy(slots).to(device), gk.tensor, gv.tensor,
                      None if gks is None else gks.tensor, None if gvs is None else gvs.tensor)
        _append_oracle(case, inp.hist_k, inp.hist_v, slots)
    return case


def step_slots(case: Case, s: int) -> np.ndarray:
    inp = case.inp
    start = (inp.prefix_lens + s).astype(np.int32)
    slots = pkv.kv_slot_mapping(inp.block_tables, case.wl.block_size, start)
    oslots = O.slot_mapping(inp.block_tables, case.wl.block_size, start,
                            np.ones(case.wl.batch, np.int32))
    assert np.array_equal(slots, oslots), "decode-step slot mapping differs"
    return np.where(inp.idle, -1, slots).astype(np.int32)


def append_step(case: Case, s: int, device="cuda"):
    wl = case.wl
    slots = step_slots(case, s)
    rows_k, rows_v = case.inp.step_k[s], case.inp.step_v[s]
    pkv.kv_append(case.pool, to_device(rows_k, wl.src_dtype, device),
                  to_device(rows_v, wl.src_dtype, device), torch.from_numpy(slots).to(device),
                  case.gk.tensor, case.gv.tensor,
                  None if case.gks is None else case.gks.tensor,
                  None if case.gvs is None else case.gvs.tensor)
    _append_oracle(case, rows_k, rows_v, slots)


def attend_gpu(case: Case, s: int, device="cuda", scale=None) -> np.ndarray:
    wl = case.wl
    lens = case.inp.lens_after_step(s)
    q = to_device(case.inp.step_q[s], wl.q_dtype, device)
    out = torch.empty((wl.batch, wl.num_q_heads, wl.head_dim), dtype=torch.float32, device=device)
    scale = 1.0 / np.sqrt(wl.head_dim) if scale is None else scale
    pkv.paged_decode_attention(case.pool, q, case.gk.tensor, case.gv.tensor, case.tables_d,
                               torch.from_numpy(lens).to(device), scale, out, case.workspace,
                               int(lens.max()) if lens.size else 0,
                               None if case.gks is None else case.gks.tensor,
                               None if case.gvs is None else case.gvs.tensor)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def attend_oracle(case: Case, s: int, seqs=None, scale=None) -> np.ndarray:
    wl = case.wl
    lens = case.inp.lens_after_step(s)
    q = case.inp.step_q[s]
    tables = case.inp.block_tables
    if seqs is not None:
        lens, q, tables = lens[seqs], q[seqs], tables[seqs]
    scale = 1.0 / np.sqrt(wl.head_dim) if scale is None else scale
    return O.paged_decode_attention(q, wl.q_dtype, case.ok, case.ov, wl.kv_dtype, tables, lens,
                                    float(np.float32(scale)), case.oks, case.ovs)


def caches_equal(case: Case) -> bool:
    wl = case.wl
    same = np.array_equal(to_raw(case.gk.tensor, wl.kv_dtype), case.ok) and \
        np.array_equal(to_raw(case.gv.tensor, wl.kv_dtype), case.ov)
    if wl.kv_dtype in _QUANT:
        same = same and np.array_equal(to_raw(case.gks.tensor, W.F16), case.oks) and \
            np.array_equal(to_raw(case.gvs.tensor, W.F16), case.ovs)
    return same


def run(inp: W.Inputs, steps=None, check_steps=None, seqs=None, device="cuda") -> dict:
    """Build, then for each decode step append and attend; compare with the oracle.

    Returns {"max_err": ..., "tol": ..., "cache_equal": bool, "error_word": status}.
    """
    wl = inp.workload
    case = build(inp, device)
    torch.cuda.synchronize()
    result = {"cache_equal_history": caches_equal(case)}
    nsteps = wl.decode_steps if steps is None else steps
    check = set(range(nsteps)) if check_steps is None else set(check_steps)
    max_err = 0.0
    for s in range(nsteps):
        append_step(case, s, device)
        if s in check:
            got = attend_gpu(case, s, device)
            want = attend_oracle(case, s, seqs)
            if seqs is not None:
                got = got[seqs]
            err = float(np.max(np.abs(got - want))) if got.size else 0.0
            max_err = max(max_err, err)
    torch.cuda.synchronize()
    result["cache_equal"] = caches_equal(case)
    result["max_err"] = max_err
    result["tol"] = TOL[wl.kv_dtype]
    result["error_word"] = pkv.pkv_check_error(case.pool)
    result["guards"] = case.guards_intact()
    result["counters_zero"] = counters_zero(case)
    return result


def counters_zero(case: Case) -> bool:
    """Every call must leave the workspace's per-(sequence, KV head) counters at zero."""
    n = case.wl.batch * case.wl.num_kv_heads
    return not bool(case.workspace[:n * 4].view(torch.int32).any().item())
