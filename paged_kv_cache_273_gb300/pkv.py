"""Python binding of libpkv (ctypes), one function per C-ABI entry point.

Argument marshalling only: every step of the hot path runs in libpkv's CUDA
kernels.  PyTorch supplies device memory and streams.  If libpkv.so has not
been built, importing the library raises; there is no CPU fallback.

Device tensors follow the layouts of ``include/pkv.h``:
  k_cache, v_cache   [NB, Hkv, bs, D]   (float32 | float16 | bfloat16 | int8)
  k_scales, v_scales [NB, Hkv, bs]      float16 (int8 pools only)
  q                  [B, Hq, D];  out [B, Hq, D] float32
  block_tables       [B, max_blocks_per_seq] int32;  seq_lens [B] int32
  slot_mapping       [T] int32
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkv.so")

PKV_F32, PKV_F16, PKV_BF16, PKV_I8, PKV_I4 = 0, 1, 2, 3, 4
PKV_OK = 0
PKV_ERR_INVALID = -1
PKV_ERR_NO_BLOCKS = -2
PKV_ERR_CUDA = -3
PKV_ERR_UNSUPPORTED = -4
PKV_ERR_BAD_INDEX = -5
PKV_ERR_TIMEOUT = -6

TORCH_DTYPE = {PKV_F32: torch.float32, PKV_F16: torch.float16, PKV_BF16: torch.bfloat16,
               PKV_I8: torch.int8}
PKV_DTYPE = {v: k for k, v in TORCH_DTYPE.items()}
# 4-bit caches are held as bytes, two codes each: [NB, Hkv, bs, D/2] uint8.
TORCH_DTYPE[PKV_I4] = torch.uint8

# Every symbol the header declares (checked by the tests).
SYMBOLS = ("pkv_status_string", "kv_block_pool_init", "kv_block_pool_destroy", "kv_cache_bytes",
           "kv_scales_bytes", "kv_num_free_blocks", "kv_block_refcount", "kv_block_alloc",
           "kv_block_share", "kv_block_free", "kv_reserve_slots", "kv_reserve_slots_cow",
           "kv_slot_mapping", "kv_append", "kv_block_copy", "paged_decode_workspace_bytes", "paged_decode_attention",
           "paged_decode_attention_window", "paged_prefill_attention", "kv_prefix_groups",
           "paged_decode_cascade_workspace_bytes", "paged_decode_attention_cascade",
           "paged_decode_attention_noalloc", "paged_decode_step", "pkv_selftest_wait_timeout",
           "pkv_check_error")


class StepLayout(ctypes.Structure):
    """pkv_step_layout: byte offsets of one decode step's inputs in a staging
    buffer."""
    _fields_ = [("k_new", ctypes.c_size_t), ("v_new", ctypes.c_size_t), ("q", ctypes.c_size_t),
                ("slot_mapping", ctypes.c_size_t), ("seq_lens", ctypes.c_size_t)]


class PkvError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s (status %d)" % (where, status_string(status), status))


_lock = threading.Lock()
_lib = None


def load() -> ctypes.CDLL:
    """Load libpkv.so (built by ``paged_kv_cache_273_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError("libpkv.so is not built (%s); run "
                              "`python -m paged_kv_cache_273_gb300.build`" % LIB_PATH)
        lib = ctypes.CDLL(LIB_PATH)
        P, I, I32P, SZ, F = (ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_int32),
                             ctypes.c_size_t, ctypes.c_float)
        lib.pkv_status_string.argtypes = [I]
        lib.pkv_status_string.restype = ctypes.c_char_p
        lib.kv_block_pool_init.argtypes = [ctypes.POINTER(P), I, I, I, I, I]
        lib.kv_block_pool_init.restype = I
        lib.kv_block_pool_destroy.argtypes = [P]
        lib.kv_block_pool_destroy.restype = None
        lib.kv_cache_bytes.argtypes = [P]
        lib.kv_cache_bytes.restype = SZ
        lib.kv_scales_bytes.argtypes = [P]
        lib.kv_scales_bytes.restype = SZ
        lib.kv_num_free_blocks.argtypes = [P]
        lib.kv_num_free_blocks.restype = I
        lib.kv_block_refcount.argtypes = [P, ctypes.c_int32]
        lib.kv_block_refcount.restype = I
        lib.kv_block_alloc.argtypes = [P, I, I32P]
        lib.kv_block_alloc.restype = I
        lib.kv_block_share.argtypes = [P, I32P, I]
        lib.kv_block_share.restype = I
        lib.kv_block_free.argtypes = [P, I32P, I]
        lib.kv_block_free.restype = I
        lib.kv_reserve_slots.argtypes = [P, I, I32P, I32P, I32P, I, I32P]
        lib.kv_reserve_slots.restype = I
        lib.kv_reserve_slots_cow.argtypes = [P, I, I32P, I32P, I32P, I, I32P, I32P, I32P,
                                             ctypes.POINTER(I)]
        lib.kv_reserve_slots_cow.restype = I
        lib.kv_block_copy.argtypes = [P, P, P, I, P, P, P, P, P]
        lib.kv_block_copy.restype = I
        lib.kv_slot_mapping.argtypes = [I32P, I, I, I, I32P, I32P, I32P]
        lib.kv_slot_mapping.restype = I
        lib.kv_append.argtypes = [P, P, P, I, P, I, P, P, P, P, P]
        lib.kv_append.restype = I
        lib.paged_decode_workspace_bytes.argtypes = [P, I, I]
        lib.paged_decode_workspace_bytes.restype = SZ
        lib.paged_decode_attention.argtypes = [P, P, I, I, P, P, P, P, P, I, P, I, I, F, P, P,
                                               SZ, P]
        lib.paged_decode_attention.restype = I
        lib.paged_decode_attention_window.argtypes = [P, P, I, I, P, P, P, P, P, I, P, I, I, I,
                                                      F, P, P, SZ, P]
        lib.paged_decode_attention_window.restype = I
        lib.paged_prefill_attention.argtypes = [P, P, I, P, P, P, I, P, P, I, I, F, P, P]
        lib.paged_prefill_attention.restype = I
        IP = ctypes.POINTER(I)
        lib.kv_prefix_groups.argtypes = [I32P, I, I32P, I, I, I, I32P, I32P, I32P, I32P, IP, IP,
                                         IP]
        lib.kv_prefix_groups.restype = I
        lib.paged_decode_cascade_workspace_bytes.argtypes = [P, I, I, I]
        lib.paged_decode_cascade_workspace_bytes.restype = SZ
        lib.paged_decode_attention_cascade.argtypes = [P, P, I, I, P, P, P, I, P, I, I, P, P, P,
                                                       P, I, I, I, F, P, P, SZ, P]
        lib.paged_decode_attention_cascade.restype = I
        lib.paged_decode_attention_noalloc.argtypes = [P, P, I, I, P, P, P, P, P, I, P, I, I, F,
                                                       P, P]
        lib.paged_decode_attention_noalloc.restype = I
        lib.paged_decode_step.argtypes = [P, P, P, SZ, ctypes.POINTER(StepLayout), I, I, I, P, P,
                                          P, P, P, I, I, I, F, P, P, P, SZ, P]
        lib.paged_decode_step.restype = I
        lib.pkv_selftest_wait_timeout.argtypes = [P, P]
        lib.pkv_selftest_wait_timeout.restype = I
        lib.pkv_check_error.argtypes = [P, P]
        lib.pkv_check_error.restype = I
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().pkv_status_string(int(status)).decode()


def _check(status: int, where: str) -> int:
    if status < 0:
        raise PkvError(status, where)
    return status


def _i32(a) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a


def _i32p(a: np.ndarray | None):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _dptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


class Pool:
    """Handle of a ``pkv_pool`` (host bookkeeping of one shared block pool)."""

    def __init__(self, handle: int, num_blocks: int, block_size: int, num_kv_heads: int,
                 head_dim: int, kv_dtype: int):
        self.handle = ctypes.c_void_p(handle)
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.num_kv_heads = num_kv_heads
        self.head_dim = head_dim
        self.kv_dtype = kv_dtype

    def close(self):
        if self.handle:
            load().kv_block_pool_destroy(self.handle)
            self.handle = ctypes.c_void_p(None)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # convenience: caller-owned device buffers of the right shape
    def alloc_cache(self, device="cuda"):
        shape = (self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim)
        dt = TORCH_DTYPE[self.kv_dtype]
        if self.kv_dtype == PKV_I4:
            shape = shape[:3] + (self.head_dim // 2,)
        k = torch.zeros(shape, dtype=dt, device=device)
        v = torch.zeros(shape, dtype=dt, device=device)
        if self.kv_dtype in (PKV_I8, PKV_I4):
            sshape = shape[:3]
            return (k, v, torch.zeros(sshape, dtype=torch.float16, device=device),
                    torch.zeros(sshape, dtype=torch.float16, device=device))
        return k, v, None, None


# ------------------------------------------------------------------ pool (host)
def kv_block_pool_init(num_blocks, block_size, num_kv_heads, head_dim, kv_dtype) -> Pool:
    h = ctypes.c_void_p()
    _check(load().kv_block_pool_init(ctypes.byref(h), num_blocks, block_size, num_kv_heads,
                                     head_dim, int(kv_dtype)), "kv_block_pool_init")
    return Pool(h.value, num_blocks, block_size, num_kv_heads, head_dim, int(kv_dtype))


def kv_block_pool_destroy(pool: Pool) -> None:
    pool.close()


def kv_cache_bytes(pool: Pool) -> int:
    return int(load().kv_cache_bytes(pool.handle))


def kv_scales_bytes(pool: Pool) -> int:
    return int(load().kv_scales_bytes(pool.handle))


def kv_num_free_blocks(pool: Pool) -> int:
    return _check(load().kv_num_free_blocks(pool.handle), "kv_num_free_blocks")


def kv_block_refcount(pool: Pool, block_id: int) -> int:
    return _check(load().kv_block_refcount(pool.handle, int(block_id)), "kv_block_refcount")


def kv_block_alloc(pool: Pool, n: int) -> np.ndarray:
    out = np.zeros(max(n, 1), np.int32)
    _check(load().kv_block_alloc(pool.handle, n, _i32p(out)), "kv_block_alloc")
    return out[:n]


def kv_block_share(pool: Pool, ids) -> None:
    ids = _i32(ids)
    _check(load().kv_block_share(pool.handle, _i32p(ids), ids.size), "kv_block_share")


def kv_block_free(pool: Pool, ids) -> None:
    ids = _i32(ids)
    _check(load().kv_block_free(pool.handle, _i32p(ids), ids.size), "kv_block_free")


def kv_reserve_slots(pool: Pool, seq_lens, block_tables: np.ndarray, num_new=None) -> np.ndarray:
    """Allocate blocks for one append step; block_tables (int32 numpy, C order) is updated
    in place.  Returns the slot mapping."""
    if block_tables.dtype != np.int32 or not block_tables.flags.c_contiguous:
        raise ValueError("block_tables must be a C-contiguous int32 array")
    sl = _i32(seq_lens)
    nn = None if num_new is None else _i32(num_new)
    total = sl.size if nn is None else int(nn.sum())
    slots = np.zeros(max(total, 1), np.int32)
    _check(load().kv_reserve_slots(pool.handle, sl.size, _i32p(sl), _i32p(nn),
                                   _i32p(block_tables), block_tables.shape[1], _i32p(slots)),
           "kv_reserve_slots")
    return slots[:total]


def kv_reserve_slots_cow(pool: Pool, seq_lens, block_tables: np.ndarray, num_new=None):
    """kv_reserve_slots for tables that may share blocks.  Returns (slots, copy_src,
    copy_dst): the pairs of blocks to copy with kv_block_copy before the append."""
    if block_tables.dtype != np.int32 or not block_tables.flags.c_contiguous:
        raise ValueError("block_tables must be a C-contiguous int32 array")
    sl = _i32(seq_lens)
    nn = None if num_new is None else _i32(num_new)
    total = sl.size if nn is None else int(nn.sum())
    slots = np.zeros(max(total, 1), np.int32)
    src = np.zeros(max(sl.size, 1), np.int32)
    dst = np.zeros(max(sl.size, 1), np.int32)
    ncopy = ctypes.c_int(0)
    _check(load().kv_reserve_slots_cow(pool.handle, sl.size, _i32p(sl), _i32p(nn),
                                       _i32p(block_tables), block_tables.shape[1], _i32p(slots),
                                       _i32p(src), _i32p(dst), ctypes.byref(ncopy)),
           "kv_reserve_slots_cow")
    n = ncopy.value
    return slots[:total], src[:n].copy(), dst[:n].copy()


def kv_slot_mapping(block_tables, block_size: int, start, num_new=None,
                    out: np.ndarray | None = None) -> np.ndarray:
    """Slots of the new tokens; `out` (contiguous int32 of the slot count, for
    example a slice of a staging buffer) receives them in place if given."""
    bt = _i32(block_tables)
    st = _i32(start)
    nn = None if num_new is None else _i32(num_new)
    total = st.size if nn is None else int(nn.sum())
    if out is None:
        slots = np.zeros(max(total, 1), np.int32)
    else:
        if out.dtype != np.int32 or out.size != total or not out.flags.c_contiguous:
            raise ValueError("out must be a contiguous int32 array of the slot count")
        slots = out
    _check(load().kv_slot_mapping(_i32p(bt), bt.shape[1], block_size, st.size, _i32p(st),
                                  _i32p(nn), _i32p(slots) if slots.size else None),
           "kv_slot_mapping")
    return slots[:total]


# ------------------------------------------------------------------ device calls
def kv_append(pool: Pool, k_new, v_new, slot_mapping, k_cache, v_cache, k_scales=None,
              v_scales=None, stream=None) -> None:
    if k_new.dtype not in PKV_DTYPE:
        raise ValueError("unsupported k_new dtype %s" % k_new.dtype)
    if slot_mapping.dtype != torch.int32:
        raise ValueError("slot_mapping must be int32")
    T = k_new.shape[0]
    _check(load().kv_append(pool.handle, _dptr(k_new), _dptr(v_new), PKV_DTYPE[k_new.dtype],
                            _dptr(slot_mapping), T, _dptr(k_cache), _dptr(v_cache),
                            _dptr(k_scales), _dptr(v_scales), _stream(stream)), "kv_append")


def kv_block_copy(pool: Pool, src, dst, k_cache, v_cache, k_scales=None, v_scales=None,
                  stream=None) -> None:
    """Copy blocks src[i] -> dst[i] (device int32 tensors) in the caches."""
    if src.dtype != torch.int32 or dst.dtype != torch.int32 or src.numel() != dst.numel():
        raise ValueError("src and dst must be int32 tensors of equal length")
    _check(load().kv_block_copy(pool.handle, _dptr(src), _dptr(dst), src.numel(),
                                _dptr(k_cache), _dptr(v_cache), _dptr(k_scales),
                                _dptr(v_scales), _stream(stream)), "kv_block_copy")


def paged_decode_workspace_bytes(pool: Pool, batch: int, num_q_heads: int) -> int:
    return int(load().paged_decode_workspace_bytes(pool.handle, batch, num_q_heads))


def alloc_workspace(pool: Pool, batch: int, num_q_heads: int, device="cuda") -> torch.Tensor:
    """A zeroed workspace (its counters must start at zero)."""
    n = paged_decode_workspace_bytes(pool, batch, num_q_heads)
    if n == 0:
        raise PkvError(PKV_ERR_INVALID, "paged_decode_workspace_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def paged_decode_attention(pool: Pool, q, k_cache, v_cache, block_tables, seq_lens, scale: float,
                           out, workspace, max_seq_len: int, k_scales=None, v_scales=None,
                           stream=None) -> None:
    if q.dtype not in PKV_DTYPE:
        raise ValueError("unsupported q dtype %s" % q.dtype)
    if out.dtype != torch.float32:
        raise ValueError("out must be float32")
    if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise ValueError("block_tables and seq_lens must be int32")
    B, Hq, _ = q.shape
    _check(load().paged_decode_attention(
        pool.handle, _dptr(q), PKV_DTYPE[q.dtype], Hq, _dptr(k_cache), _dptr(v_cache),
        _dptr(k_scales), _dptr(v_scales), _dptr(block_tables), block_tables.shape[1],
        _dptr(seq_lens), B, int(max_seq_len), float(scale), _dptr(out), _dptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)), "paged_decode_attention")


def paged_decode_attention_window(pool: Pool, q, k_cache, v_cache, block_tables, seq_lens,
                                  scale: float, out, workspace, max_seq_len: int, window: int,
                                  k_scales=None, v_scales=None, stream=None) -> None:
    """paged_decode_attention over the last `window` rows of each sequence (0 = all)."""
    if q.dtype not in PKV_DTYPE:
        raise ValueError("unsupported q dtype %s" % q.dtype)
    if out.dtype != torch.float32:
        raise ValueError("out must be float32")
    if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise ValueError("block_tables and seq_lens must be int32")
    B, Hq, _ = q.shape
    _check(load().paged_decode_attention_window(
        pool.handle, _dptr(q), PKV_DTYPE[q.dtype], Hq, _dptr(k_cache), _dptr(v_cache),
        _dptr(k_scales), _dptr(v_scales), _dptr(block_tables), block_tables.shape[1],
        _dptr(seq_lens), B, int(max_seq_len), int(window), float(scale), _dptr(out),
        _dptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)),
        "paged_decode_attention_window")


def paged_prefill_attention(pool: Pool, q, k_cache, v_cache, block_tables, q_start, seq_lens,
                            scale: float, out, max_q_len: int, stream=None) -> None:
    """Causal attention of the new tokens (q: [T, Hq, D], sequence-major, offsets
    q_start [B+1]) over their cached rows; out fp32 [T, Hq, D]."""
    if out.dtype != torch.float32:
        raise ValueError("out must be float32")
    for t in (block_tables, q_start, seq_lens):
        if t.dtype != torch.int32:
            raise ValueError("block_tables, q_start and seq_lens must be int32")
    _check(load().paged_prefill_attention(
        pool.handle, _dptr(q), q.shape[1], _dptr(k_cache), _dptr(v_cache), _dptr(block_tables),
        block_tables.shape[1], _dptr(q_start), _dptr(seq_lens), seq_lens.numel(), int(max_q_len),
        float(scale), _dptr(out), _stream(stream)), "paged_prefill_attention")


def kv_prefix_groups(block_tables, seq_lens, block_size: int, min_prefix_blocks: int = 1) -> dict:
    """Host: groups of sequences sharing leading blocks (see include/pkv.h).
    Returns numpy int32 arrays group_start, group_seqs, group_prefix,
    seq_prefix and the ints num_groups, max_group_size, max_prefix_len."""
    bt = _i32(block_tables)
    sl = _i32(seq_lens)
    B = sl.size
    gs = np.zeros(B + 1, np.int32)
    gq = np.zeros(max(B, 1), np.int32)
    gp = np.zeros(max(B, 1), np.int32)
    sp = np.zeros(max(B, 1), np.int32)
    ng, mg, mp = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    _check(load().kv_prefix_groups(_i32p(bt), bt.shape[1] if bt.ndim == 2 else 0, _i32p(sl), B,
                                   block_size, min_prefix_blocks, _i32p(gs), _i32p(gq), _i32p(gp),
                                   _i32p(sp), ctypes.byref(ng), ctypes.byref(mg),
                                   ctypes.byref(mp)), "kv_prefix_groups")
    n = ng.value
    return {"group_start": gs[:n + 1].copy(), "group_seqs": gq[:int(gs[n])].copy(),
            "group_prefix": gp[:n].copy(), "seq_prefix": sp[:B].copy(), "num_groups": n,
            "max_group_size": mg.value, "max_prefix_len": mp.value}


def paged_decode_cascade_workspace_bytes(pool: Pool, batch: int, num_q_heads: int,
                                         max_prefix_len: int) -> int:
    return int(load().paged_decode_cascade_workspace_bytes(pool.handle, batch, num_q_heads,
                                                           max_prefix_len))


def alloc_cascade_workspace(pool: Pool, batch: int, num_q_heads: int, max_prefix_len: int,
                            device="cuda") -> torch.Tensor:
    """A zeroed workspace for paged_decode_attention_cascade."""
    n = paged_decode_cascade_workspace_bytes(pool, batch, num_q_heads, max_prefix_len)
    if n == 0:
        raise PkvError(PKV_ERR_INVALID, "paged_decode_cascade_workspace_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def prefix_groups_to_device(groups: dict, device="cuda") -> dict:
    """kv_prefix_groups' arrays as device int32 tensors (the ints unchanged)."""
    out = dict(groups)
    for k in ("group_start", "group_seqs", "group_prefix", "seq_prefix"):
        a = groups[k]
        out[k] = torch.from_numpy(a if a.size else np.zeros(1, np.int32)).to(device)
    return out


def paged_decode_attention_cascade(pool: Pool, q, k_cache, v_cache, block_tables, seq_lens,
                                   scale: float, out, workspace, max_seq_len: int, groups: dict,
                                   stream=None) -> None:
    """paged_decode_attention with shared prefixes scored once per group;
    groups: prefix_groups_to_device(kv_prefix_groups(...))."""
    if q.dtype not in PKV_DTYPE:
        raise ValueError("unsupported q dtype %s" % q.dtype)
    if out.dtype != torch.float32:
        raise ValueError("out must be float32")
    if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise ValueError("block_tables and seq_lens must be int32")
    B, Hq, _ = q.shape
    _check(load().paged_decode_attention_cascade(
        pool.handle, _dptr(q), PKV_DTYPE[q.dtype], Hq, _dptr(k_cache), _dptr(v_cache),
        _dptr(block_tables), block_tables.shape[1], _dptr(seq_lens), B, int(max_seq_len),
        _dptr(groups["group_start"]), _dptr(groups["group_seqs"]), _dptr(groups["group_prefix"]),
        _dptr(groups["seq_prefix"]), int(groups["num_groups"]), int(groups["max_group_size"]),
        int(groups["max_prefix_len"]), float(scale), _dptr(out), _dptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)),
        "paged_decode_attention_cascade")


def paged_decode_attention_noalloc(pool: Pool, q, k_cache, v_cache, block_tables, seq_lens,
                                   scale: float, out, max_seq_len: int, k_scales=None,
                                   v_scales=None, stream=None) -> None:
    """paged_decode_attention without a caller workspace (for callers that
    cannot allocate device memory; the library's fixed scratch array is used)."""
    if q.dtype not in PKV_DTYPE:
        raise ValueError("unsupported q dtype %s" % q.dtype)
    if out.dtype != torch.float32:
        raise ValueError("out must be float32")
    if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise ValueError("block_tables and seq_lens must be int32")
    B, Hq, _ = q.shape
    _check(load().paged_decode_attention_noalloc(
        pool.handle, _dptr(q), PKV_DTYPE[q.dtype], Hq, _dptr(k_cache), _dptr(v_cache),
        _dptr(k_scales), _dptr(v_scales), _dptr(block_tables), block_tables.shape[1],
        _dptr(seq_lens), B, int(max_seq_len), float(scale), _dptr(out), _stream(stream)),
        "paged_decode_attention_noalloc")


def _hptr(t: torch.Tensor | None):
    if t is None:
        return None
    if t.is_cuda:
        raise ValueError("expected a host tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


class DecodeStep:
    """paged_decode_step with its fixed arguments marshalled once: a serving
    loop calls step(host_in, host_out) per decode step.  host_in: a host
    uint8 tensor (page-locked for an asynchronous copy) holding the step's
    inputs at the offsets of `layout` (a StepLayout); dev_in: a device uint8
    tensor of at least host_in's size; host_out: a host fp32 tensor of
    out's shape, or None (a page-locked host_out receives the output
    directly and `out` is then left unwritten).  Nothing waits: record an
    event after the call and synchronize on it before reusing host_in or
    reading host_out."""

    def __init__(self, pool: Pool, dev_in, layout: StepLayout, in_dtype, q_dtype,
                 num_q_heads: int, k_cache, v_cache, block_tables, batch: int, max_seq_len: int,
                 scale: float, out, workspace, k_scales=None, v_scales=None, stream=None):
        if in_dtype not in PKV_DTYPE or q_dtype not in PKV_DTYPE:
            raise ValueError("unsupported dtype")
        if out.dtype != torch.float32:
            raise ValueError("out must be float32")
        if block_tables.dtype != torch.int32:
            raise ValueError("block_tables must be int32")
        if dev_in.dtype != torch.uint8:
            raise ValueError("dev_in must be a uint8 tensor")
        self.pool = pool
        self.layout = layout
        self.in_bytes = dev_in.numel()
        self._keep = (dev_in, k_cache, v_cache, block_tables, out, workspace, k_scales,
                      v_scales)
        self._head = (pool.handle,)
        self._mid = (_dptr(dev_in), ctypes.c_size_t(self.in_bytes), ctypes.byref(layout),
                     PKV_DTYPE[in_dtype], PKV_DTYPE[q_dtype], int(num_q_heads), _dptr(k_cache),
                     _dptr(v_cache), _dptr(k_scales), _dptr(v_scales), _dptr(block_tables),
                     block_tables.shape[1], int(batch), int(max_seq_len), float(scale),
                     _dptr(out))
        self._tail = (_dptr(workspace), workspace.numel() * workspace.element_size(),
                      _stream(stream))
        self._fn = load().paged_decode_step

    def __call__(self, host_in, host_out=None) -> None:
        if host_in.numel() * host_in.element_size() != self.in_bytes:
            raise ValueError("host_in must have dev_in's size")
        _check(self._fn(*self._head, _hptr(host_in), *self._mid, _hptr(host_out),
                        *self._tail), "paged_decode_step")


def paged_decode_step(pool: Pool, host_in, dev_in, layout: StepLayout, in_dtype, q_dtype,
                      num_q_heads: int, k_cache, v_cache, block_tables, batch: int,
                      max_seq_len: int, scale: float, out, host_out, workspace, k_scales=None,
                      v_scales=None, stream=None) -> None:
    """One decode step with host buffers (see DecodeStep)."""
    DecodeStep(pool, dev_in, layout, in_dtype, q_dtype, num_q_heads, k_cache, v_cache,
               block_tables, batch, max_seq_len, scale, out, workspace, k_scales, v_scales,
               stream)(host_in, host_out)


def pkv_selftest_wait_timeout(pool: Pool, stream=None) -> None:
    """Launch a kernel whose bounded wait runs out (about a second); the next
    pkv_check_error() returns PKV_ERR_TIMEOUT."""
    _check(load().pkv_selftest_wait_timeout(pool.handle, _stream(stream)),
           "pkv_selftest_wait_timeout")


def pkv_check_error(pool: Pool, stream=None) -> int:
    """Synchronise and read/clear the device error word; returns the status (no raise)."""
    return int(load().pkv_check_error(pool.handle, _stream(stream) if torch.cuda.is_available()
                                      else ctypes.c_void_p(None)))
