"""ctypes front end of the fp64 CPU oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The CUDA library never imports,
loads or calls anything in this directory, and this module imports nothing
from the CUDA package.

Arrays go in and come out as numpy arrays; 16-bit floats travel as their raw
``uint16`` bit patterns so the oracle decodes them itself.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

F32, F16, BF16, I8, I4 = 0, 1, 2, 3, 4

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` (gcc, fp64, OpenMP).

    ``-ffp-contract=off`` keeps every fp32 step of the int8 quantizer a
    single IEEE operation, as the quantizer's definition requires.
    """
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        I64 = ctypes.c_int64
        D = ctypes.c_double
        lib.orc_half_to_double.argtypes = [ctypes.c_uint16]
        lib.orc_half_to_double.restype = D
        lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_to_double.restype = D
        lib.orc_float_to_half_rne.argtypes = [ctypes.c_float]
        lib.orc_float_to_half_rne.restype = ctypes.c_uint16
        lib.orc_slot_of.argtypes = [P, I, I64]
        lib.orc_slot_of.restype = I64
        lib.orc_slot_mapping.argtypes = [P, I, I, I, P, P, P]
        lib.orc_slot_mapping.restype = None
        lib.orc_append.argtypes = [P, P, I, P, I, I, I, I, P, P]
        lib.orc_append.restype = None
        lib.orc_block_copy.argtypes = [P, I, I, I, I, P, P, I]
        lib.orc_block_copy.restype = None
        lib.orc_quantize_row_q8.argtypes = [P, I, P, P]
        lib.orc_quantize_row_q8.restype = None
        lib.orc_append_q8.argtypes = [P, P, I, P, I, I, I, I, P, P, P, P]
        lib.orc_append_q8.restype = None
        lib.orc_quantize_row_q4.argtypes = [P, I, P, P]
        lib.orc_quantize_row_q4.restype = None
        lib.orc_pack_q4.argtypes = [P, I, P]
        lib.orc_pack_q4.restype = None
        lib.orc_append_q4.argtypes = [P, P, I, P, I, I, I, I, P, P, P, P]
        lib.orc_append_q4.restype = None
        lib.orc_gather.argtypes = [P, P, I, P, I, I, I, I, I, P]
        lib.orc_gather.restype = None
        lib.orc_attend_rows.argtypes = [P, P, P, I, I, D, P, P]
        lib.orc_attend_rows.restype = None
        lib.orc_paged_decode_attention.argtypes = [P, I, I, P, P, P, P, I, I, I, I, I, P, I, P,
                                                   I, D, P, I]
        lib.orc_paged_decode_attention.restype = I
        lib.orc_paged_decode_attention_window.argtypes = [P, I, I, P, P, P, P, I, I, I, I, I, P,
                                                          I, P, I, I, D, P, I]
        lib.orc_paged_decode_attention_window.restype = I
        lib.orc_paged_prefill_attention.argtypes = [P, I, I, P, P, I, I, I, I, I, P, I, P, P, I,
                                                    D, P, I]
        lib.orc_paged_prefill_attention.restype = I
        lib.orc_max_threads.argtypes = []
        lib.orc_max_threads.restype = I
        lib.orc_kv_bytes_per_token.argtypes = [I64, I64, I64, I64]
        lib.orc_kv_bytes_per_token.restype = I64
        lib.orc_toy_generation.argtypes = [P, I, I, I, I, P, P, P, I, P, P, P, P]
        lib.orc_toy_generation.restype = None
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


_NP_OF = {F32: np.float32, F16: np.uint16, BF16: np.uint16, I8: np.int8, I4: np.uint8}


# ---------------------------------------------------------------- formats
def half_to_double(bits: int) -> float:
    return _load().orc_half_to_double(int(bits) & 0xFFFF)


def bf16_to_double(bits: int) -> float:
    return _load().orc_bf16_to_double(int(bits) & 0xFFFF)


def float_to_half_rne(x: float) -> int:
    return int(_load().orc_float_to_half_rne(float(np.float32(x))))


def decode(bits: np.ndarray, dtype: int) -> np.ndarray:
    """Decode a raw array of the given storage type to fp64, element by element."""
    lib = _load()
    flat = np.asarray(bits).reshape(-1)
    if dtype == F32:
        return flat.astype(np.float32).astype(np.float64).reshape(np.shape(bits))
    if dtype == I8:
        return flat.astype(np.int8).astype(np.float64).reshape(np.shape(bits))
    fn = lib.orc_half_to_double if dtype == F16 else lib.orc_bf16_to_double
    out = np.empty(flat.size, np.float64)
    for i, b in enumerate(flat.tolist()):
        out[i] = fn(b)
    return out.reshape(np.shape(bits))


# ---------------------------------------------------------------- slots / append
def slot_of(block_table_row: np.ndarray, block_size: int, pos: int) -> int:
    row = _c(block_table_row, np.int32)
    return int(_load().orc_slot_of(_ptr(row), block_size, pos))


def slot_mapping(block_tables, block_size, start, n_new):
    bt = _c(block_tables, np.int32)
    start = _c(start, np.int32)
    n_new = _c(n_new, np.int32)
    out = np.empty(int(n_new.sum()), np.int32)
    _load().orc_slot_mapping(_ptr(bt), bt.shape[1], block_size, bt.shape[0], _ptr(start),
                             _ptr(n_new), _ptr(out))
    return out


def append(k_new, v_new, dtype, slots, block_size, k_cache, v_cache):
    """Bit-copy append into numpy caches (modified in place)."""
    k_new = _c(k_new, _NP_OF[dtype])
    v_new = _c(v_new, _NP_OF[dtype])
    slots = _c(slots, np.int32)
    T, H, D = k_new.shape
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    _load().orc_append(_ptr(k_new), _ptr(v_new), dtype, _ptr(slots), T, H, D, block_size,
                       _ptr(k_cache), _ptr(v_cache))


def block_copy(src, dst, block_size, k_cache, v_cache, k_scales=None, v_scales=None):
    """Copy-on-write copy of blocks src[j] -> dst[j] in numpy caches (in place)."""
    src = _c(src, np.int32)
    dst = _c(dst, np.int32)
    NB, H, bs, D = k_cache.shape
    assert bs == block_size
    for a in (k_cache, v_cache):
        assert a.flags.c_contiguous
        _load().orc_block_copy(_ptr(a), a.dtype.itemsize, H, bs, D, _ptr(src), _ptr(dst), src.size)
    for a in (k_scales, v_scales):
        if a is not None:
            assert a.flags.c_contiguous and a.shape == (NB, H, bs)
            _load().orc_block_copy(_ptr(a), a.dtype.itemsize, H, bs, 1, _ptr(src), _ptr(dst),
                                   src.size)


def quantize_row_q8(x):
    x = _c(x, np.float32)
    codes = np.empty(x.size, np.int8)
    sb = np.zeros(1, np.uint16)
    _load().orc_quantize_row_q8(_ptr(x), x.size, _ptr(codes), _ptr(sb))
    return codes, int(sb[0])


def append_q8(k_new, v_new, in_dtype, slots, block_size, k_cache, v_cache, k_scales, v_scales):
    k_new = _c(k_new, _NP_OF[in_dtype])
    v_new = _c(v_new, _NP_OF[in_dtype])
    slots = _c(slots, np.int32)
    T, H, D = k_new.shape
    for a, t in ((k_cache, np.int8), (v_cache, np.int8), (k_scales, np.uint16), (v_scales, np.uint16)):
        assert a.dtype == t and a.flags.c_contiguous
    _load().orc_append_q8(_ptr(k_new), _ptr(v_new), in_dtype, _ptr(slots), T, H, D, block_size,
                          _ptr(k_cache), _ptr(v_cache), _ptr(k_scales), _ptr(v_scales))


def quantize_row_q4(x):
    """4-bit codes (one int8 per element, -7..7) and the fp16 scale bits."""
    x = _c(x, np.float32)
    codes = np.empty(x.size, np.int8)
    sb = np.zeros(1, np.uint16)
    _load().orc_quantize_row_q4(_ptr(x), x.size, _ptr(codes), _ptr(sb))
    return codes, int(sb[0])


def pack_q4(codes):
    codes = _c(codes, np.int8)
    out = np.empty(codes.size // 2, np.uint8)
    _load().orc_pack_q4(_ptr(codes), codes.size, _ptr(out))
    return out


def append_q4(k_new, v_new, in_dtype, slots, block_size, k_cache, v_cache, k_scales, v_scales):
    """Quantize-on-append to a 4-bit cache (uint8 [NB, H, bs, D/2], two codes a byte)."""
    k_new = _c(k_new, _NP_OF[in_dtype])
    v_new = _c(v_new, _NP_OF[in_dtype])
    slots = _c(slots, np.int32)
    T, H, D = k_new.shape
    for a, t in ((k_cache, np.uint8), (v_cache, np.uint8), (k_scales, np.uint16),
                 (v_scales, np.uint16)):
        assert a.dtype == t and a.flags.c_contiguous
    assert k_cache.shape[3] * 2 == D
    _load().orc_append_q4(_ptr(k_new), _ptr(v_new), in_dtype, _ptr(slots), T, H, D, block_size,
                          _ptr(k_cache), _ptr(v_cache), _ptr(k_scales), _ptr(v_scales))


# ---------------------------------------------------------------- attention
def gather(cache, scales, dtype, block_table_row, seq_len, head, block_size):
    cache = np.ascontiguousarray(cache)
    NB, H, bs, D = cache.shape
    if dtype == I4:
        D *= 2                      # two codes per byte
    row = _c(block_table_row, np.int32)
    out = np.empty((seq_len, D), np.float64)
    sc = None if scales is None else _c(scales, np.uint16)
    _load().orc_gather(_ptr(cache), _ptr(sc), dtype, _ptr(row), seq_len, head, H, D, block_size,
                       _ptr(out))
    return out


def attend_rows(q, krows, vrows, scale):
    q = _c(q, np.float64)
    krows = _c(krows, np.float64)
    vrows = _c(vrows, np.float64)
    L = krows.shape[0]
    D = q.size
    out = np.empty(D, np.float64)
    sc = np.empty(max(L, 1), np.float64)
    _load().orc_attend_rows(_ptr(q), _ptr(krows), _ptr(vrows), L, D, float(scale), _ptr(out),
                            _ptr(sc))
    return out


def paged_decode_attention(q, q_dtype, k_cache, v_cache, kv_dtype, block_tables, seq_lens, scale,
                           k_scales=None, v_scales=None, nthreads=0, window=0):
    """fp64 attention of every (sequence, query head) against its cached rows
    (with window > 0: against its last min(window, L) rows only).

    q: [B, Hq, D] raw (fp32 or uint16 bits); caches [NB, Hkv, bs, D] raw;
    returns out [B, Hq, D] float64.
    """
    q = _c(q, _NP_OF[q_dtype])
    k_cache = np.ascontiguousarray(k_cache)
    v_cache = np.ascontiguousarray(v_cache)
    NB, Hkv, bs, D = k_cache.shape
    if kv_dtype == I4:
        D *= 2                      # two codes per byte
    B, Hq, Dq = q.shape
    assert Dq == D
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    ks = None if k_scales is None else _c(k_scales, np.uint16)
    vs = None if v_scales is None else _c(v_scales, np.uint16)
    out = np.zeros((B, Hq, D), np.float64)
    if window:
        rc = _load().orc_paged_decode_attention_window(
            _ptr(q), q_dtype, Hq, _ptr(k_cache), _ptr(v_cache), _ptr(ks), _ptr(vs), kv_dtype, NB,
            Hkv, D, bs, _ptr(bt), bt.shape[1], _ptr(sl), B, int(window), float(scale), _ptr(out),
            int(nthreads))
    else:
        rc = _load().orc_paged_decode_attention(_ptr(q), q_dtype, Hq, _ptr(k_cache),
                                                _ptr(v_cache), _ptr(ks), _ptr(vs), kv_dtype, NB,
                                                Hkv, D, bs, _ptr(bt), bt.shape[1], _ptr(sl), B,
                                                float(scale), _ptr(out), int(nthreads))
    if rc != 0:
        raise ValueError("oracle: block table entry or sequence length out of range")
    return out


def paged_prefill_attention(q, q_dtype, k_cache, v_cache, kv_dtype, block_tables, q_start,
                            seq_lens, scale, nthreads=0):
    """fp64 causal attention of the new tokens of every sequence over its cached rows.

    q: [T, Hq, D] raw, sequence-major (sequence b's tokens at q_start[b] ..
    q_start[b+1]-1, the last ones of its seq_lens[b] cached rows); returns
    out [T, Hq, D] float64.
    """
    q = _c(q, _NP_OF[q_dtype])
    k_cache = np.ascontiguousarray(k_cache)
    v_cache = np.ascontiguousarray(v_cache)
    NB, Hkv, bs, D = k_cache.shape
    T, Hq, Dq = q.shape
    assert Dq == D
    bt = _c(block_tables, np.int32)
    qs = _c(q_start, np.int32)
    sl = _c(seq_lens, np.int32)
    B = sl.size
    assert qs.size == B + 1 and qs[-1] == T
    out = np.zeros((T, Hq, D), np.float64)
    rc = _load().orc_paged_prefill_attention(_ptr(q), q_dtype, Hq, _ptr(k_cache), _ptr(v_cache),
                                             kv_dtype, NB, Hkv, D, bs, _ptr(bt), bt.shape[1],
                                             _ptr(qs), _ptr(sl), B, float(scale), _ptr(out),
                                             int(nthreads))
    if rc != 0:
        raise ValueError("oracle: block table entry or length out of range")
    return out


def max_threads() -> int:
    return int(_load().orc_max_threads())


def kv_bytes_per_token(n_layers, n_kv_heads, head_dim, bytes_per_number) -> int:
    return int(_load().orc_kv_bytes_per_token(n_layers, n_kv_heads, head_dim, bytes_per_number))


def toy_generation(x, prompt_len, decode_steps, Wq, Wk, Wv, block_size):
    """Run the cached and uncached lanes of the toy loop; see ``oracle.c``."""
    x = _c(x, np.float64)
    Wq = _c(Wq, np.float64)
    Wk = _c(Wk, np.float64)
    Wv = _c(Wv, np.float64)
    D, E = Wq.shape
    steps = decode_steps + 1
    on = np.empty((steps, D), np.float64)
    oc = np.empty((steps, D), np.float64)
    rn = np.empty(steps, np.int64)
    rc = np.empty(steps, np.int64)
    _load().orc_toy_generation(_ptr(x), prompt_len, decode_steps, E, D, _ptr(Wq), _ptr(Wk),
                               _ptr(Wv), block_size, _ptr(on), _ptr(oc), _ptr(rn), _ptr(rc))
    return on, oc, rn, rc
