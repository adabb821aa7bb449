"""Seeded synthetic inputs for paged decode attention.

This module only draws inputs: sequence lengths, block placement in the pool,
and the raw K / V / q values.  It holds none of the attention, slot-mapping
or quantization arithmetic, so both the CUDA path and the CPU oracle can
consume its arrays.  It imports numpy only.

The five workloads mirror the shapes the KV cache pages use for their memory
figures (GPT-2 small, Llama-3-8B, Llama-2-70B; KV cache visualization page,
"How much memory") plus a tiny case sized like its canvas (block size 4,
"PagedAttention: the cache in blocks") and an int8-cache case ("Quantized KV
cache" on "KV cache: the engine behind fast LLM inference").

Dtype codes match the library's: 0 f32, 1 f16, 2 bf16, 3 int8.  16-bit
values travel as raw uint16 bit patterns.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

F32, F16, BF16, I8, I4 = 0, 1, 2, 3, 4


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    batch: int
    kv_dtype: int          # cache element type
    q_dtype: int
    src_dtype: int         # type of the generated K/V rows (f16 for the int8 cache)
    seed: int
    lengths: str           # "tiny", "fixed", "uniform", "loguniform"
    len_lo: int
    len_hi: int
    decode_steps: int      # appended tokens after the prefix
    shared_prefix_tokens: int = 0   # > 0: half the batch shares this many leading tokens
    outlier_p: float = 0.0          # probability of an outlier element
    outlier_scale: float = 1.0
    pool_slack: float = 0.10        # extra free blocks in the pool

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads


WORKLOADS = {
    # 4 q / 2 KV heads, d 64, block size 4, 16 blocks; sequences end at 7 and 3
    # tokens after one decode step (a 3-token prompt plus 4 decode steps, and a
    # bare 3-token prompt).
    "tiny": Workload("tiny", 4, 2, 64, 4, 2, F32, F32, F32, 0, "tiny", 0, 0, 1),
    # GPT-2-small-shaped MHA layer: 12 = 12 heads, d 64, bs 16, 64 sequences
    # with lengths uniform in [1, 2048], fp16.
    "gpt2": Workload("gpt2", 12, 12, 64, 16, 64, F16, F16, F16, 1, "uniform", 1, 2048, 1),
    # Llama-3-8B-shaped GQA layer: 32 q / 8 KV heads, d 128, bs 16, 16
    # sequences of 4096 tokens, bf16, then 64 decode steps.
    "llama3_8b": Workload("llama3_8b", 32, 8, 128, 16, 16, BF16, BF16, BF16, 2, "fixed", 4096,
                          4096, 64),
    # Llama-2-70B-shaped GQA layer: 64 q / 8 KV heads, d 128, bs 16, 32
    # sequences with log-uniform lengths in [16, 32768], fp16; half share a
    # 1024-token prefix.
    "llama2_70b": Workload("llama2_70b", 64, 8, 128, 16, 32, F16, F16, F16, 3, "loguniform", 16,
                           32768, 1, shared_prefix_tokens=1024),
    # int8 cache on the Llama-3-8B shape: 128 sequences, lengths uniform in
    # [512, 8192], K/V drawn in fp16 with 1% outliers x8, fp16 q.
    "int8": Workload("int8", 32, 8, 128, 16, 128, I8, F16, F16, 4, "uniform", 512, 8192, 1,
                     outlier_p=0.01, outlier_scale=8.0),
    # 4-bit cache on the same shape (a variant beyond the five configurations
    # above): 64 sequences, lengths uniform in [512, 8192], fp16 rows with 1%
    # outliers x8, fp16 q.
    "int4": Workload("int4", 32, 8, 128, 16, 64, I4, F16, F16, 5, "uniform", 512, 8192, 1,
                     outlier_p=0.01, outlier_scale=8.0),
}


@dataclasses.dataclass
class Inputs:
    workload: Workload
    num_blocks: int
    final_lens: np.ndarray        # [B] tokens cached after all decode steps
    prefix_lens: np.ndarray       # [B] tokens cached before the decode steps
    block_tables: np.ndarray      # [B, max_blocks] int32, covers final_lens
    hist_k: np.ndarray            # [sum(prefix_lens), Hkv, D] raw, sequence-major
    hist_v: np.ndarray
    hist_offsets: np.ndarray      # [B+1] row offsets into hist_*
    hist_write: np.ndarray        # [sum(prefix_lens)] bool: row is written by this sequence
    step_k: np.ndarray            # [steps, B, Hkv, D] raw
    step_v: np.ndarray
    step_q: np.ndarray            # [steps, B, Hq, D] raw (q of each decode step)
    sharers: np.ndarray           # [B] bool: sequence uses the shared prefix blocks
    idle: np.ndarray              # [B] bool: empty sequence, no tokens appended

    def lens_after_step(self, s: int) -> np.ndarray:
        """Cached tokens of every sequence after decode step s (0-based)."""
        return np.where(self.idle, 0, self.prefix_lens + s + 1).astype(np.int32)

    @property
    def max_blocks_per_seq(self) -> int:
        return self.block_tables.shape[1]


def _blocks_for(tokens: int, block_size: int) -> int:
    # number of blocks a table must list to cover `tokens` positions
    return -(-int(tokens) // block_size)


def _values(rng: np.random.Generator, shape, dtype: int, outlier_p=0.0, outlier_scale=1.0):
    """N(0,1) draws stored as dtype (f32 array, or uint16 bits for f16/bf16)."""
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if outlier_p > 0.0:
        mask = rng.random(size=shape, dtype=np.float32) < outlier_p
        x = np.where(mask, x * np.float32(outlier_scale), x)
    if dtype == F32:
        return x
    if dtype == F16:
        return x.astype(np.float16).view(np.uint16)
    if dtype == BF16:
        # bfloat16 by truncation of the fp32 pattern (a valid N(0,1)-like draw)
        return (x.view(np.uint32) >> 16).astype(np.uint16)
    raise ValueError("no value generator for dtype %d" % dtype)


def _lengths(rng: np.random.Generator, wl: Workload) -> np.ndarray:
    if wl.lengths == "tiny":
        return np.array([7, 3], np.int64)
    if wl.lengths == "fixed":
        return np.full(wl.batch, wl.len_lo + wl.decode_steps, np.int64)
    if wl.lengths == "uniform":
        return rng.integers(wl.len_lo, wl.len_hi + 1, size=wl.batch).astype(np.int64)
    if wl.lengths == "loguniform":
        u = rng.uniform(math.log(wl.len_lo), math.log(wl.len_hi), size=wl.batch)
        return np.clip(np.round(np.exp(u)), wl.len_lo, wl.len_hi).astype(np.int64)
    raise ValueError(wl.lengths)


def make_inputs(wl: Workload | str, lengths=None, values=True) -> Inputs:
    """Draw the inputs of a workload.

    lengths: explicit final lengths (one per sequence) instead of the
    workload's recipe; e.g. (8, 4) for the tiny workload is the reading in
    which 7 and 3 are the lengths before the decode step.
    values: False skips the K/V rows (lengths, tables and q only), for
    timing runs that fill the caches on the device.
    """
    if isinstance(wl, str):
        wl = WORKLOADS[wl]
    rng = np.random.default_rng(wl.seed)
    final = _lengths(rng, wl)
    if lengths is not None:
        final = np.asarray(lengths, np.int64)
        wl = dataclasses.replace(wl, batch=len(final))
    B, Hq, Hkv, D, bs = wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.block_size
    steps = wl.decode_steps

    sharers = np.zeros(B, bool)
    P = wl.shared_prefix_tokens
    if P > 0:
        who = rng.permutation(B)[: B // 2]
        sharers[who] = True
        # a sharer's decode step must land past the shared blocks
        final = np.where(sharers, np.maximum(final, P + steps), final)
    # An empty sequence (final length 0) takes no part in the decode steps.
    idle = final == 0
    prefix = np.where(idle, 0, final - steps)
    if np.any(prefix < 0):
        raise ValueError("lengths shorter than the decode steps")

    # ---- block placement
    nblk = np.array([_blocks_for(L, bs) for L in final], np.int64)
    shared_blocks = P // bs if P > 0 else 0
    private = nblk - np.where(sharers, shared_blocks, 0)
    unique = int(private.sum()) + shared_blocks
    if wl.name == "tiny" and unique <= 16:
        num_blocks = 16
    else:
        num_blocks = max(1, int(math.ceil(unique * (1.0 + wl.pool_slack))))
    perm = rng.permutation(num_blocks).astype(np.int32)
    max_blocks = int(nblk.max()) if B else 1
    tables = np.zeros((B, max(max_blocks, 1)), np.int32)
    cursor = 0
    shared_ids = perm[cursor: cursor + shared_blocks]
    cursor += shared_blocks
    for b in range(B):
        k = 0
        if sharers[b]:
            tables[b, :shared_blocks] = shared_ids
            k = shared_blocks
        n = int(nblk[b]) - k
        tables[b, k: k + n] = perm[cursor: cursor + n]
        cursor += n

    # ---- values: history rows, per-step rows, per-step q
    offs = np.zeros(B + 1, np.int64)
    offs[1:] = np.cumsum(prefix)
    total = int(offs[-1])
    if not values:
        sq = _values(rng, (steps, B, Hq, D), wl.q_dtype)
        empty = np.zeros((0, Hkv, D), np.float32)
        return Inputs(wl, num_blocks, final.astype(np.int32), prefix.astype(np.int32), tables,
                      empty, empty, offs, np.ones(total, bool), empty, empty, sq, sharers, idle)
    hk = _values(rng, (total, Hkv, D), wl.src_dtype, wl.outlier_p, wl.outlier_scale)
    hv = _values(rng, (total, Hkv, D), wl.src_dtype, wl.outlier_p, wl.outlier_scale)
    write = np.ones(total, bool)
    if P > 0:
        first = int(np.argmax(sharers))
        src = slice(int(offs[first]), int(offs[first]) + P)
        for b in range(B):
            if sharers[b] and b != first:
                dst = slice(int(offs[b]), int(offs[b]) + P)
                hk[dst] = hk[src]
                hv[dst] = hv[src]
                write[dst] = False            # the blocks already hold these rows
    sk = _values(rng, (steps, B, Hkv, D), wl.src_dtype, wl.outlier_p, wl.outlier_scale)
    sv = _values(rng, (steps, B, Hkv, D), wl.src_dtype, wl.outlier_p, wl.outlier_scale)
    sq = _values(rng, (steps, B, Hq, D), wl.q_dtype)
    return Inputs(wl, num_blocks, final.astype(np.int32), prefix.astype(np.int32), tables, hk, hv,
                  offs, write, sk, sv, sq, sharers, idle)


def positions_of_history(inp: Inputs) -> tuple[np.ndarray, np.ndarray]:
    """(sequence index, position) of every history row, sequence-major."""
    B = inp.workload.batch
    seq = np.repeat(np.arange(B, dtype=np.int32), inp.prefix_lens)
    pos = np.concatenate([np.arange(L, dtype=np.int32) for L in inp.prefix_lens]) if B else \
        np.zeros(0, np.int32)
    return seq, pos
