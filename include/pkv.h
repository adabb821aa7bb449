/*
 * pkv.h — C ABI of libpkv: single-token decode attention over a paged KV
 * cache, for NVIDIA GB300 (sm_103a).
 *
 * Sources of the operations (three web pages on the KV cache):
 *   [NOTES] "KV cache: the engine behind fast LLM inference"
 *           (curiosity-9m6.pages.dev/notes/0043)
 *   [VIS]   KV cache visualization (cuuduongthancong.com/~galles/visualization/KVCache.html)
 *   [GUIDE] jovanaeducation.com/guides/l-is-2
 *
 * Conventions shared by every call
 * --------------------------------
 * Shapes.  B = batch (sequences), Hq = query heads, Hkv = KV heads,
 * G = Hq / Hkv (query heads per KV head; consecutive query heads
 * h = kvh*G .. kvh*G+G-1 share KV head kvh), D = head_dim, bs = block_size
 * (tokens per block), NB = number of blocks in the pool.
 *
 * Layouts (all row-major, all device buffers owned by the caller):
 *   k_cache, v_cache   [NB][Hkv][bs][D]  element type = the pool's kv_dtype.
 *                      Each (block, KV head) tile of bs*D elements is contiguous.
 *   k_scales, v_scales [NB][Hkv][bs]     fp16, int8 pools only (one scale per
 *                      cached token per KV head); NULL otherwise.
 *   q                  [B][Hq][D]        q_dtype.
 *   out                [B][Hq][D]        fp32.
 *   block_tables       [B][max_blocks_per_seq] int32: entry j of row b is the
 *                      physical block that holds tokens j*bs .. j*bs+bs-1 of
 *                      sequence b ([VIS] "PagedAttention: the cache in blocks").
 *   seq_lens           [B] int32: tokens cached for each sequence, counting the
 *                      token appended in this step.
 *   slot_mapping       [T] int32: cache slot of each new token,
 *                      slot = block * bs + offset; slot < 0 marks a padding
 *                      token that is skipped.
 * Device pointers must be 16-byte aligned.
 *
 * Errors.  Every call returns a pkv_status.  Argument and shape errors are
 * reported synchronously, before anything is launched.  Device calls are
 * asynchronous on the given stream and return the launch status; bad
 * indices met on the device (slot or block id outside the pool, a sequence
 * length beyond its block table) are recorded in the pool's device error
 * word, the offending access is skipped (nothing traps), and
 * pkv_check_error() reports them.
 *
 * Threads.  A pool's host bookkeeping (alloc/share/free/reserve) is not
 * thread safe; serialise those calls per pool.  Device calls may be issued
 * from any thread.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without pulling in the CUDA headers. */
typedef struct CUstream_st *pkv_stream_t;

typedef enum {
    PKV_F32 = 0,
    PKV_F16 = 1,
    PKV_BF16 = 2,
    PKV_I8 = 3,
    PKV_I4 = 4
} pkv_dtype;

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID = -1,     /* bad argument, shape or pointer alignment            */
    PKV_ERR_NO_BLOCKS = -2,   /* the pool has too few free blocks                    */
    PKV_ERR_CUDA = -3,        /* a CUDA runtime call failed (or no device)           */
    PKV_ERR_UNSUPPORTED = -4, /* valid but not a compiled shape / dtype combination  */
    PKV_ERR_BAD_INDEX = -5,   /* device saw a slot / block id / length out of range  */
    PKV_ERR_TIMEOUT = -6      /* a bounded device wait gave up                       */
} pkv_status;

typedef struct pkv_pool pkv_pool; /* opaque; host-side bookkeeping only */

/* Human-readable name of a status code (static string). */
const char *pkv_status_string(int status);

/* ====================================================================== */
/* Block pool (host).                                                      */
/* ====================================================================== */

/*
 * kv_block_pool_init — describe one shared pool of fixed-size cache blocks.
 * [VIS] "PagedAttention: the cache in blocks" (every request's rows live in
 * equal-size blocks that all come out of a single pool); [GUIDE] "Paging:
 * borrow the trick operating systems already use".
 *
 *   out          receives the new pool (owned by the caller; free with
 *                kv_block_pool_destroy).
 *   num_blocks   NB >= 1; NB * block_size must be < 2^31.
 *   block_size   power of two, 1..256 (>= 8 for int8 pools).
 *   num_kv_heads Hkv >= 1.
 *   head_dim     64 or 128.
 *   kv_dtype     element type of the cache: F32, F16, BF16, or I8 (int8 codes
 *                with per-token-per-head fp16 scales).
 *
 * The pool keeps a free list (all NB blocks free at start), one reference
 * count per block, and a 4-byte device error word on the current device.  It
 * does not own the cache memory: the caller allocates k_cache / v_cache of
 * kv_cache_bytes() each (and k_scales / v_scales of kv_scales_bytes() for
 * int8).  If no CUDA device is usable the pool is still created for its host
 * calls, and every device call on it returns PKV_ERR_CUDA.
 * Returns PKV_OK, PKV_ERR_INVALID or PKV_ERR_UNSUPPORTED.
 */
int kv_block_pool_init(pkv_pool **out, int num_blocks, int block_size, int num_kv_heads,
                       int head_dim, pkv_dtype kv_dtype);

/* Free the pool's host state and its device error word.  NULL is a no-op. */
void kv_block_pool_destroy(pkv_pool *pool);

/* Bytes of one of k_cache / v_cache: NB * Hkv * bs * D * sizeof(kv_dtype). */
size_t kv_cache_bytes(const pkv_pool *pool);

/* Bytes of one of k_scales / v_scales: NB * Hkv * bs * 2 for int8 pools, else 0. */
size_t kv_scales_bytes(const pkv_pool *pool);

/* Number of blocks currently on the free list. */
int kv_num_free_blocks(const pkv_pool *pool);

/* Reference count of block id (0 = free), or PKV_ERR_INVALID for a bad id. */
int kv_block_refcount(const pkv_pool *pool, int32_t id);

/*
 * kv_block_alloc — take n blocks off the free list, reference count 1 each,
 * ids written to out_ids[0..n).  A sequence takes blocks as it needs them
 * and gives them back when it is done ([GUIDE] "Paging…").
 * All-or-nothing: PKV_ERR_NO_BLOCKS (and no change) if fewer than n are free.
 */
int kv_block_alloc(pkv_pool *pool, int n, int32_t *out_ids);

/*
 * kv_block_share — add one reference to each of ids[0..n), so that another
 * request's table may list these blocks too ([VIS] "PagedAttention: the cache in
 * blocks": sequences that begin with the same prompt tokens can reference a
 * single stored copy of those tokens' blocks).
 * All-or-nothing: PKV_ERR_INVALID if any id is out of range or free.
 */
int kv_block_share(pkv_pool *pool, const int32_t *ids, int n);

/*
 * kv_block_free — drop one reference from each of ids[0..n); a block whose
 * count reaches 0 returns to the free list.  All-or-nothing: PKV_ERR_INVALID
 * (no change) if any id is out of range or already free, counting repeats.
 */
int kv_block_free(pkv_pool *pool, const int32_t *ids, int n);

/*
 * kv_reserve_slots — host bookkeeping of one append step (prefill or decode).
 * For each sequence b with seq_lens[b] tokens already cached and num_new[b]
 * new tokens (num_new == NULL means 1 each), allocate a new block whenever a
 * new token's position starts a block (allocation on demand, [VIS]
 * "PagedAttention: the cache in blocks": a sequence gains a block only when
 * its tokens need one, so no more than its last block is incomplete),
 * record it in the host array block_tables ([B][max_blocks_per_seq],
 * updated in place), and write the slot of every
 * new token to slot_mapping (sequence-major, sum(num_new) entries).
 * All-or-nothing: PKV_ERR_NO_BLOCKS if the pool cannot cover the step,
 * PKV_ERR_INVALID if a table row would overflow max_blocks_per_seq.
 * seq_lens itself is not modified.
 */
int kv_reserve_slots(pkv_pool *pool, int batch, const int32_t *seq_lens, const int32_t *num_new,
                     int32_t *block_tables, int max_blocks_per_seq, int32_t *slot_mapping);

/*
 * kv_reserve_slots_cow — kv_reserve_slots for tables that may point at shared
 * blocks.  [VIS] "PagedAttention: the cache in blocks": sequences that start
 * with the same tokens may reference one physical copy of those blocks, and a
 * private copy is made only at the moment a sharer must modify one.  The only
 * existing block an append step writes into is a
 * sequence's last, partly filled one (at position seq_lens[b] when
 * seq_lens[b] % bs != 0 and num_new[b] > 0); if its reference count is above
 * one, the sequence gets a private copy first: a fresh block is allocated,
 * the pair (old id, new id) is written to copy_src[i], copy_dst[i], one
 * reference of the old block is dropped and the table entry is replaced.
 * Sequences are handled in order, so when every holder of a shared block
 * appends in one step, all but the last one to be handled get copies and
 * that last one writes in place.  At most `batch` pairs; *num_copies
 * receives their number.  The caller must run kv_block_copy on the pairs
 * before the kv_append of this step.  Slots and new blocks are then handled
 * as in kv_reserve_slots.
 * All-or-nothing: PKV_ERR_NO_BLOCKS if the pool cannot cover the new blocks
 * and the copies; PKV_ERR_INVALID for a table row that would overflow or a
 * written entry that is out of range or free.
 */
int kv_reserve_slots_cow(pkv_pool *pool, int batch, const int32_t *seq_lens,
                         const int32_t *num_new, int32_t *block_tables, int max_blocks_per_seq,
                         int32_t *slot_mapping, int32_t *copy_src, int32_t *copy_dst,
                         int *num_copies);

/*
 * kv_slot_mapping — pure host computation of slots from existing block
 * tables: token j of sequence b sits at position start[b] + j, in logical
 * block p / bs at offset p % bs, so its slot is
 * block_tables[b][p / bs] * bs + p % bs.  num_new == NULL means 1 each.
 * Returns PKV_ERR_INVALID if a position falls outside its table row.
 */
int kv_slot_mapping(const int32_t *block_tables, int max_blocks_per_seq, int block_size,
                    int batch, const int32_t *start, const int32_t *num_new,
                    int32_t *slot_mapping);

/* ====================================================================== */
/* Device calls.                                                           */
/* ====================================================================== */

/*
 * kv_append — write the new tokens' K and V rows into the cache.
 * [NOTES] "What happens at each decoding step", step 4; [GUIDE] "How the
 * cache turns the loop cheap" (only the new token's key and value are
 * computed, then stored).  With num_tokens = a whole prompt it is the bulk
 * write of prefill.
 *
 *   k_new, v_new  device [T][Hkv][D], element type in_dtype.
 *   slot_mapping  device [T] int32 (see conventions; < 0 = skip).
 *   k_cache, v_cache  device caches of the pool's layout.
 *   k_scales, v_scales  device fp16 [NB][Hkv][bs] for int8 pools, else NULL.
 *
 * fp pools: in_dtype must equal the pool's kv_dtype; rows are copied bit for
 * bit.  int8 pools ([NOTES] "Quantized KV cache"): in_dtype F16, BF16 or F32;
 * each (token, head) row x of D values is quantized in fp32 as
 *   amax = max|x_i|, s = fp16_round_nearest_even(amax / 127),
 *   code_i = clamp(round_half_even(x_i / s), -127, 127)   (codes 0 if s == 0)
 * and s is stored as that token's scale.  Inputs must be finite with
 * |x| <= 65504.  A slot outside [0, NB*bs) sets PKV_ERR_BAD_INDEX in the
 * error word and that token is skipped.  num_tokens == 0 is a no-op.
 */
int kv_append(const pkv_pool *pool, const void *k_new, const void *v_new, pkv_dtype in_dtype,
              const int32_t *slot_mapping, int num_tokens, void *k_cache, void *v_cache,
              void *k_scales, void *v_scales, pkv_stream_t stream);

/*
 * kv_block_copy — the copy half of copy-on-write ([VIS] "PagedAttention: the
 * cache in blocks"): for i < n, every cached K and V row of block src[i] (all
 * KV heads; and the fp16 scales for int8 pools) is copied bit for bit to
 * block dst[i].
 *
 *   src, dst   device int32 [n] block ids (as kv_reserve_slots_cow writes
 *              them).  The dst blocks must be distinct and none may be a src
 *              block of the same call (overlapping pairs give an undefined
 *              result).
 *   k_cache, v_cache, k_scales, v_scales  as for kv_append.
 *
 * An id outside [0, NB) sets PKV_ERR_BAD_INDEX in the error word and that
 * pair is skipped.  n == 0 is a no-op.
 */
int kv_block_copy(const pkv_pool *pool, const int32_t *src, const int32_t *dst, int n,
                  void *k_cache, void *v_cache, void *k_scales, void *v_scales,
                  pkv_stream_t stream);

/*
 * paged_decode_workspace_bytes — size of the scratch buffer that
 * paged_decode_attention needs for a batch of `batch` sequences and
 * num_q_heads query heads on the pool's device.  The workspace holds
 * per-piece partial softmax states and one counter per (sequence, KV head).
 * Returns 0 for invalid arguments.
 */
size_t paged_decode_workspace_bytes(const pkv_pool *pool, int batch, int num_q_heads);

/*
 * paged_decode_attention — one decode step of attention for a batch.
 * [NOTES] "Concept" and step 3 of "What happens at each decoding step": for
 * every sequence b and query head h, with kvh = h / G,
 *   out[b][h] = softmax(scale * q[b][h] . K_b^T) . V_b
 * over the seq_lens[b] cached rows K_b, V_b of KV head kvh, reached through
 * block_tables[b] ([VIS] "PagedAttention: the cache in blocks"; GQA sharing
 * from [VIS] "How much memory").  int8 pools dequantize each row as
 * code * scale.  scale is normally 1/sqrt(D).
 *
 *   q          device [B][Hq][D]; q_dtype = kv_dtype for fp pools, F16 or
 *              BF16 for int8 pools.
 *   num_q_heads  Hq, a multiple of Hkv with G in {1, 2, 4, 8}.
 *   block_tables, seq_lens  device int32 (see conventions).  A length of 0
 *              gives a zero output row; a length above
 *              max_blocks_per_seq * bs, or a block id outside [0, NB), sets
 *              PKV_ERR_BAD_INDEX and the sequence's output is unspecified.
 *   max_seq_len  an upper bound of seq_lens (only sizes the launch, so the
 *              host never waits for the device).
 *   out        device fp32 [B][Hq][D].
 *   workspace  device scratch of at least paged_decode_workspace_bytes();
 *              its counters must be zero before the first call (e.g. zeroed
 *              by the caller at allocation); every call leaves them zero.  A
 *              workspace must not be shared by calls that run concurrently.
 *              After a call that reported PKV_ERR_TIMEOUT, zero it again.
 *
 * Batch is limited to 4096 sequences per call (PKV_ERR_UNSUPPORTED beyond).
 * Split-K: the batch's K/V tiles are divided over the GPU's SMs in shares of
 * equal cost (each tile, and each (sequence, KV head) piece end, counted); a
 * sequence split across several CTAs is merged by the last CTA to finish it.
 * The result does not depend on timing.
 */
int paged_decode_attention(const pkv_pool *pool, const void *q, pkv_dtype q_dtype,
                           int num_q_heads, const void *k_cache, const void *v_cache,
                           const void *k_scales, const void *v_scales,
                           const int32_t *block_tables, int max_blocks_per_seq,
                           const int32_t *seq_lens, int batch, int max_seq_len, float scale,
                           float *out, void *workspace, size_t workspace_bytes,
                           pkv_stream_t stream);

/*
 * kv_prefix_groups — host: find the groups of sequences that share a prefix
 * of physical blocks ([VIS] "PagedAttention: the cache in blocks": sequences
 * that begin with the same prompt tokens can reference one stored copy of
 * those tokens' blocks).  Sequences with at least min_prefix_blocks * block
 * _size rows are grouped by their first table entry; a group of two or more
 * shares its members' longest common run of leading table entries, capped
 * at the shortest member's length: group_prefix[g] tokens (P).  block_tables
 * [B][max_blocks_per_seq] and seq_lens [B] are host arrays.  Outputs (host,
 * caller-allocated, batch entries each, group_start batch + 1):
 * group_start[g]..group_start[g+1] index group g's members in group_seqs
 * (ascending sequence order; the first member's table is the one read for
 * the prefix), group_prefix[g] = P, seq_prefix[b] = P of b's group or 0,
 * and *num_groups, *max_group_size, *max_prefix_len.  PKV_ERR_INVALID for a
 * null pointer, batch < 0, block_size < 1, min_prefix_blocks < 1 or a length
 * outside its table row.
 */
int kv_prefix_groups(const int32_t *block_tables, int max_blocks_per_seq, const int32_t *seq_lens,
                     int batch, int block_size, int min_prefix_blocks, int32_t *group_start,
                     int32_t *group_seqs, int32_t *group_prefix, int32_t *seq_prefix,
                     int *num_groups, int *max_group_size, int *max_prefix_len);

/*
 * paged_decode_cascade_workspace_bytes — bytes of the workspace of
 * paged_decode_attention_cascade: the decode workspace, then the prefix
 * partials for prefixes of up to max_prefix_len tokens (fp32, [chunks][batch]
 * [num_q_heads][head_dim + 4], at most 16 chunks of 128-key tiles; a merge
 * step leaves the merged prefix of every row in chunk 0).  0 on bad
 * arguments.
 */
size_t paged_decode_cascade_workspace_bytes(const pkv_pool *pool, int batch, int num_q_heads,
                                            int max_prefix_len);

/*
 * paged_decode_attention_cascade — paged_decode_attention for a batch in
 * which groups of sequences share the leading blocks of their tables ([VIS]
 * "PagedAttention: the cache in blocks"; groups as kv_prefix_groups finds
 * them).  The result is the same softmax of [NOTES] "Concept" over each
 * sequence's rows; only the work is arranged differently:
 *  1. a prefix pass (tensor cores, tcgen05) scores group g's P shared rows
 *     once for all q heads of all its members (members x G query rows per
 *     KV head), in key chunks, and leaves per (sequence, q head, chunk) the
 *     unnormalised weighted sum of V, the running maximum and the sum;
 *  2. a merge step combines each row's chunks (all SMs, one thread per row
 *     and 4 columns);
 *  3. the decode pass attends each sequence over its own rows [P, L) only
 *     and folds the merged prefix into its output (a sequence with P = L
 *     gets the prefix alone).
 * Arguments as paged_decode_attention, without scales (fp16 / bf16 caches
 * only; q of the cache's type, else PKV_ERR_INVALID; other caches
 * PKV_ERR_UNSUPPORTED), plus the device arrays group_start [num_groups + 1],
 * group_seqs, group_prefix [num_groups] and seq_prefix [batch] (seq_prefix[b]
 * = P of b's group or 0, consistent with the groups: a sequence with
 * seq_prefix[b] > 0 must be a member of a group with that prefix), their
 * maxima max_group_size and max_prefix_len (<= max_seq_len), and a
 * workspace of paged_decode_cascade_workspace_bytes(pool, batch,
 * num_q_heads, max_prefix_len), zeroed once by the caller like
 * paged_decode_attention's.  Every member's table must hold the same block
 * ids for the prefix's blocks and every member's length must be >= P; the
 * result is undefined otherwise.  seq_prefix[b] < 0 or > seq_lens[b] is
 * recorded in the pool's error word (pkv_check_error then returns
 * PKV_ERR_BAD_INDEX) and the sequence is attended in full.  Three kernels are
 * launched on `stream` (one when no group is given).
 */
int paged_decode_attention_cascade(const pkv_pool *pool, const void *q, pkv_dtype q_dtype,
                                   int num_q_heads, const void *k_cache, const void *v_cache,
                                   const int32_t *block_tables, int max_blocks_per_seq,
                                   const int32_t *seq_lens, int batch, int max_seq_len,
                                   const int32_t *group_start, const int32_t *group_seqs,
                                   const int32_t *group_prefix, const int32_t *seq_prefix,
                                   int num_groups, int max_group_size, int max_prefix_len,
                                   float scale, float *out, void *workspace,
                                   size_t workspace_bytes, pkv_stream_t stream);

/*
 * paged_decode_attention_window — paged_decode_attention restricted to a
 * sliding window: sequence b attends over its last min(window,
 * seq_lens[b]) cached rows only, positions [seq_lens[b] - window,
 * seq_lens[b]).  [VIS] "What the page leaves out" names sliding-window
 * attention as a variant it does not show; this is the plain reading: the
 * softmax of [NOTES] "Concept" taken over the window's rows.  Rows before the
 * window are not read (their table entries are not looked at either), so a
 * caller may already have freed those blocks.  window == 0 is full attention
 * (identical to paged_decode_attention); window < 0 is PKV_ERR_INVALID.  All
 * other arguments, the workspace and the error behaviour are those of
 * paged_decode_attention.
 */
int paged_decode_attention_window(const pkv_pool *pool, const void *q, pkv_dtype q_dtype,
                                  int num_q_heads, const void *k_cache, const void *v_cache,
                                  const void *k_scales, const void *v_scales,
                                  const int32_t *block_tables, int max_blocks_per_seq,
                                  const int32_t *seq_lens, int batch, int max_seq_len,
                                  int window, float scale, float *out, void *workspace,
                                  size_t workspace_bytes, pkv_stream_t stream);

/*
 * paged_prefill_attention — causal attention of a batch of new tokens over
 * the paged cache: the prefill half of serving ([VIS] "Prefill and decode
 * feel different": the whole prompt in one pass, limited by arithmetic
 * rather than memory traffic).
 * Sequence b has n_b = q_start[b+1] - q_start[b] new tokens, the last n_b of
 * its seq_lens[b] cached rows (their K and V already written by kv_append);
 * new token i sits at position p = seq_lens[b] - n_b + i and, for each query
 * head h (KV head h / G),
 *   out[q_start[b] + i][h] = softmax(scale * q[q_start[b] + i][h] . K^T) . V
 * over cached positions 0..p ([NOTES] "Concept").  With n_b = seq_lens[b]
 * this is the prefill of a whole prompt; with fewer it continues a prompt in
 * chunks, and n_b = 1 is a decode step.
 *
 *   q          device [T][Hq][D] of the pool's dtype (F16 or BF16 pools only),
 *              T = q_start[batch]; sequence-major.
 *   q_start    device int32 [batch + 1], q_start[0] = 0, non-decreasing.
 *   seq_lens   device int32 [batch], seq_lens[b] >= n_b.
 *   block_tables, max_blocks_per_seq  as for paged_decode_attention.
 *   max_q_len  >= every n_b (sizes the grid; host value, no device read).
 *   out        device fp32 [T][Hq][D].
 *
 * Runs on the fifth-generation tensor cores (tcgen05.mma, fp16/bf16 inputs,
 * fp32 accumulators in tensor memory; the softmax weights are rounded to the
 * input type for the P.V product), one persistent CTA per SM; K and V are
 * read through tensor maps built on the host for this call's k_cache and
 * v_cache (so both must stay valid until the kernel has run, as for any
 * stream-ordered call).  Head dim 64 or 128.
 * fp32 and quantized pools return PKV_ERR_UNSUPPORTED, and so do shapes
 * whose (256-query tiles x heads x batch) count reaches 2^31; PKV_ERR_CUDA
 * if a tensor map cannot be encoded.  A length out of range sets
 * PKV_ERR_BAD_INDEX in the error word and that sequence is skipped; a block
 * id out of range sets it too and its rows are read as zeros (the
 * sequence's output is unspecified).  No workspace.
 */
int paged_prefill_attention(const pkv_pool *pool, const void *q, int num_q_heads,
                            const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *q_start, const int32_t *seq_lens, int batch,
                            int max_q_len, float scale, float *out, pkv_stream_t stream);

/*
 * pkv_step_layout — where one decode step's inputs sit in a staging buffer:
 * byte offsets from its start.  B = batch, Hkv/D the pool's, Hq = the call's
 * num_q_heads.
 *   k_new, v_new   [B][Hkv][D] of in_dtype, offsets multiples of 16.
 *   q              [B][Hq][D] of q_dtype, offset a multiple of 16.
 *   slot_mapping   int32 [B] (the new token of sequence b goes to slot
 *                  slot_mapping[b]; < 0 = no token), offset a multiple of 4.
 *   seq_lens       int32 [B], the lengths after the append, offset a
 *                  multiple of 4.
 */
typedef struct {
    size_t k_new, v_new, q, slot_mapping, seq_lens;
} pkv_step_layout;

/*
 * paged_decode_step — one whole decode step with the inputs and the result
 * in host memory ([NOTES] "What happens at each decoding step": the new
 * token's key and value are stored, then its query attends over every cached
 * row; [GUIDE] "How the cache turns the loop cheap").  Enqueued on `stream`,
 * in this order:
 *   1. one host-to-device copy of in_bytes from host_in to dev_in (the
 *      step's k_new, v_new, q, slot mapping and lengths at the offsets of
 *      `layout`);
 *   2. kv_append of the B new tokens (slot_mapping, k_new, v_new in dev_in);
 *   3. paged_decode_attention of q over the caches into `out` (device);
 *   4. if host_out is not NULL, one device-to-host copy of out
 *      (B * Hq * D fp32) to host_out.  A page-locked host_out takes the
 *      output directly instead (the attention writes it there through its
 *      device mapping) and `out` is then left unwritten: pass host_out =
 *      NULL to keep the result on the device.
 * Arguments as for kv_append and paged_decode_attention; host_in and
 * host_out should be page-locked (cudaHostAlloc) for the copies to be
 * asynchronous.  Nothing waits: host_in must not change, and host_out must
 * not be read, until the stream has passed the call (an event recorded after
 * it).  PKV_ERR_INVALID for a region of `layout` outside in_bytes or
 * misaligned, or a NULL buffer.  The append's and the attention's argument
 * checks run before anything is enqueued, with their usual results; an
 * error at launch (PKV_ERR_CUDA) stops the sequence where it happened and
 * undoes nothing.  Page-locked host buffers whose size is a multiple of 16
 * bytes are copied by small kernels through their device mapping (so the
 * stream stays a chain of kernels that overlap under programmatic dependent
 * launch; over fp caches the input copy and the append are one kernel);
 * other host memory by cudaMemcpyAsync.  host_in and host_out must not
 * overlap.  `out` must be a valid device buffer in every case.
 */
int paged_decode_step(const pkv_pool *pool, const void *host_in, void *dev_in, size_t in_bytes,
                      const pkv_step_layout *layout, pkv_dtype in_dtype, pkv_dtype q_dtype,
                      int num_q_heads, void *k_cache, void *v_cache, void *k_scales,
                      void *v_scales, const int32_t *block_tables, int max_blocks_per_seq,
                      int batch, int max_seq_len, float scale, float *out, float *host_out,
                      void *workspace, size_t workspace_bytes, pkv_stream_t stream);

/*
 * paged_decode_attention_noalloc — paged_decode_attention for callers that
 * cannot allocate device memory.  The pages have no counterpart; this is a
 * property of this library's interface, not of the method.
 *
 * Same arguments and result as paged_decode_attention, without the
 * workspace: the scratch comes from a fixed 4 MiB array in the library's
 * device image (every GPU that loads the library holds it until exit).  It
 * suits code that may not call cudaMalloc at the point of the call: an
 * allocator hook or host callback that would re-enter the allocator, a
 * serving loop that must not allocate after start-up, or a process whose
 * device memory is fully reserved by another runtime's pool.
 *
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.  The address is kept for the rest of the
 *    process: after a cudaDeviceReset (which unloads the array with the
 *    library's device image) do not call this entry point on that device.
 *  - Each call clears the part of the array it uses (cudaMemsetAsync on
 *    `stream`), then runs the same kernel as paged_decode_attention.  It
 *    calls no cudaMalloc/cudaFree and no allocating library routine.
 *  - All calls on a device share the array: calls that may overlap on the
 *    GPU (different streams without ordering) race; order them.
 *  - Returns PKV_ERR_UNSUPPORTED when the batch needs more scratch than the
 *    array holds (paged_decode_workspace_bytes() > 4 MiB: on 152 SMs, more
 *    than about 1,800 sequence x KV-head pairs at G = 4, d = 128, or about
 *    850 at G = 8).
 */
int paged_decode_attention_noalloc(const pkv_pool *pool, const void *q, pkv_dtype q_dtype,
                                   int num_q_heads, const void *k_cache, const void *v_cache,
                                   const void *k_scales, const void *v_scales,
                                   const int32_t *block_tables, int max_blocks_per_seq,
                                   const int32_t *seq_lens, int batch, int max_seq_len,
                                   float scale, float *out, pkv_stream_t stream);

/*
 * pkv_selftest_wait_timeout — a check of the failure path of the library's
 * bounded device waits (not part of the method).  Launches one kernel whose
 * single waiting thread waits, the way every mbarrier wait in this library
 * does, on a phase that nothing completes; after the wait's time limit
 * (about one second) it records a timeout in the pool's error word and
 * returns.  The next pkv_check_error() then returns PKV_ERR_TIMEOUT and the
 * device stays usable.  Returns PKV_OK when the kernel was launched,
 * PKV_ERR_INVALID for a null pool, PKV_ERR_CUDA without a device.
 */
int pkv_selftest_wait_timeout(const pkv_pool *pool, pkv_stream_t stream);

/*
 * pkv_check_error — synchronise the stream, read and clear the pool's device
 * error word.  Returns PKV_OK, PKV_ERR_BAD_INDEX, PKV_ERR_TIMEOUT (a bounded
 * wait inside a kernel gave up; the kernel returned without finishing), or
 * PKV_ERR_CUDA.
 */
int pkv_check_error(const pkv_pool *pool, pkv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
