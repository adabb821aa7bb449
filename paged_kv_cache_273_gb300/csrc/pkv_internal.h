// Internal declarations shared by the host pool and the CUDA launchers of
// libpkv.  Not part of the public ABI (that is include/pkv.h).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstddef>
#include <cstdint>
#include <vector>

#include "pkv.h"

// Bits of the device error word.
enum : unsigned int {
    PKV_EBIT_SLOT = 1u,      // kv_append: slot outside [0, NB*bs)
    PKV_EBIT_BLOCK = 2u,     // attention, block copy: block id outside [0, NB)
    PKV_EBIT_SEQLEN = 4u,    // attention: seq_len < 0 or beyond its block table row
    PKV_EBIT_TIMEOUT = 8u,   // a bounded mbarrier wait gave up
};

struct pkv_pool {
    int num_blocks = 0;
    int block_size = 0;
    int num_kv_heads = 0;
    int head_dim = 0;
    pkv_dtype kv_dtype = PKV_F32;

    std::vector<int32_t> free_stack;  // free block ids; alloc pops from the back
    std::vector<int32_t> refcount;    // per block, 0 = free

    // Device side (absent when no CUDA device was usable at init).
    bool has_device = false;
    int device = -1;
    int num_sms = 0;
    int max_smem_optin = 0;
    unsigned int *d_err = nullptr;    // device error word
};

namespace pkv {

inline int dtype_bytes(pkv_dtype t)
{
    switch (t) {
    case PKV_F32: return 4;
    case PKV_F16: case PKV_BF16: return 2;
    case PKV_I8: return 1;
    case PKV_I4: return 0;      // two per byte: use row_bytes()
    }
    return 0;
}

// Bytes of one cached row of head_dim elements (4-bit codes: two per byte).
inline int64_t row_bytes(pkv_dtype t, int head_dim)
{
    return t == PKV_I4 ? head_dim / 2 : (int64_t)head_dim * dtype_bytes(t);
}

// Caches with one fp16 scale per cached row.
inline bool quantized_dtype(pkv_dtype t) { return t == PKV_I8 || t == PKV_I4; }

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launchers (defined in the .cu files).  They assume validated arguments.
int launch_prefill(const pkv_pool *pool, const void *q, int num_q_heads, const void *k_cache,
                   const void *v_cache, const int32_t *block_tables, int max_blocks_per_seq,
                   const int32_t *q_start, const int32_t *seq_lens, int batch, int max_q_len,
                   float scale, float *out, pkv_stream_t stream);
int launch_selftest_wait_timeout(const pkv_pool *pool, pkv_stream_t stream);
// 16-byte-chunk copy kernel of paged_decode_step (both pointers device-
// addressable and 16-byte aligned, bytes a multiple of 16; PKV_ERR_INVALID
// otherwise).  load_first: src is not written by earlier kernels of the
// stream, so its loads may overlap the previous kernel.
int launch_stage_copy(const void *src, void *dst, size_t bytes, bool load_first,
                      pkv_stream_t stream);
// The input side of paged_decode_step over an fp cache in one kernel: the
// staging copy of bytes from src (page-locked host memory, by its device
// address) to dst, and the append of the batch's new K and V rows (at byte
// offsets k_off, v_off of the buffer, slots at slot_off) into the caches.
// PKV_ERR_INVALID for quantized pools or misaligned arguments.
int launch_step_in(const pkv_pool *pool, const void *src, void *dst, size_t bytes,
                   size_t k_off, size_t v_off, size_t slot_off, int batch, void *k_cache,
                   void *v_cache, pkv_stream_t stream);
int launch_block_copy(const pkv_pool *pool, const int32_t *src, const int32_t *dst, int n,
                      void *k_cache, void *v_cache, void *k_scales, void *v_scales,
                      pkv_stream_t stream);
int launch_append(const pkv_pool *pool, const void *k_new, const void *v_new, pkv_dtype in_dtype,
                  const int32_t *slot_mapping, int num_tokens, void *k_cache, void *v_cache,
                  void *k_scales, void *v_scales, pkv_stream_t stream);

size_t decode_workspace_bytes(const pkv_pool *pool, int batch, int num_q_heads);

// Shared-prefix (cascade) decode: the prefix pass splits a prefix of up to
// max_prefix_len tokens into at most 16 chunks of *kc_tiles 128-key tiles
// (*nkc chunks when the prefix is that long).
inline void prefix_chunks(int max_prefix_len, int *kc_tiles, int *nkc)
{
    const int tiles = (max_prefix_len + 127) / 128;
    int kc = (tiles + 15) / 16;
    if (kc < 1)
        kc = 1;
    *kc_tiles = kc;
    *nkc = tiles > 0 ? (tiles + kc - 1) / kc : 1;
}

// Floats of one prefix partial row: O[D], running maximum, sum, 2 pad (16-byte rows).
inline int prefix_row_floats(int head_dim) { return head_dim + 4; }

// Bytes of the prefix partials [nkc][batch][num_q_heads][D + 4] fp32 (chunk 0
// ends up holding the merged prefix of every row).
inline size_t prefix_partials_bytes(const pkv_pool *pool, int batch, int num_q_heads,
                                    int max_prefix_len)
{
    int kc = 1, nkc = 1;
    prefix_chunks(max_prefix_len, &kc, &nkc);
    return (size_t)nkc * batch * num_q_heads * prefix_row_floats(pool->head_dim) * sizeof(float);
}


// The prefix pass (tcgen05, the prefill kernel's machinery): partials of
// every group member's q heads over its group's shared prefix.
int launch_prefix_pass(const pkv_pool *pool, const void *q, int num_q_heads, const void *k_cache,
                       const void *v_cache, const int32_t *block_tables, int max_blocks_per_seq,
                       const int32_t *seq_lens, int batch, const int32_t *grp_start,
                       const int32_t *grp_seqs, const int32_t *grp_len, int ngroups,
                       int max_group_size, int max_prefix_len, float scale, float *part,
                       int *kc_tiles, pkv_stream_t stream);

// Merge the prefix pass's chunk partials of every row of a sequence with a
// prefix into chunk 0 (O; maximum and sum at D + 2, D + 3).
int launch_prefix_merge(const pkv_pool *pool, const int32_t *seq_prefix, float *part, int batch,
                        int num_q_heads, int kc_tiles, pkv_stream_t stream);

// The driver's tensor-map encoder (cuTensorMapEncodeTiled), looked up once
// through the runtime; null if unavailable.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// A cache [NB][Hkv][bs][row_bytes] (row_bytes 128 or 256) as the tensor the
// decode kernel's swizzled tile copies read: bytes in 128-byte segments,
// {128, bs, NB * Hkv} or {128, 2, bs, NB * Hkv}, boxes of 16 rows, 128-byte
// swizzle.  False if the encoder is unavailable or refuses.
bool encode_swizzled_tile_map(CUtensorMap *map, const void *base, int row_bytes,
                              const pkv_pool *pool);

// A cache [NB][Hkv][bs][row_bytes] as a 2-D tensor of rows of rt cached
// rows each (rt divides bs; 8-byte elements), boxes of one such row, for
// four-row gather copies.  False if the encoder is unavailable or refuses.
bool encode_gather_row_map(CUtensorMap *map, const void *base, int row_bytes, int rt,
                           const pkv_pool *pool);

// seq_prefix / prefix_part: shared-prefix decode (null: none), see Params.
int launch_decode(const pkv_pool *pool, const void *q, pkv_dtype q_dtype, int num_q_heads,
                  const void *k_cache, const void *v_cache, const void *k_scales,
                  const void *v_scales, const int32_t *block_tables, int max_blocks_per_seq,
                  const int32_t *seq_lens, int batch, int max_seq_len, int window, float scale,
                  float *out,
                  void *workspace, size_t workspace_bytes, pkv_stream_t stream,
                  const int32_t *seq_prefix = nullptr, const float *prefix_part = nullptr);

}  // namespace pkv
