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
int launch_block_copy(const pkv_pool *pool, const int32_t *src, const int32_t *dst, int n,
                      void *k_cache, void *v_cache, void *k_scales, void *v_scales,
                      pkv_stream_t stream);
int launch_append(const pkv_pool *pool, const void *k_new, const void *v_new, pkv_dtype in_dtype,
                  const int32_t *slot_mapping, int num_tokens, void *k_cache, void *v_cache,
                  void *k_scales, void *v_scales, pkv_stream_t stream);

size_t decode_workspace_bytes(const pkv_pool *pool, int batch, int num_q_heads);

// The driver's tensor-map encoder (cuTensorMapEncodeTiled), looked up once
// through the runtime; null if unavailable.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

int launch_decode(const pkv_pool *pool, const void *q, pkv_dtype q_dtype, int num_q_heads,
                  const void *k_cache, const void *v_cache, const void *k_scales,
                  const void *v_scales, const int32_t *block_tables, int max_blocks_per_seq,
                  const int32_t *seq_lens, int batch, int max_seq_len, int window, float scale,
                  float *out,
                  void *workspace, size_t workspace_bytes, pkv_stream_t stream);

}  // namespace pkv
