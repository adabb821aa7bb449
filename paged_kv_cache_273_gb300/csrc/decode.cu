// Host side of paged_decode_attention: workspace sizing and the dispatch to
// the kernel instantiation for the pool's K/V dtype (each dtype is compiled
// in its own translation unit, decode_<dtype>.cu).

#include <cuda_runtime.h>

#include <algorithm>

#include "pkv_internal.h"

#include "decode_kernel.cuh"

// Instantiated in decode_<dtype>.cu.
namespace pkv {
namespace kern {
extern template int launch_d<PKV_F32>(const pkv_pool *, int, const Params &, int, int, cudaStream_t);
extern template int launch_d<PKV_F16>(const pkv_pool *, int, const Params &, int, int, cudaStream_t);
extern template int launch_d<PKV_BF16>(const pkv_pool *, int, const Params &, int, int, cudaStream_t);
extern template int launch_d<PKV_I8>(const pkv_pool *, int, const Params &, int, int, cudaStream_t);
extern template int launch_d<PKV_I4>(const pkv_pool *, int, const Params &, int, int, cudaStream_t);
}  // namespace kern
}  // namespace pkv

namespace pkv {
namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

bool encode_swizzled_tile_map(CUtensorMap *map, const void *base, int row_bytes,
                              const pkv_pool *pool)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc || (row_bytes != 128 && row_bytes != 256) || pool->block_size < 16)
        return false;
    const cuuint64_t bs = (cuuint64_t)pool->block_size;
    const cuuint64_t nbh = (cuuint64_t)pool->num_blocks * (cuuint64_t)pool->num_kv_heads;
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    if (row_bytes == 128) {
        const cuuint64_t dims[3] = {128, bs, nbh};
        const cuuint64_t strides[2] = {128, bs * 128};
        const cuuint32_t box[3] = {128, 16, 1};
        return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
    const cuuint64_t dims[4] = {128, 2, bs, nbh};
    const cuuint64_t strides[3] = {128, 256, bs * 256};
    const cuuint32_t box[4] = {128, 2, 16, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_gather_row_map(CUtensorMap *map, const void *base, int row_bytes, int rt,
                           const pkv_pool *pool)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    const int bs = pool->block_size;
    const int64_t rb = (int64_t)rt * row_bytes;
    if (!enc || rt < 1 || bs % rt != 0 || rb % 16 != 0 || rb / 8 > 256)
        return false;
    const cuuint64_t dims[2] = {(cuuint64_t)(rb / 8),
                                (cuuint64_t)pool->num_blocks * pool->num_kv_heads * (bs / rt)};
    const cuuint64_t strides[1] = {(cuuint64_t)rb};
    const cuuint32_t box[2] = {(cuuint32_t)(rb / 8), 1};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void *>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t decode_workspace_bytes(const pkv_pool *pool, int batch, int num_q_heads)
{
    const int G = num_q_heads / pool->num_kv_heads;
    const size_t counters = align_up((size_t)batch * pool->num_kv_heads * sizeof(int), 256);
    const size_t entries = (size_t)std::max(pool->num_sms, 1) + (size_t)batch * pool->num_kv_heads;
    const size_t partials = entries * (size_t)G * (pool->head_dim + 2) * sizeof(float);
    return counters + align_up(partials, 256);
}

int launch_decode(const pkv_pool *pool, const void *q, pkv_dtype q_dtype, int num_q_heads,
                  const void *k_cache, const void *v_cache, const void *k_scales,
                  const void *v_scales, const int32_t *block_tables, int max_blocks_per_seq,
                  const int32_t *seq_lens, int batch, int max_seq_len, int window, float scale,
                  float *out,
                  void *workspace, size_t workspace_bytes, pkv_stream_t stream,
                  const int32_t *seq_prefix, const float *prefix_part)
{
    (void)workspace_bytes;
    const int Hkv = pool->num_kv_heads;
    const int G = num_q_heads / Hkv;
    // tiles, and their cost for the split over CTAs, must count in 31 bits
    const int64_t tiles_bound =
        (int64_t)batch * Hkv *
        (((int64_t)max_seq_len + kern::TILE - 1) / kern::TILE + kern::piece_cost(G));
    if (tiles_bound >= ((int64_t)1 << 31))
        return PKV_ERR_UNSUPPORTED;
    kern::Params prm{};
    prm.q = q;
    prm.k_cache = static_cast<const unsigned char *>(k_cache);
    prm.v_cache = static_cast<const unsigned char *>(v_cache);
    prm.k_scales = static_cast<const __half *>(k_scales);
    prm.v_scales = static_cast<const __half *>(v_scales);
    prm.block_tables = block_tables;
    prm.seq_lens = seq_lens;
    prm.out = out;
    const size_t counters = align_up((size_t)batch * Hkv * sizeof(int), 256);
    prm.counters = static_cast<int *>(workspace);
    prm.partials = reinterpret_cast<float *>(static_cast<unsigned char *>(workspace) + counters);
    prm.err = pool->d_err;
    prm.batch = batch;
    prm.num_q_heads = num_q_heads;
    prm.num_kv_heads = Hkv;
    prm.block_size = pool->block_size;
    int lg = 0;
    while ((1 << lg) < pool->block_size)
        ++lg;
    prm.bs_log2 = lg;
    prm.max_blocks_per_seq = max_blocks_per_seq;
    prm.max_seq_len = max_seq_len;
    const int64_t table_cap = (int64_t)max_blocks_per_seq * pool->block_size;
    prm.len_cap = (int)std::min<int64_t>(max_seq_len, table_cap);
    prm.window = window > 0 ? window : 0;
    prm.seq_prefix = seq_prefix;
    prm.prefix_part = prefix_part;
    prm.num_blocks = pool->num_blocks;
    prm.q_dtype = q_dtype;
    prm.q_bytes = dtype_bytes(q_dtype);
    prm.scale_log2 = (float)((double)scale * 1.4426950408889634);  // log2(e)
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    switch (pool->kv_dtype) {
    case PKV_F32: return kern::launch_d<PKV_F32>(pool, G, prm, batch, max_seq_len, s);
    case PKV_F16: return kern::launch_d<PKV_F16>(pool, G, prm, batch, max_seq_len, s);
    case PKV_BF16: return kern::launch_d<PKV_BF16>(pool, G, prm, batch, max_seq_len, s);
    case PKV_I8: return kern::launch_d<PKV_I8>(pool, G, prm, batch, max_seq_len, s);
    case PKV_I4: return kern::launch_d<PKV_I4>(pool, G, prm, batch, max_seq_len, s);
    }
    return PKV_ERR_UNSUPPORTED;
}

}  // namespace pkv
