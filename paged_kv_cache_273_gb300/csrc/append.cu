// kv_append: write the new tokens' K and V rows into the paged cache.
//
// "KV cache: the engine behind fast LLM inference", "What happens at each
// decoding step", step 4: only the new token's key and value are computed,
// and they join the cache.  The cache slot of a token comes from its block
// table (KV cache visualization page, "PagedAttention: the cache in blocks").
//
// fp caches: a bit copy, 16 bytes per thread.  int8 caches ("Quantized KV
// cache" on the same page): one warp per (token, head, K-or-V) row computes the
// row's absolute maximum, an fp16 scale amax/127 and round-half-even codes.
//
// kv_block_copy: the copy half of copy-on-write (KV cache visualization page,
// "PagedAttention: the cache in blocks": a shared block is copied only when a
// request writes to it), a bit copy of whole blocks.

#include <cuda_runtime.h>

#include "device_common.cuh"

namespace pkv {
namespace {

using namespace dev;

// One thread per 16-byte chunk of a (token, head) row, K and V in the same
// pass.  chunks_per_row = D * eb / 16.
__global__ void __launch_bounds__(256) append_copy_kernel(
    const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
    const int32_t *__restrict__ slot_mapping, int64_t total_chunks, int chunks_per_row,
    int num_kv_heads, int block_size, int64_t num_slots, uint4 *__restrict__ k_cache,
    uint4 *__restrict__ v_cache, unsigned int *__restrict__ err)
{
    grid_dependency_wait();
    grid_dependents_launch();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < total_chunks;
         c += stride) {
        const int64_t row = c / chunks_per_row;          // (token, head)
        const int chunk = (int)(c - row * chunks_per_row);
        const int64_t t = row / num_kv_heads;
        const int h = (int)(row - t * num_kv_heads);
        const int32_t slot = __ldg(slot_mapping + t);
        if (slot < 0)
            continue;                                     // padding token
        if ((int64_t)slot >= num_slots) {
            atomicOr(err, PKV_EBIT_SLOT);
            continue;
        }
        const int64_t blk = slot / block_size;
        const int64_t off = slot - blk * block_size;
        const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * chunks_per_row + chunk;
        k_cache[dst] = __ldg(k_new + c);
        v_cache[dst] = __ldg(v_new + c);
    }
}

template <typename T>
__device__ __forceinline__ float load_as_float(const T *p);
template <>
__device__ __forceinline__ float load_as_float<float>(const float *p) { return __ldg(p); }
template <>
__device__ __forceinline__ float load_as_float<__half>(const __half *p) { return __half2float(__ldg(p)); }
template <>
__device__ __forceinline__ float load_as_float<__nv_bfloat16>(const __nv_bfloat16 *p)
{
    return __bfloat162float(__ldg(p));
}

// One warp per (token, head, K|V) row.  D = 32 * E.
template <typename T, int E>
__global__ void __launch_bounds__(256) append_q8_kernel(
    const T *__restrict__ k_new, const T *__restrict__ v_new,
    const int32_t *__restrict__ slot_mapping, int64_t num_rows /* T*Hkv */, int num_kv_heads,
    int block_size, int64_t num_slots, int8_t *__restrict__ k_cache, int8_t *__restrict__ v_cache,
    __half *__restrict__ k_scales, __half *__restrict__ v_scales, unsigned int *__restrict__ err)
{
    constexpr int D = 32 * E;
    grid_dependency_wait();
    grid_dependents_launch();
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t w = warp; w < 2 * num_rows; w += nwarps) {
        const bool is_v = w >= num_rows;
        const int64_t row = is_v ? w - num_rows : w;
        const int64_t t = row / num_kv_heads;
        const int h = (int)(row - t * num_kv_heads);
        const int32_t slot = __ldg(slot_mapping + t);
        if (slot < 0)
            continue;
        if ((int64_t)slot >= num_slots) {
            if (lane == 0)
                atomicOr(err, PKV_EBIT_SLOT);
            continue;
        }
        const T *src = (is_v ? v_new : k_new) + row * D + lane * E;
        float x[E];
        float amax = 0.0f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            x[e] = load_as_float<T>(src + e);
            amax = fmaxf(amax, fabsf(x[e]));
        }
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1)
            amax = fmaxf(amax, __shfl_xor_sync(FULL_MASK, amax, m));
        // IEEE fp32 division and round-to-nearest-even conversions only.
        const __half s16 = __float2half_rn(__fdiv_rn(amax, 127.0f));
        const float s = __half2float(s16);
        const int64_t blk = slot / block_size;
        const int64_t off = slot - blk * block_size;
        const int64_t srow = (blk * num_kv_heads + h) * block_size + off;
        int8_t *dst = (is_v ? v_cache : k_cache) + srow * D + lane * E;
        static_assert(E == 2 || E == 4, "two or four codes per lane");
        uint32_t word = 0;
#pragma unroll
        for (int u = 0; u < E; ++u) {
            int code = 0;
            if (s != 0.0f) {
                float c = rintf(__fdiv_rn(x[u], s));     // round half to even
                c = fminf(fmaxf(c, -127.0f), 127.0f);
                code = (int)c;
            }
            word |= (uint32_t)(code & 0xff) << (8 * u);
        }
        if (E == 4)
            *reinterpret_cast<uint32_t *>(dst) = word;
        else
            *reinterpret_cast<uint16_t *>(dst) = (uint16_t)word;
        if (lane == 0)
            (is_v ? v_scales : k_scales)[srow] = s16;
    }
}

// 4-bit cache ([NOTES] "Quantized KV cache": fewer bits per number; the
// pages name 4-bit caches without fixing a scheme): one warp per (token,
// head, K|V) row of D = 128 values, the same symmetric per-row scheme as int8
// with range +-7: s = fp16_rne(amax / 7), code = clamp(round_half_even(x/s)).
// Codes are two's-complement nibbles, element 2j in the low nibble of byte j;
// each lane packs its 4 codes into 2 bytes.
template <typename T>
__global__ void __launch_bounds__(256) append_q4_kernel(
    const T *__restrict__ k_new, const T *__restrict__ v_new,
    const int32_t *__restrict__ slot_mapping, int64_t num_rows /* T*Hkv */, int num_kv_heads,
    int block_size, int64_t num_slots, uint8_t *__restrict__ k_cache,
    uint8_t *__restrict__ v_cache, __half *__restrict__ k_scales, __half *__restrict__ v_scales,
    unsigned int *__restrict__ err)
{
    constexpr int D = 128, E = 4;
    grid_dependency_wait();
    grid_dependents_launch();
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t w = warp; w < 2 * num_rows; w += nwarps) {
        const bool is_v = w >= num_rows;
        const int64_t row = is_v ? w - num_rows : w;
        const int64_t t = row / num_kv_heads;
        const int h = (int)(row - t * num_kv_heads);
        const int32_t slot = __ldg(slot_mapping + t);
        if (slot < 0)
            continue;
        if ((int64_t)slot >= num_slots) {
            if (lane == 0)
                atomicOr(err, PKV_EBIT_SLOT);
            continue;
        }
        const T *src = (is_v ? v_new : k_new) + row * D + lane * E;
        float x[E];
        float amax = 0.0f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            x[e] = load_as_float<T>(src + e);
            amax = fmaxf(amax, fabsf(x[e]));
        }
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1)
            amax = fmaxf(amax, __shfl_xor_sync(FULL_MASK, amax, m));
        // IEEE fp32 division and round-to-nearest-even conversions only.
        const __half s16 = __float2half_rn(__fdiv_rn(amax, 7.0f));
        const float s = __half2float(s16);
        const int64_t blk = slot / block_size;
        const int64_t off = slot - blk * block_size;
        const int64_t srow = (blk * num_kv_heads + h) * block_size + off;
        uint32_t word = 0;
#pragma unroll
        for (int u = 0; u < E; ++u) {
            int code = 0;
            if (s != 0.0f) {
                float c = rintf(__fdiv_rn(x[u], s));     // round half to even
                c = fminf(fmaxf(c, -7.0f), 7.0f);
                code = (int)c;
            }
            word |= (uint32_t)(code & 0xf) << (4 * u);
        }
        uint8_t *dst = (is_v ? v_cache : k_cache) + srow * (D / 2) + lane * (E / 2);
        *reinterpret_cast<uint16_t *>(dst) = (uint16_t)word;
        if (lane == 0)
            (is_v ? v_scales : k_scales)[srow] = s16;
    }
}

// Copy whole blocks (copy-on-write): K and V of block src[i] -> dst[i], one
// thread per 16-byte chunk; a block-head tile row is a multiple of 16 bytes.
// int8 scales ([NB][Hkv][bs] fp16) follow as 2-byte elements.
__global__ void __launch_bounds__(256) block_copy_kernel(
    const int32_t *__restrict__ src, const int32_t *__restrict__ dst, int n,
    int64_t chunks_per_block, int64_t scales_per_block, int num_blocks,
    uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache, __half *__restrict__ k_scales,
    __half *__restrict__ v_scales, unsigned int *__restrict__ err)
{
    grid_dependency_wait();
    grid_dependents_launch();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t per_pair = 2 * chunks_per_block + 2 * scales_per_block;
    for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < (int64_t)n * per_pair;
         c += stride) {
        const int i = (int)(c / per_pair);
        int64_t r = c - (int64_t)i * per_pair;
        const int32_t s = __ldg(src + i), d = __ldg(dst + i);
        if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
            if (r == 0)
                atomicOr(err, PKV_EBIT_BLOCK);
            continue;
        }
        if (r < 2 * chunks_per_block) {
            uint4 *cache = r < chunks_per_block ? k_cache : v_cache;
            if (r >= chunks_per_block)
                r -= chunks_per_block;
            cache[(int64_t)d * chunks_per_block + r] = cache[(int64_t)s * chunks_per_block + r];
        } else {
            r -= 2 * chunks_per_block;
            __half *sc = r < scales_per_block ? k_scales : v_scales;
            if (r >= scales_per_block)
                r -= scales_per_block;
            sc[(int64_t)d * scales_per_block + r] = sc[(int64_t)s * scales_per_block + r];
        }
    }
}

// Staging copies of a decode step with host buffers (paged_decode_step):
// 16-byte chunks between page-locked host memory, reached through its
// device mapping, and device memory.  Thread t of block b moves chunks
// b*256*SC + c*256 + t (c < SC).  LOAD_FIRST: the source is not written by
// the previous kernels of the stream (the caller's host input), so the
// chunks are loaded before the wait for the previous kernel and stored after
// it; with programmatic dependent launch the loads then overlap that
// kernel's tail.  Otherwise (the device output) the wait comes first.
constexpr int SC = 4;

template <bool LOAD_FIRST>
__global__ void __launch_bounds__(256) stage_copy_kernel(const uint4 *__restrict__ src,
                                                         uint4 *__restrict__ dst, int64_t n)
{
    grid_dependents_launch();
    const int64_t base = (int64_t)blockIdx.x * blockDim.x * SC + threadIdx.x;
    uint4 v[SC];
    if (!LOAD_FIRST)
        grid_dependency_wait();
#pragma unroll
    for (int c = 0; c < SC; ++c) {
        const int64_t i = base + (int64_t)c * blockDim.x;
        if (i < n)
            v[c] = src[i];
    }
    if (LOAD_FIRST)
        grid_dependency_wait();
#pragma unroll
    for (int c = 0; c < SC; ++c) {
        const int64_t i = base + (int64_t)c * blockDim.x;
        if (i < n)
            dst[i] = v[c];
    }
}

// The input side of a decode step with a page-locked host staging buffer
// over an fp cache, in one kernel: the staging copy above, and for the
// chunks of the new K and V rows also the append (the bit copy of
// append_copy_kernel) into the cache slots the staged slot mapping names.
// Host loads (the chunks, each K/V chunk's slot) come before the wait for
// the previous kernel; the stores after it.
struct StepIn {
    int64_t k_new, v_new, slots;   // 16-byte chunk offsets / int32 index of the regions
    int B, H, chunks_per_row, block_size;
    int64_t num_slots;
};

__global__ void __launch_bounds__(256) step_in_kernel(const uint4 *__restrict__ src,
                                                      uint4 *__restrict__ dst, int64_t n,
                                                      StepIn a, uint4 *__restrict__ k_cache,
                                                      uint4 *__restrict__ v_cache,
                                                      unsigned int *__restrict__ err)
{
    grid_dependents_launch();
    const int32_t *slot_mapping = reinterpret_cast<const int32_t *>(src) + a.slots;
    const int64_t row_chunks = (int64_t)a.B * a.H * a.chunks_per_row;
    const int64_t base = (int64_t)blockIdx.x * blockDim.x * SC + threadIdx.x;
    uint4 v[SC];
    int64_t kd[SC], vd[SC];   // cache chunk a K / V chunk goes to, or -1
#pragma unroll
    for (int c = 0; c < SC; ++c) {
        const int64_t i = base + (int64_t)c * blockDim.x;
        kd[c] = vd[c] = -1;
        if (i < n) {
            v[c] = src[i];
#pragma unroll
            for (int kv = 0; kv < 2; ++kv) {
                const int64_t rel = i - (kv == 0 ? a.k_new : a.v_new);
                if (rel >= 0 && rel < row_chunks) {
                    const int64_t row = rel / a.chunks_per_row;   // (token, head)
                    const int chunk = (int)(rel - row * a.chunks_per_row);
                    const int64_t t = row / a.H;
                    const int h = (int)(row - t * a.H);
                    const int32_t slot = slot_mapping[t];
                    int64_t d = -1;
                    if (slot >= 0 && (int64_t)slot < a.num_slots) {
                        const int64_t blk = slot / a.block_size;
                        const int64_t off = slot - blk * a.block_size;
                        d = ((blk * a.H + h) * a.block_size + off) * a.chunks_per_row + chunk;
                    } else if (slot >= 0) {
                        d = -2;                                  // slot out of range
                    }
                    (kv == 0 ? kd[c] : vd[c]) = d;
                }
            }
        }
    }
    grid_dependency_wait();
#pragma unroll
    for (int c = 0; c < SC; ++c) {
        const int64_t i = base + (int64_t)c * blockDim.x;
        if (i < n) {
            dst[i] = v[c];
            if (kd[c] >= 0)
                k_cache[kd[c]] = v[c];
            if (vd[c] >= 0)
                v_cache[vd[c]] = v[c];
            if (kd[c] == -2 || vd[c] == -2)
                atomicOr(err, PKV_EBIT_SLOT);
        }
    }
}

int grid_for(int64_t work_items, int threads, int num_sms)
{
    int64_t blocks = (work_items + threads - 1) / threads;
    int64_t cap = (int64_t)num_sms * 8;
    if (blocks > cap)
        blocks = cap;
    if (blocks < 1)
        blocks = 1;
    return (int)blocks;
}

}  // namespace

int launch_stage_copy(const void *src, void *dst, size_t bytes, bool load_first,
                      pkv_stream_t stream)
{
    if (bytes % 16 != 0 || !aligned16(src) || !aligned16(dst))
        return PKV_ERR_INVALID;
    const int64_t n = (int64_t)(bytes / 16);
    if (n == 0)
        return PKV_OK;
    const int threads = 256;
    const int64_t blocks = (n + threads * SC - 1) / (threads * SC);
    if (blocks > INT32_MAX)
        return PKV_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const cudaError_t e =
        load_first
            ? launch_pdl(stage_copy_kernel<true>, dim3((unsigned)blocks), dim3(threads), 0, s,
                         static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), n)
            : launch_pdl(stage_copy_kernel<false>, dim3((unsigned)blocks), dim3(threads), 0, s,
                         static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), n);
    if (e != cudaSuccess)
        return PKV_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

int launch_step_in(const pkv_pool *pool, const void *src, void *dst, size_t bytes,
                   size_t k_off, size_t v_off, size_t slot_off, int batch, void *k_cache,
                   void *v_cache, pkv_stream_t stream)
{
    if (quantized_dtype(pool->kv_dtype) || bytes % 16 != 0 || k_off % 16 != 0 ||
        v_off % 16 != 0 || slot_off % 4 != 0 || !aligned16(src) || !aligned16(dst) ||
        !aligned16(k_cache) || !aligned16(v_cache))
        return PKV_ERR_INVALID;
    const int64_t n = (int64_t)(bytes / 16);
    if (n == 0 || batch == 0)
        return PKV_OK;
    StepIn a;
    a.k_new = (int64_t)(k_off / 16);
    a.v_new = (int64_t)(v_off / 16);
    a.slots = (int64_t)(slot_off / 4);
    a.B = batch;
    a.H = pool->num_kv_heads;
    a.chunks_per_row = pool->head_dim * dtype_bytes(pool->kv_dtype) / 16;
    a.block_size = pool->block_size;
    a.num_slots = (int64_t)pool->num_blocks * pool->block_size;
    const int threads = 256;
    const int64_t blocks = (n + threads * SC - 1) / (threads * SC);
    if (blocks > INT32_MAX)
        return PKV_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (launch_pdl(step_in_kernel, dim3((unsigned)blocks), dim3(threads), 0, s,
                   static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), n, a,
                   static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache),
                   pool->d_err) != cudaSuccess)
        return PKV_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

int launch_block_copy(const pkv_pool *pool, const int32_t *src, const int32_t *dst, int n,
                      void *k_cache, void *v_cache, void *k_scales, void *v_scales,
                      pkv_stream_t stream)
{
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t rows = (int64_t)pool->num_kv_heads * pool->block_size;
    const int64_t chunks = rows * row_bytes(pool->kv_dtype, pool->head_dim) / 16;
    const int64_t scales = quantized_dtype(pool->kv_dtype) ? rows : 0;
    const int threads = 256;
    const int64_t total = (int64_t)n * (2 * chunks + 2 * scales);
    launch_pdl(block_copy_kernel, dim3(grid_for(total, threads, pool->num_sms)), dim3(threads), 0,
               s, src, dst, n, chunks, scales, pool->num_blocks, static_cast<uint4 *>(k_cache),
               static_cast<uint4 *>(v_cache), static_cast<__half *>(k_scales),
               static_cast<__half *>(v_scales), pool->d_err);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

int launch_append(const pkv_pool *pool, const void *k_new, const void *v_new, pkv_dtype in_dtype,
                  const int32_t *slot_mapping, int num_tokens, void *k_cache, void *v_cache,
                  void *k_scales, void *v_scales, pkv_stream_t stream)
{
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int H = pool->num_kv_heads, D = pool->head_dim, bs = pool->block_size;
    const int64_t num_slots = (int64_t)pool->num_blocks * bs;
    if (pool->kv_dtype == PKV_I4) {
        const int64_t rows = (int64_t)num_tokens * H;
        const int threads = 256;
        const int grid = grid_for(2 * rows * 32, threads, pool->num_sms);
        uint8_t *kc = static_cast<uint8_t *>(k_cache);
        uint8_t *vc = static_cast<uint8_t *>(v_cache);
        __half *ks = static_cast<__half *>(k_scales);
        __half *vs = static_cast<__half *>(v_scales);
#define PKV_Q4(T)                                                                           \
    launch_pdl(append_q4_kernel<T>, dim3(grid), dim3(threads), 0, s,                         \
               static_cast<const T *>(k_new), static_cast<const T *>(v_new), slot_mapping,   \
               rows, H, bs, num_slots, kc, vc, ks, vs, pool->d_err)
        if (in_dtype == PKV_F16) PKV_Q4(__half);
        else if (in_dtype == PKV_BF16) PKV_Q4(__nv_bfloat16);
        else PKV_Q4(float);
#undef PKV_Q4
    } else if (pool->kv_dtype != PKV_I8) {
        const int chunks_per_row = D * dtype_bytes(pool->kv_dtype) / 16;
        const int64_t total = (int64_t)num_tokens * H * chunks_per_row;
        const int threads = 256;
        launch_pdl(append_copy_kernel, dim3(grid_for(total, threads, pool->num_sms)),
                   dim3(threads), 0, s, static_cast<const uint4 *>(k_new),
                   static_cast<const uint4 *>(v_new), slot_mapping, total, chunks_per_row, H, bs,
                   num_slots, static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache),
                   pool->d_err);
    } else {
        const int64_t rows = (int64_t)num_tokens * H;
        const int threads = 256;
        const int grid = grid_for(2 * rows * 32, threads, pool->num_sms);
        int8_t *kc = static_cast<int8_t *>(k_cache);
        int8_t *vc = static_cast<int8_t *>(v_cache);
        __half *ks = static_cast<__half *>(k_scales);
        __half *vs = static_cast<__half *>(v_scales);
#define PKV_Q8(T, E)                                                                        \
    launch_pdl(append_q8_kernel<T, E>, dim3(grid), dim3(threads), 0, s,                      \
               static_cast<const T *>(k_new), static_cast<const T *>(v_new), slot_mapping,   \
               rows, H, bs, num_slots, kc, vc, ks, vs, pool->d_err)
        if (D == 128) {
            if (in_dtype == PKV_F16) PKV_Q8(__half, 4);
            else if (in_dtype == PKV_BF16) PKV_Q8(__nv_bfloat16, 4);
            else PKV_Q8(float, 4);
        } else {
            if (in_dtype == PKV_F16) PKV_Q8(__half, 2);
            else if (in_dtype == PKV_BF16) PKV_Q8(__nv_bfloat16, 2);
            else PKV_Q8(float, 2);
        }
#undef PKV_Q8
    }
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
