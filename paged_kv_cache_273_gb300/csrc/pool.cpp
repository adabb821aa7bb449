// Host side of libpkv: the shared block pool, its free list and reference
// counts, slot bookkeeping, argument validation, and the device error word.
//
// The block pool follows the KV cache visualization page, "PagedAttention:
// the cache in blocks": fixed-size blocks from one shared pool, a block table
// per request, a new block only when the last one is full, and shared prefix
// blocks.  Blocks are reclaimed when their last reference goes away
// (jovanaeducation.com/guides/l-is-2, "Paging: borrow the trick operating
// systems already use").

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <new>
#include <unordered_map>

#include "pkv_internal.h"

namespace {

// An NVTX range around an entry point's host work and launches, so that a
// timeline profiler shows the library's calls by name (a no-op when no
// profiler is attached).
struct Range {
    explicit Range(const char *name) { nvtxRangePushA(name); }
    ~Range() { nvtxRangePop(); }
    Range(const Range &) = delete;
    Range &operator=(const Range &) = delete;
};

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

extern "C" {

const char *pkv_status_string(int status)
{
    switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID: return "invalid argument";
    case PKV_ERR_NO_BLOCKS: return "not enough free blocks";
    case PKV_ERR_CUDA: return "CUDA error or no device";
    case PKV_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case PKV_ERR_BAD_INDEX: return "slot, block id or sequence length out of range";
    case PKV_ERR_TIMEOUT: return "bounded device wait timed out";
    default: return "unknown status";
    }
}

int kv_block_pool_init(pkv_pool **out, int num_blocks, int block_size, int num_kv_heads,
                       int head_dim, pkv_dtype kv_dtype)
{
    if (!out)
        return PKV_ERR_INVALID;
    *out = nullptr;
    if (num_blocks < 1 || num_kv_heads < 1 || !is_pow2(block_size) || block_size > 256)
        return PKV_ERR_INVALID;
    if ((int64_t)num_blocks * block_size >= ((int64_t)1 << 31))
        return PKV_ERR_INVALID;
    if (kv_dtype != PKV_F32 && kv_dtype != PKV_F16 && kv_dtype != PKV_BF16 &&
        kv_dtype != PKV_I8 && kv_dtype != PKV_I4)
        return PKV_ERR_INVALID;
    if (head_dim != 64 && head_dim != 128)
        return PKV_ERR_UNSUPPORTED;
    if (kv_dtype == PKV_I4 && head_dim != 128)
        return PKV_ERR_UNSUPPORTED;
    if (block_size < 4 || (pkv::quantized_dtype(kv_dtype) && block_size < 8))
        return PKV_ERR_UNSUPPORTED;

    pkv_pool *p = new (std::nothrow) pkv_pool;
    if (!p)
        return PKV_ERR_INVALID;
    p->num_blocks = num_blocks;
    p->block_size = block_size;
    p->num_kv_heads = num_kv_heads;
    p->head_dim = head_dim;
    p->kv_dtype = kv_dtype;
    p->refcount.assign(num_blocks, 0);
    p->free_stack.resize(num_blocks);
    for (int i = 0; i < num_blocks; ++i)          // pops yield 0, 1, 2, ...
        p->free_stack[i] = num_blocks - 1 - i;

    int dev = -1;
    if (cudaGetDevice(&dev) == cudaSuccess) {
        cudaDeviceProp prop;
        unsigned int *err = nullptr;
        if (cudaGetDeviceProperties(&prop, dev) == cudaSuccess &&
            cudaMalloc(&err, sizeof(unsigned int)) == cudaSuccess) {
            if (cudaMemset(err, 0, sizeof(unsigned int)) == cudaSuccess) {
                p->has_device = true;
                p->device = dev;
                p->num_sms = prop.multiProcessorCount;
                p->max_smem_optin = (int)prop.sharedMemPerBlockOptin;
                p->d_err = err;
            } else {
                cudaFree(err);
            }
        }
    }
    cudaGetLastError();  // a missing device is not sticky for the caller
    *out = p;
    return PKV_OK;
}

void kv_block_pool_destroy(pkv_pool *pool)
{
    if (!pool)
        return;
    if (pool->d_err)
        cudaFree(pool->d_err);
    delete pool;
}

size_t kv_cache_bytes(const pkv_pool *pool)
{
    if (!pool)
        return 0;
    return (size_t)pool->num_blocks * pool->num_kv_heads * pool->block_size *
           (size_t)pkv::row_bytes(pool->kv_dtype, pool->head_dim);
}

size_t kv_scales_bytes(const pkv_pool *pool)
{
    if (!pool || !pkv::quantized_dtype(pool->kv_dtype))
        return 0;
    return (size_t)pool->num_blocks * pool->num_kv_heads * pool->block_size * 2;
}

int kv_num_free_blocks(const pkv_pool *pool)
{
    return pool ? (int)pool->free_stack.size() : PKV_ERR_INVALID;
}

int kv_block_refcount(const pkv_pool *pool, int32_t id)
{
    if (!pool || id < 0 || id >= pool->num_blocks)
        return PKV_ERR_INVALID;
    return pool->refcount[id];
}

int kv_block_alloc(pkv_pool *pool, int n, int32_t *out_ids)
{
    if (!pool || n < 0 || (n > 0 && !out_ids))
        return PKV_ERR_INVALID;
    if ((size_t)n > pool->free_stack.size())
        return PKV_ERR_NO_BLOCKS;
    for (int i = 0; i < n; ++i) {
        int32_t id = pool->free_stack.back();
        pool->free_stack.pop_back();
        pool->refcount[id] = 1;
        out_ids[i] = id;
    }
    return PKV_OK;
}

int kv_block_share(pkv_pool *pool, const int32_t *ids, int n)
{
    if (!pool || n < 0 || (n > 0 && !ids))
        return PKV_ERR_INVALID;
    for (int i = 0; i < n; ++i)
        if (ids[i] < 0 || ids[i] >= pool->num_blocks || pool->refcount[ids[i]] <= 0)
            return PKV_ERR_INVALID;
    for (int i = 0; i < n; ++i)
        ++pool->refcount[ids[i]];
    return PKV_OK;
}

int kv_block_free(pkv_pool *pool, const int32_t *ids, int n)
{
    if (!pool || n < 0 || (n > 0 && !ids))
        return PKV_ERR_INVALID;
    std::unordered_map<int32_t, int> drops;
    for (int i = 0; i < n; ++i) {
        if (ids[i] < 0 || ids[i] >= pool->num_blocks)
            return PKV_ERR_INVALID;
        if (++drops[ids[i]] > pool->refcount[ids[i]])
            return PKV_ERR_INVALID;               // double free / underflow
    }
    for (int i = 0; i < n; ++i) {
        int32_t id = ids[i];
        if (--pool->refcount[id] == 0)
            pool->free_stack.push_back(id);
    }
    return PKV_OK;
}

int kv_slot_mapping(const int32_t *block_tables, int max_blocks_per_seq, int block_size,
                    int batch, const int32_t *start, const int32_t *num_new,
                    int32_t *slot_mapping)
{
    if (batch < 0 || max_blocks_per_seq < 0 || block_size < 1 || (batch > 0 && (!start || !block_tables)))
        return PKV_ERR_INVALID;
    int64_t k = 0;
    for (int b = 0; b < batch; ++b) {
        int n = num_new ? num_new[b] : 1;
        if (start[b] < 0 || n < 0)
            return PKV_ERR_INVALID;
        if (n > 0 && !slot_mapping)
            return PKV_ERR_INVALID;
        if ((int64_t)start[b] + n > (int64_t)max_blocks_per_seq * block_size)
            return PKV_ERR_INVALID;
        const int32_t *row = block_tables + (int64_t)b * max_blocks_per_seq;
        for (int j = 0; j < n; ++j) {
            int64_t pos = (int64_t)start[b] + j;
            int64_t slot = (int64_t)row[pos / block_size] * block_size + pos % block_size;
            slot_mapping[k++] = (int32_t)slot;
        }
    }
    return PKV_OK;
}

int kv_reserve_slots(pkv_pool *pool, int batch, const int32_t *seq_lens, const int32_t *num_new,
                     int32_t *block_tables, int max_blocks_per_seq, int32_t *slot_mapping)
{
    if (!pool || batch < 0 || max_blocks_per_seq < 0 ||
        (batch > 0 && (!seq_lens || !block_tables)))
        return PKV_ERR_INVALID;
    const int bs = pool->block_size;
    int64_t need = 0, total_new = 0;
    for (int b = 0; b < batch; ++b) {
        int n = num_new ? num_new[b] : 1;
        if (seq_lens[b] < 0 || n < 0)
            return PKV_ERR_INVALID;
        int64_t before = ceil_div(seq_lens[b], bs);
        int64_t after = ceil_div((int64_t)seq_lens[b] + n, bs);
        if (after > max_blocks_per_seq)
            return PKV_ERR_INVALID;
        need += after - before;
        total_new += n;
    }
    if (total_new > 0 && !slot_mapping)
        return PKV_ERR_INVALID;
    if (need > (int64_t)pool->free_stack.size())
        return PKV_ERR_NO_BLOCKS;
    int64_t k = 0;
    for (int b = 0; b < batch; ++b) {
        int n = num_new ? num_new[b] : 1;
        int32_t *row = block_tables + (int64_t)b * max_blocks_per_seq;
        for (int j = 0; j < n; ++j) {
            int64_t pos = (int64_t)seq_lens[b] + j;
            if (pos % bs == 0) {                  // first token of a new block
                int32_t id;
                kv_block_alloc(pool, 1, &id);     // cannot fail: counted above
                row[pos / bs] = id;
            }
            slot_mapping[k++] = (int32_t)((int64_t)row[pos / bs] * bs + pos % bs);
        }
    }
    return PKV_OK;
}

int kv_reserve_slots_cow(pkv_pool *pool, int batch, const int32_t *seq_lens,
                         const int32_t *num_new, int32_t *block_tables, int max_blocks_per_seq,
                         int32_t *slot_mapping, int32_t *copy_src, int32_t *copy_dst,
                         int *num_copies)
{
    if (!pool || batch < 0 || max_blocks_per_seq < 0 || !num_copies ||
        (batch > 0 && (!seq_lens || !block_tables || !copy_src || !copy_dst)))
        return PKV_ERR_INVALID;
    const int bs = pool->block_size;
    // First pass: validate and count the blocks the step needs, playing the
    // reference drops of earlier copies forward so that the count is exact.
    std::unordered_map<int32_t, int> dropped;
    int64_t need = 0, total_new = 0;
    for (int b = 0; b < batch; ++b) {
        const int n = num_new ? num_new[b] : 1;
        if (seq_lens[b] < 0 || n < 0)
            return PKV_ERR_INVALID;
        const int64_t before = ceil_div(seq_lens[b], bs);
        const int64_t after = ceil_div((int64_t)seq_lens[b] + n, bs);
        if (after > max_blocks_per_seq)
            return PKV_ERR_INVALID;
        need += after - before;
        total_new += n;
        if (n > 0 && seq_lens[b] % bs != 0) {      // writes into its last block
            const int32_t id = block_tables[(int64_t)b * max_blocks_per_seq + seq_lens[b] / bs];
            if (id < 0 || id >= pool->num_blocks || pool->refcount[id] <= 0)
                return PKV_ERR_INVALID;
            int &d = dropped[id];
            if (pool->refcount[id] - d > 1) {
                ++need;
                ++d;
            }
        }
    }
    if (total_new > 0 && !slot_mapping)
        return PKV_ERR_INVALID;
    if (need > (int64_t)pool->free_stack.size())
        return PKV_ERR_NO_BLOCKS;
    // Second pass: copies, new blocks and slots.
    int copies = 0;
    int64_t k = 0;
    for (int b = 0; b < batch; ++b) {
        const int n = num_new ? num_new[b] : 1;
        int32_t *row = block_tables + (int64_t)b * max_blocks_per_seq;
        if (n > 0 && seq_lens[b] % bs != 0) {
            int32_t &entry = row[seq_lens[b] / bs];
            if (pool->refcount[entry] > 1) {
                int32_t fresh;
                kv_block_alloc(pool, 1, &fresh);    // cannot fail: counted above
                copy_src[copies] = entry;
                copy_dst[copies] = fresh;
                ++copies;
                --pool->refcount[entry];            // still held by the others
                entry = fresh;
            }
        }
        for (int j = 0; j < n; ++j) {
            const int64_t pos = (int64_t)seq_lens[b] + j;
            if (pos % bs == 0) {
                int32_t id;
                kv_block_alloc(pool, 1, &id);       // cannot fail: counted above
                row[pos / bs] = id;
            }
            slot_mapping[k++] = (int32_t)((int64_t)row[pos / bs] * bs + pos % bs);
        }
    }
    *num_copies = copies;
    return PKV_OK;
}

// ---------------------------------------------------------------- device calls

int kv_block_copy(const pkv_pool *pool, const int32_t *src, const int32_t *dst, int n,
                  void *k_cache, void *v_cache, void *k_scales, void *v_scales,
                  pkv_stream_t stream)
{
    Range range("pkv.kv_block_copy");
    if (!pool || n < 0)
        return PKV_ERR_INVALID;
    if (n == 0)
        return PKV_OK;
    if (!src || !dst || !k_cache || !v_cache || (reinterpret_cast<uintptr_t>(src) & 3u) ||
        (reinterpret_cast<uintptr_t>(dst) & 3u) || !pkv::aligned16(k_cache) ||
        !pkv::aligned16(v_cache))
        return PKV_ERR_INVALID;
    if (pkv::quantized_dtype(pool->kv_dtype) && (!k_scales || !v_scales ||
                                     (reinterpret_cast<uintptr_t>(k_scales) & 1u) ||
                                     (reinterpret_cast<uintptr_t>(v_scales) & 1u)))
        return PKV_ERR_INVALID;
    if (!pool->has_device)
        return PKV_ERR_CUDA;
    return pkv::launch_block_copy(pool, src, dst, n, k_cache, v_cache, k_scales, v_scales,
                                  stream);
}

namespace {

// kv_append's argument checks (everything but the device).
int append_check(const pkv_pool *pool, const void *k_new, const void *v_new, pkv_dtype in_dtype,
                 const int32_t *slot_mapping, int num_tokens, const void *k_cache,
                 const void *v_cache, const void *k_scales, const void *v_scales)
{
    if (!pool || num_tokens < 0)
        return PKV_ERR_INVALID;
    if (pkv::quantized_dtype(pool->kv_dtype)) {
        if (in_dtype != PKV_F16 && in_dtype != PKV_BF16 && in_dtype != PKV_F32)
            return PKV_ERR_UNSUPPORTED;
    } else if (in_dtype != pool->kv_dtype) {
        return PKV_ERR_INVALID;
    }
    if (num_tokens == 0)
        return PKV_OK;
    if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache)
        return PKV_ERR_INVALID;
    if (!pkv::aligned16(k_new) || !pkv::aligned16(v_new) || !pkv::aligned16(k_cache) ||
        !pkv::aligned16(v_cache) || (reinterpret_cast<uintptr_t>(slot_mapping) & 3u))
        return PKV_ERR_INVALID;
    if (pkv::quantized_dtype(pool->kv_dtype) && (!k_scales || !v_scales || !pkv::aligned16(k_scales) ||
                                     !pkv::aligned16(v_scales)))
        return PKV_ERR_INVALID;
    return PKV_OK;
}

}  // namespace

int kv_append(const pkv_pool *pool, const void *k_new, const void *v_new, pkv_dtype in_dtype,
              const int32_t *slot_mapping, int num_tokens, void *k_cache, void *v_cache,
              void *k_scales, void *v_scales, pkv_stream_t stream)
{
    Range range("pkv.kv_append");
    const int rc = append_check(pool, k_new, v_new, in_dtype, slot_mapping, num_tokens, k_cache,
                                v_cache, k_scales, v_scales);
    if (rc != PKV_OK || num_tokens == 0)
        return rc;
    if (!pool->has_device)
        return PKV_ERR_CUDA;
    return pkv::launch_append(pool, k_new, v_new, in_dtype, slot_mapping, num_tokens, k_cache,
                              v_cache, k_scales, v_scales, stream);
}

size_t paged_decode_workspace_bytes(const pkv_pool *pool, int batch, int num_q_heads)
{
    if (!pool || batch < 0 || num_q_heads < 1 || num_q_heads % pool->num_kv_heads != 0)
        return 0;
    return pkv::decode_workspace_bytes(pool, batch, num_q_heads);
}

namespace {

// The decode calls' argument checks (everything but the device): PKV_OK when
// the call can be launched (or has nothing to do: batch 0).
int decode_check(const pkv_pool *pool, const void *q, pkv_dtype q_dtype, int num_q_heads,
                 const void *k_cache, const void *v_cache, const void *k_scales,
                 const void *v_scales, const int32_t *block_tables, int max_blocks_per_seq,
                 const int32_t *seq_lens, int batch, int max_seq_len, int window,
                 const float *out, const void *workspace, size_t workspace_bytes)
{
    if (window < 0)
        return PKV_ERR_INVALID;
    if (!pool || batch < 0 || max_blocks_per_seq < 0 || max_seq_len < 0 || num_q_heads < 1)
        return PKV_ERR_INVALID;
    if (num_q_heads % pool->num_kv_heads != 0)
        return PKV_ERR_INVALID;
    int G = num_q_heads / pool->num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8)
        return PKV_ERR_UNSUPPORTED;
    if (pkv::quantized_dtype(pool->kv_dtype)) {
        if (q_dtype != PKV_F16 && q_dtype != PKV_BF16)
            return PKV_ERR_UNSUPPORTED;
    } else if (q_dtype != pool->kv_dtype) {
        return PKV_ERR_INVALID;
    }
    if (batch > 4096)
        return PKV_ERR_UNSUPPORTED;
    if (batch == 0)
        return PKV_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !seq_lens || !out || !workspace)
        return PKV_ERR_INVALID;
    if (!pkv::aligned16(q) || !pkv::aligned16(k_cache) || !pkv::aligned16(v_cache) ||
        !pkv::aligned16(out) || !pkv::aligned16(workspace) ||
        (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
        (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
        return PKV_ERR_INVALID;
    if (pkv::quantized_dtype(pool->kv_dtype) && (!k_scales || !v_scales || !pkv::aligned16(k_scales) ||
                                     !pkv::aligned16(v_scales)))
        return PKV_ERR_INVALID;
    if (workspace_bytes < pkv::decode_workspace_bytes(pool, batch, num_q_heads))
        return PKV_ERR_INVALID;
    return PKV_OK;
}

int decode_call(const pkv_pool *pool, const void *q, pkv_dtype q_dtype, int num_q_heads,
                const void *k_cache, const void *v_cache, const void *k_scales,
                const void *v_scales, const int32_t *block_tables, int max_blocks_per_seq,
                const int32_t *seq_lens, int batch, int max_seq_len, int window, float scale,
                float *out, void *workspace, size_t workspace_bytes, pkv_stream_t stream)
{
    const int rc = decode_check(pool, q, q_dtype, num_q_heads, k_cache, v_cache, k_scales,
                                v_scales, block_tables, max_blocks_per_seq, seq_lens, batch,
                                max_seq_len, window, out, workspace, workspace_bytes);
    if (rc != PKV_OK || batch == 0)
        return rc;
    if (!pool->has_device)
        return PKV_ERR_CUDA;
    return pkv::launch_decode(pool, q, q_dtype, num_q_heads, k_cache, v_cache, k_scales, v_scales,
                              block_tables, max_blocks_per_seq, seq_lens, batch, max_seq_len,
                              window, scale, out, workspace, workspace_bytes, stream);
}

}  // namespace

int paged_decode_attention(const pkv_pool *pool, const void *q, pkv_dtype q_dtype,
                           int num_q_heads, const void *k_cache, const void *v_cache,
                           const void *k_scales, const void *v_scales,
                           const int32_t *block_tables, int max_blocks_per_seq,
                           const int32_t *seq_lens, int batch, int max_seq_len, float scale,
                           float *out, void *workspace, size_t workspace_bytes,
                           pkv_stream_t stream)
{
    Range range("pkv.paged_decode_attention");
    return decode_call(pool, q, q_dtype, num_q_heads, k_cache, v_cache, k_scales, v_scales,
                       block_tables, max_blocks_per_seq, seq_lens, batch, max_seq_len, 0, scale,
                       out, workspace, workspace_bytes, stream);
}

namespace {

// [off, off + bytes) inside [0, total) and off a multiple of align
bool region_ok(size_t off, size_t bytes, size_t total, size_t align)
{
    return off % align == 0 && off <= total && bytes <= total - off;
}

// The device address of page-locked host memory (its mapping into the device
// address space), or null for other memory, and for page-locked memory that
// another device's context allocated (it need not be mapped for this one).
void *mapped_host(const void *p)
{
    cudaPointerAttributes a{};
    int dev = -1;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess || cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();   // clear the error these queries may leave
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost && a.device == dev ? a.devicePointer : nullptr;
}

// Copy between host and device memory for the step: page-locked host memory
// in whole 16-byte chunks goes through the staging kernel (programmatic
// dependent launch keeps the stream's kernels overlapping), other memory
// through cudaMemcpyAsync.
int step_copy(const void *src, void *dst, size_t bytes, bool to_device, cudaStream_t s)
{
    const void *hs = to_device ? mapped_host(src) : src;
    void *hd = to_device ? dst : mapped_host(dst);
    if (hs && hd && bytes % 16 == 0 && pkv::aligned16(hs) && pkv::aligned16(hd))
        return pkv::launch_stage_copy(hs, hd, bytes, to_device,
                                      reinterpret_cast<pkv_stream_t>(s));
    return cudaMemcpyAsync(dst, src, bytes,
                           to_device ? cudaMemcpyHostToDevice : cudaMemcpyDeviceToHost,
                           s) == cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
}

}  // namespace

int paged_decode_step(const pkv_pool *pool, const void *host_in, void *dev_in, size_t in_bytes,
                      const pkv_step_layout *layout, pkv_dtype in_dtype, pkv_dtype q_dtype,
                      int num_q_heads, void *k_cache, void *v_cache, void *k_scales,
                      void *v_scales, const int32_t *block_tables, int max_blocks_per_seq,
                      int batch, int max_seq_len, float scale, float *out, float *host_out,
                      void *workspace, size_t workspace_bytes, pkv_stream_t stream)
{
    Range range("pkv.paged_decode_step");
    if (!pool || !layout || batch < 0 || num_q_heads < 1 ||
        num_q_heads % pool->num_kv_heads != 0)
        return PKV_ERR_INVALID;
    if (in_dtype != PKV_F32 && in_dtype != PKV_F16 && in_dtype != PKV_BF16)
        return PKV_ERR_INVALID;
    if (q_dtype != PKV_F32 && q_dtype != PKV_F16 && q_dtype != PKV_BF16)
        return PKV_ERR_INVALID;
    if (batch == 0)
        return PKV_OK;
    if (!host_in || !dev_in || !pkv::aligned16(dev_in))
        return PKV_ERR_INVALID;
    const size_t B = (size_t)batch;
    const size_t kv_bytes =
        B * pool->num_kv_heads * pool->head_dim * (size_t)pkv::dtype_bytes(in_dtype);
    const size_t q_bytes = B * num_q_heads * pool->head_dim * (size_t)pkv::dtype_bytes(q_dtype);
    if (!region_ok(layout->k_new, kv_bytes, in_bytes, 16) ||
        !region_ok(layout->v_new, kv_bytes, in_bytes, 16) ||
        !region_ok(layout->q, q_bytes, in_bytes, 16) ||
        !region_ok(layout->slot_mapping, B * 4, in_bytes, 4) ||
        !region_ok(layout->seq_lens, B * 4, in_bytes, 4))
        return PKV_ERR_INVALID;
    // the append's and the attention's own checks, before any device work
    unsigned char *d = static_cast<unsigned char *>(dev_in);
    const int32_t *slots = reinterpret_cast<const int32_t *>(d + layout->slot_mapping);
    const int32_t *lens = reinterpret_cast<const int32_t *>(d + layout->seq_lens);
    int rc = append_check(pool, d + layout->k_new, d + layout->v_new, in_dtype, slots, batch,
                          k_cache, v_cache, k_scales, v_scales);
    if (rc == PKV_OK)
        rc = decode_check(pool, d + layout->q, q_dtype, num_q_heads, k_cache, v_cache, k_scales,
                          v_scales, block_tables, max_blocks_per_seq, lens, batch, max_seq_len,
                          0, out, workspace, workspace_bytes);
    if (rc != PKV_OK)
        return rc;
    if (!pool->has_device)
        return PKV_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const void *h = mapped_host(host_in);
    if (h && !pkv::quantized_dtype(pool->kv_dtype) && in_bytes % 16 == 0 && pkv::aligned16(h)) {
        // fp cache, page-locked input: the staging copy and the append are one kernel
        rc = pkv::launch_step_in(pool, h, dev_in, in_bytes, layout->k_new, layout->v_new,
                                 layout->slot_mapping, batch, k_cache, v_cache, stream);
        if (rc != PKV_OK)
            return rc;
    } else {
        rc = step_copy(host_in, dev_in, in_bytes, true, s);
        if (rc != PKV_OK)
            return rc;
        rc = kv_append(pool, d + layout->k_new, d + layout->v_new, in_dtype, slots, batch,
                       k_cache, v_cache, k_scales, v_scales, stream);
        if (rc != PKV_OK)
            return rc;
    }
    // a page-locked host_out takes the attention's output directly, through
    // its device mapping (the attention only writes its output)
    void *mapped_out = host_out ? mapped_host(host_out) : nullptr;
    const bool direct = mapped_out && pkv::aligned16(mapped_out);
    rc = paged_decode_attention(pool, d + layout->q, q_dtype, num_q_heads, k_cache, v_cache,
                                k_scales, v_scales, block_tables, max_blocks_per_seq, lens,
                                batch, max_seq_len, scale,
                                direct ? static_cast<float *>(mapped_out) : out, workspace,
                                workspace_bytes, stream);
    if (rc != PKV_OK || !host_out || direct)
        return rc;
    const size_t out_bytes = B * num_q_heads * pool->head_dim * sizeof(float);
    return step_copy(out, host_out, out_bytes, false, s);
}

int paged_decode_attention_window(const pkv_pool *pool, const void *q, pkv_dtype q_dtype,
                                  int num_q_heads, const void *k_cache, const void *v_cache,
                                  const void *k_scales, const void *v_scales,
                                  const int32_t *block_tables, int max_blocks_per_seq,
                                  const int32_t *seq_lens, int batch, int max_seq_len,
                                  int window, float scale, float *out, void *workspace,
                                  size_t workspace_bytes, pkv_stream_t stream)
{
    Range range("pkv.paged_decode_attention_window");
    return decode_call(pool, q, q_dtype, num_q_heads, k_cache, v_cache, k_scales, v_scales,
                       block_tables, max_blocks_per_seq, seq_lens, batch, max_seq_len, window,
                       scale, out, workspace, workspace_bytes, stream);
}

int kv_prefix_groups(const int32_t *block_tables, int max_blocks_per_seq, const int32_t *seq_lens,
                     int batch, int block_size, int min_prefix_blocks, int32_t *group_start,
                     int32_t *group_seqs, int32_t *group_prefix, int32_t *seq_prefix,
                     int *num_groups, int *max_group_size, int *max_prefix_len)
{
    if (batch < 0 || max_blocks_per_seq < 0 || block_size < 1 || min_prefix_blocks < 1 ||
        !num_groups || !max_group_size || !max_prefix_len)
        return PKV_ERR_INVALID;
    if (batch > 0 && (!block_tables || !seq_lens || !group_start || !group_seqs ||
                      !group_prefix || !seq_prefix))
        return PKV_ERR_INVALID;
    *num_groups = 0;
    *max_group_size = 0;
    *max_prefix_len = 0;
    if (batch > 0)
        group_start[0] = 0;
    for (int b = 0; b < batch; ++b) {
        seq_prefix[b] = 0;
        if (seq_lens[b] < 0 || (int64_t)seq_lens[b] > (int64_t)max_blocks_per_seq * block_size)
            return PKV_ERR_INVALID;
    }
    // Candidates: sequences with at least min_prefix_blocks whole blocks,
    // ordered by first block id (then by index, so a group lists its
    // members in batch order).
    std::vector<int> cand;
    for (int b = 0; b < batch; ++b)
        if (seq_lens[b] >= min_prefix_blocks * block_size)
            cand.push_back(b);
    std::stable_sort(cand.begin(), cand.end(), [&](int a, int c) {
        return block_tables[(int64_t)a * max_blocks_per_seq] <
               block_tables[(int64_t)c * max_blocks_per_seq];
    });
    int ng = 0, used = 0;
    for (size_t i = 0; i < cand.size();) {
        size_t j = i + 1;
        const int32_t first = block_tables[(int64_t)cand[i] * max_blocks_per_seq];
        while (j < cand.size() && block_tables[(int64_t)cand[j] * max_blocks_per_seq] == first)
            ++j;
        if (j - i >= 2) {
            // the table entries every member shares, within every member's rows
            const int32_t *lead = block_tables + (int64_t)cand[i] * max_blocks_per_seq;
            int minlen = seq_lens[cand[i]];
            for (size_t k = i; k < j; ++k)
                minlen = std::min(minlen, (int)seq_lens[cand[k]]);
            int common = (minlen + block_size - 1) / block_size;
            for (size_t k = i + 1; k < j; ++k) {
                const int32_t *row = block_tables + (int64_t)cand[k] * max_blocks_per_seq;
                int n = 0;
                while (n < common && row[n] == lead[n])
                    ++n;
                common = n;
            }
            const int P = std::min(common * block_size, minlen);
            if (common >= min_prefix_blocks && P > 0) {
                std::vector<int> mem(cand.begin() + i, cand.begin() + j);
                std::sort(mem.begin(), mem.end());
                for (int m : mem) {
                    group_seqs[used++] = m;
                    seq_prefix[m] = P;
                }
                group_prefix[ng] = P;
                group_start[ng + 1] = used;
                *max_group_size = std::max(*max_group_size, (int)mem.size());
                *max_prefix_len = std::max(*max_prefix_len, P);
                ++ng;
            }
        }
        i = j;
    }
    *num_groups = ng;
    return PKV_OK;
}

size_t paged_decode_cascade_workspace_bytes(const pkv_pool *pool, int batch, int num_q_heads,
                                            int max_prefix_len)
{
    if (!pool || batch < 0 || num_q_heads < 1 || num_q_heads % pool->num_kv_heads != 0 ||
        max_prefix_len < 0)
        return 0;
    const size_t dec = pkv::decode_workspace_bytes(pool, batch, num_q_heads);
    return (dec + 255) / 256 * 256 +
           pkv::prefix_partials_bytes(pool, batch, num_q_heads, max_prefix_len);
}

int paged_decode_attention_cascade(const pkv_pool *pool, const void *q, pkv_dtype q_dtype,
                                   int num_q_heads, const void *k_cache, const void *v_cache,
                                   const int32_t *block_tables, int max_blocks_per_seq,
                                   const int32_t *seq_lens, int batch, int max_seq_len,
                                   const int32_t *group_start, const int32_t *group_seqs,
                                   const int32_t *group_prefix, const int32_t *seq_prefix,
                                   int num_groups, int max_group_size, int max_prefix_len,
                                   float scale, float *out, void *workspace,
                                   size_t workspace_bytes, pkv_stream_t stream)
{
    Range range("pkv.paged_decode_attention_cascade");
    if (!pool || batch < 0 || max_blocks_per_seq < 0 || max_seq_len < 0 || num_q_heads < 1 ||
        num_groups < 0 || max_group_size < 0 || max_prefix_len < 0)
        return PKV_ERR_INVALID;
    if (num_q_heads % pool->num_kv_heads != 0)
        return PKV_ERR_INVALID;
    const int G = num_q_heads / pool->num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8)
        return PKV_ERR_UNSUPPORTED;
    // the prefix pass multiplies q and K on the tensor cores as they are
    if (pool->kv_dtype != PKV_F16 && pool->kv_dtype != PKV_BF16)
        return PKV_ERR_UNSUPPORTED;
    if (q_dtype != pool->kv_dtype)
        return PKV_ERR_INVALID;
    if (batch > 4096 || max_group_size > batch || max_prefix_len > max_seq_len)
        return batch > 4096 ? PKV_ERR_UNSUPPORTED : PKV_ERR_INVALID;
    if (batch == 0)
        return PKV_OK;
    if (num_groups > 0 && (!group_start || !group_seqs || !group_prefix))
        return PKV_ERR_INVALID;
    if (!q || !k_cache || !v_cache || !block_tables || !seq_lens || !seq_prefix || !out ||
        !workspace)
        return PKV_ERR_INVALID;
    if (!pkv::aligned16(q) || !pkv::aligned16(k_cache) || !pkv::aligned16(v_cache) ||
        !pkv::aligned16(out) || !pkv::aligned16(workspace) ||
        (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
        (reinterpret_cast<uintptr_t>(seq_lens) & 3u) ||
        (reinterpret_cast<uintptr_t>(seq_prefix) & 3u))
        return PKV_ERR_INVALID;
    if (!pool->has_device)
        return PKV_ERR_CUDA;
    if (workspace_bytes <
        paged_decode_cascade_workspace_bytes(pool, batch, num_q_heads, max_prefix_len))
        return PKV_ERR_INVALID;
    // workspace: decode's counters and partials | the prefix partials
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    const size_t dec = (pkv::decode_workspace_bytes(pool, batch, num_q_heads) + 255) / 256 * 256;
    float *part = reinterpret_cast<float *>(ws + dec);
    if (num_groups > batch)
        return PKV_ERR_INVALID;
    if (num_groups > 0 && max_group_size > 0 && max_prefix_len > 0) {
        int kc = 1;
        int rc = pkv::launch_prefix_pass(pool, q, num_q_heads, k_cache, v_cache, block_tables,
                                         max_blocks_per_seq, seq_lens, batch, group_start,
                                         group_seqs, group_prefix, num_groups, max_group_size,
                                         max_prefix_len, scale, part, &kc, stream);
        if (rc == PKV_OK)
            rc = pkv::launch_prefix_merge(pool, seq_prefix, part, batch, num_q_heads, kc, stream);
        if (rc != PKV_OK)
            return rc;
    }
    return pkv::launch_decode(pool, q, q_dtype, num_q_heads, k_cache, v_cache, nullptr, nullptr,
                              block_tables, max_blocks_per_seq, seq_lens, batch, max_seq_len, 0,
                              scale, out, workspace, dec, stream, seq_prefix, part);
}

int paged_prefill_attention(const pkv_pool *pool, const void *q, int num_q_heads,
                            const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *q_start, const int32_t *seq_lens, int batch,
                            int max_q_len, float scale, float *out, pkv_stream_t stream)
{
    Range range("pkv.paged_prefill_attention");
    if (!pool || batch < 0 || max_blocks_per_seq < 0 || max_q_len < 0 || num_q_heads < 1 ||
        num_q_heads % pool->num_kv_heads != 0)
        return PKV_ERR_INVALID;
    if (pool->kv_dtype != PKV_F16 && pool->kv_dtype != PKV_BF16)
        return PKV_ERR_UNSUPPORTED;
    if (batch > 65535 || num_q_heads > 65535)
        return PKV_ERR_UNSUPPORTED;
    if (batch == 0 || max_q_len == 0)
        return PKV_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !q_start || !seq_lens || !out)
        return PKV_ERR_INVALID;
    if (!pkv::aligned16(q) || !pkv::aligned16(k_cache) || !pkv::aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(out) & 7u) ||
        (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
        (reinterpret_cast<uintptr_t>(q_start) & 3u) ||
        (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
        return PKV_ERR_INVALID;
    if (!pool->has_device)
        return PKV_ERR_CUDA;
    return pkv::launch_prefill(pool, q, num_q_heads, k_cache, v_cache, block_tables,
                               max_blocks_per_seq, q_start, seq_lens, batch, max_q_len, scale,
                               out, stream);
}

int pkv_selftest_wait_timeout(const pkv_pool *pool, pkv_stream_t stream)
{
    if (!pool)
        return PKV_ERR_INVALID;
    if (!pool->has_device)
        return PKV_ERR_CUDA;
    return pkv::launch_selftest_wait_timeout(pool, stream);
}

int pkv_check_error(const pkv_pool *pool, pkv_stream_t stream)
{
    if (!pool)
        return PKV_ERR_INVALID;
    if (!pool->has_device)
        return PKV_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned int h = 0;
    if (cudaMemcpyAsync(&h, pool->d_err, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (h == 0)
        return PKV_OK;
    if (cudaMemsetAsync(pool->d_err, 0, sizeof(unsigned int), s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (h & PKV_EBIT_TIMEOUT)
        return PKV_ERR_TIMEOUT;
    return PKV_ERR_BAD_INDEX;
}

}  // extern "C"
