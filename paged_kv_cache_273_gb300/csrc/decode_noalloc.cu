// paged_decode_attention_noalloc: the decode-attention call for callers that
// cannot allocate device memory.
//
// paged_decode_attention needs a caller-provided workspace (split-merge
// counters and partial softmax states).  Some callers have no way to get
// one: code running where device allocation is forbidden or would re-enter
// the allocator (an allocator hook, a host callback holding the caching
// allocator's lock), serving loops that promise no allocation after start-up,
// or processes whose device memory is entirely reserved by another runtime's
// memory pool, so that cudaMalloc fails.  This entry point takes the
// workspace from a fixed array in the library's own device image instead.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds its NOALLOC_SCRATCH_BYTES until the process exits, and all
// calls on a device share it.  Host code cannot use the array's name as a
// device address, so the address is looked up once per device with
// cudaGetSymbolAddress (the first call on a device does this; make that call
// before any stream capture) and passed to the unchanged decode path.  The
// address stays valid for the life of the device's context: cudaDeviceReset
// unloads the library's device image with the array, so a process that
// resets a device must not call this entry point on it again.

#include <cuda_runtime.h>

#include <mutex>

#include "pkv_internal.h"

namespace {

constexpr size_t NOALLOC_SCRATCH_BYTES = (size_t)4 << 20;   // 4 MiB
constexpr int MAX_DEVICES = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
void *g_scratch_addr[MAX_DEVICES];   // device address of g_noalloc_scratch, per device

// Device address of the scratch array on the current device (set-up on the
// first call for that device).
int scratch_address(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (dev < 0 || dev >= MAX_DEVICES)
        return PKV_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
            return PKV_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return PKV_OK;
}

}  // namespace

extern "C" int paged_decode_attention_noalloc(
    const pkv_pool *pool, const void *q, pkv_dtype q_dtype, int num_q_heads, const void *k_cache,
    const void *v_cache, const void *k_scales, const void *v_scales, const int32_t *block_tables,
    int max_blocks_per_seq, const int32_t *seq_lens, int batch, int max_seq_len, float scale,
    float *out, pkv_stream_t stream)
{
    if (!pool || batch < 0 || num_q_heads < 1)
        return PKV_ERR_INVALID;
    if (batch == 0)
        return PKV_OK;
    const size_t need = paged_decode_workspace_bytes(pool, batch, num_q_heads);
    if (need == 0)
        return PKV_ERR_INVALID;
    if (need > NOALLOC_SCRATCH_BYTES)
        return PKV_ERR_UNSUPPORTED;          // batch x heads too large for the fixed array
    if (!pool->has_device)
        return PKV_ERR_CUDA;
    void *scratch = nullptr;
    const int rc = scratch_address(&scratch);
    if (rc != PKV_OK)
        return rc;
    // The array keeps whatever the previous call left; the counters must
    // start at zero, so clear the part this call uses (no allocation).
    if (cudaMemsetAsync(scratch, 0, need, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return PKV_ERR_CUDA;
    return paged_decode_attention(pool, q, q_dtype, num_q_heads, k_cache, v_cache, k_scales,
                                  v_scales, block_tables, max_blocks_per_seq, seq_lens, batch,
                                  max_seq_len, scale, out, scratch, NOALLOC_SCRATCH_BYTES,
                                  stream);
}
