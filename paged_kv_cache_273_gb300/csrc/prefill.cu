// paged_prefill_attention: causal attention of a batch of new tokens over the
// paged cache (the new tokens' K and V already appended).
//
// KV cache visualization page, "Prefill and decode feel different": prefill
// handles all prompt tokens at once and is bound by arithmetic, not by bytes,
// so it runs on the tensor cores.  Token i of the n_b new tokens of sequence
// b sits at position p = seq_lens[b] - n_b + i and attends over positions
// 0..p ("KV cache: the engine behind fast LLM inference", "Concept").
//
// FlashAttention-style tiles ("Flash attention: don't build the giant
// matrix" in the guide): a CTA of 4 warps takes 64 queries of one (sequence,
// query head); each warp owns 16 query rows.  Key tiles of 64 rows stream
// through shared memory (16-byte async copies, each row found through the
// block table, double buffered); S = Q K^T and O += P V run as
// mma.sync m16n8k16 (fp16 or bf16 in, fp32 accumulate), the online softmax
// stays in registers and P is fed back as the A operand without a trip
// through shared memory.

#include <cuda_runtime.h>

#include "device_common.cuh"

namespace pkv {
namespace {

using namespace dev;

constexpr int BQ = 64;         // queries per CTA
constexpr int BK = 64;         // keys per tile
constexpr int NWARP = 4;

template <int D>
struct PCfg {
    static constexpr int LD = D + 8;                 // padded smem row (elements): conflict-free ldmatrix
    static constexpr int TILE_ELEMS = 64 * LD;
    static constexpr int SMEM_BYTES = (1 + 2 * 2) * TILE_ELEMS * 2;   // Q, K x2, V x2
    static constexpr int CHUNKS = D / 8;             // 16-byte chunks per row
};

template <typename T> struct MmaType;
template <> struct MmaType<__half> { static constexpr bool bf16 = false; };
template <> struct MmaType<__nv_bfloat16> { static constexpr bool bf16 = true; };

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, bool valid)
{
    const uint32_t s = smem_addr(smem);
    const int n = valid ? 16 : 0;             // 0: fill the 16 bytes with zeros
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(n)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void *p)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_addr(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void *p)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_addr(p)));
}

// d (16x8 fp32) += a (16x16) * b (16x8), row.col.
template <bool BF16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1)
{
    if constexpr (BF16) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
}

template <typename T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    if constexpr (MmaType<T>::bf16) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<const uint32_t *>(&h);
    } else {
        const __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t *>(&h);
    }
}

struct PrefillParams {
    const void *q;
    const void *k_cache;
    const void *v_cache;
    const int32_t *block_tables;
    const int32_t *q_start;
    const int32_t *seq_lens;
    float *out;
    unsigned int *err;
    int batch, num_q_heads, num_kv_heads, block_size, max_blocks_per_seq, num_blocks;
    float scale_log2;
};

template <int D, typename T>
__global__ void __launch_bounds__(NWARP * 32) paged_prefill_kernel(const PrefillParams p)
{
    using C = PCfg<D>;
    constexpr bool BF16 = MmaType<T>::bf16;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    T *sQ = reinterpret_cast<T *>(smem_raw);
    T *sK = sQ + C::TILE_ELEMS;                 // two buffers
    T *sV = sK + 2 * C::TILE_ELEMS;             // two buffers

    grid_dependency_wait();
    grid_dependents_launch();

    const int b = blockIdx.z;
    const int h = blockIdx.y;
    const int qt = gridDim.x - 1 - blockIdx.x;  // long (late) query tiles first
    const int q0 = __ldg(p.q_start + b);
    const int n = __ldg(p.q_start + b + 1) - q0;
    const int L = __ldg(p.seq_lens + b);
    if (qt * BQ >= n)
        return;
    if (n < 0 || L < n || L > p.max_blocks_per_seq * p.block_size) {
        if (threadIdx.x == 0 && qt == 0 && h == 0)
            atomicOr(p.err, PKV_EBIT_SEQLEN);
        return;
    }
    const int G = p.num_q_heads / p.num_kv_heads;
    const int kvh = h / G;
    const int base = L - n;                        // position of new token 0
    const int rows = min(BQ, n - qt * BQ);         // valid query rows of this tile
    const int last_pos = base + qt * BQ + rows - 1;
    const int ntiles = last_pos / BK + 1;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t *table = p.block_tables + (int64_t)b * p.max_blocks_per_seq;
    const T *qg = static_cast<const T *>(p.q);
    const T *kg = static_cast<const T *>(p.k_cache);
    const T *vg = static_cast<const T *>(p.v_cache);

    // ---- async loads: Q once, K/V tiles double buffered
    for (int idx = tid; idx < BQ * C::CHUNKS; idx += NWARP * 32) {
        const int r = idx / C::CHUNKS, c = idx % C::CHUNKS;
        const bool ok = r < rows;
        const T *src = qg + ((int64_t)(q0 + qt * BQ + (ok ? r : 0)) * p.num_q_heads + h) * D + c * 8;
        cp_async16(sQ + r * C::LD + c * 8, src, ok);
    }
    auto load_kv = [&](int kt, int buf) {
        for (int idx = tid; idx < BK * C::CHUNKS; idx += NWARP * 32) {
            const int r = idx / C::CHUNKS, c = idx % C::CHUNKS;
            const int pos = kt * BK + r;
            bool ok = pos <= last_pos;
            int64_t row = 0;
            if (ok) {
                const int32_t blk = __ldg(table + pos / p.block_size);
                if (blk < 0 || blk >= p.num_blocks) {
                    atomicOr(p.err, PKV_EBIT_BLOCK);
                    ok = false;
                } else {
                    row = ((int64_t)blk * p.num_kv_heads + kvh) * p.block_size + pos % p.block_size;
                }
            }
            cp_async16(sK + buf * C::TILE_ELEMS + r * C::LD + c * 8, kg + row * D + c * 8, ok);
            cp_async16(sV + buf * C::TILE_ELEMS + r * C::LD + c * 8, vg + row * D + c * 8, ok);
        }
    };
    load_kv(0, 0);
    cp_async_commit();

    // Per thread: query rows r0 = 16*warp + lane/4 and r0 + 8.
    const int r0 = warp * 16 + (lane >> 2);
    const int qpos0 = base + qt * BQ + min(r0, rows - 1);        // padding rows copy a valid one
    const int qpos1 = base + qt * BQ + min(r0 + 8, rows - 1);

    float o[D / 8][4];
#pragma unroll
    for (int j = 0; j < D / 8; ++j)
        o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.0f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
    uint32_t qf[D / 16][4];

    for (int kt = 0; kt < ntiles; ++kt) {
        const int buf = kt & 1;
        if (kt + 1 < ntiles) {
            load_kv(kt + 1, buf ^ 1);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        if (kt == 0) {
            // Q fragments: rows 16*warp .. +15, all of D, kept in registers
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                ldsm_x4(qf[ks], sQ + (warp * 16 + (lane & 15)) * C::LD + ks * 16 + (lane >> 4) * 8);
        }
        const T *Kt = sK + buf * C::TILE_ELEMS;
        const T *Vt = sV + buf * C::TILE_ELEMS;

        // ---- S = Q K^T for 64 keys: 8 n-tiles of 8 keys
        float s[8][4];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.0f;
#pragma unroll
        for (int np = 0; np < 4; ++np) {          // pairs of n-tiles (16 keys)
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                uint32_t kb[4];
                ldsm_x4(kb, Kt + (np * 16 + (lane & 7) + ((lane >> 4) << 3)) * C::LD + ks * 16 +
                                ((lane >> 3) & 1) * 8);
                mma16816<BF16>(s[2 * np], qf[ks], kb[0], kb[1]);
                mma16816<BF16>(s[2 * np + 1], qf[ks], kb[2], kb[3]);
            }
        }
        // ---- scale, causal mask, online softmax (rows r0 and r0 + 8)
        float mx0 = m0, mx1 = m1;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int key = kt * BK + j * 8 + 2 * (lane & 3);
            s[j][0] = key <= qpos0 ? s[j][0] * p.scale_log2 : -INFINITY;
            s[j][1] = key + 1 <= qpos0 ? s[j][1] * p.scale_log2 : -INFINITY;
            s[j][2] = key <= qpos1 ? s[j][2] * p.scale_log2 : -INFINITY;
            s[j][3] = key + 1 <= qpos1 ? s[j][3] * p.scale_log2 : -INFINITY;
            mx0 = fmaxf(mx0, fmaxf(s[j][0], s[j][1]));
            mx1 = fmaxf(mx1, fmaxf(s[j][2], s[j][3]));
        }
#pragma unroll
        for (int off = 1; off <= 2; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(FULL_MASK, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(FULL_MASK, mx1, off));
        }
        // every row sees key 0 in the first tile, so mx0, mx1 are finite
        const float c0 = exp2f(m0 - mx0), c1 = exp2f(m1 - mx1);
        m0 = mx0;
        m1 = mx1;
        float sum0 = 0.0f, sum1 = 0.0f;
        uint32_t pf[4][4];                         // P as A fragments, 4 k-steps of 16 keys
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float p0 = exp2f(s[j][0] - m0), p1 = exp2f(s[j][1] - m0);
            const float p2 = exp2f(s[j][2] - m1), p3 = exp2f(s[j][3] - m1);
            sum0 += p0 + p1;
            sum1 += p2 + p3;
            // n-tile j covers keys 8j..8j+7: k-step j/2, low (j even) or high half
            pf[j >> 1][(j & 1) * 2 + 0] = pack2<T>(p0, p1);
            pf[j >> 1][(j & 1) * 2 + 1] = pack2<T>(p2, p3);
        }
#pragma unroll
        for (int off = 1; off <= 2; off <<= 1) {
            sum0 += __shfl_xor_sync(FULL_MASK, sum0, off);
            sum1 += __shfl_xor_sync(FULL_MASK, sum1, off);
        }
        l0 = l0 * c0 + sum0;
        l1 = l1 * c1 + sum1;
#pragma unroll
        for (int j = 0; j < D / 8; ++j) {
            o[j][0] *= c0;
            o[j][1] *= c0;
            o[j][2] *= c1;
            o[j][3] *= c1;
        }
        // ---- O += P V: 4 k-steps of 16 keys, D/8 n-tiles of 8 dims
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            // A fragment order: (rows 0-7, k 0-7), (rows 8-15, k 0-7), (rows 0-7, k 8-15), (rows 8-15, k 8-15)
            const uint32_t a[4] = {pf[kk][0], pf[kk][1], pf[kk][2], pf[kk][3]};
#pragma unroll
            for (int dp = 0; dp < D / 16; ++dp) {
                uint32_t vb[4];
                ldsm_x4_t(vb, Vt + (kk * 16 + (lane & 15)) * C::LD + dp * 16 + (lane >> 4) * 8);
                mma16816<BF16>(o[2 * dp], a, vb[0], vb[1]);
                mma16816<BF16>(o[2 * dp + 1], a, vb[2], vb[3]);
            }
        }
        __syncthreads();                           // the buffer is refilled next round
    }

    // ---- normalise and store rows r0, r0 + 8 (fp32 [token][head][D])
    const float inv0 = 1.0f / l0, inv1 = 1.0f / l1;
#pragma unroll
    for (int j = 0; j < D / 8; ++j) {
        const int col = j * 8 + 2 * (lane & 3);
        if (r0 < rows) {
            float *dst = p.out + ((int64_t)(q0 + qt * BQ + r0) * p.num_q_heads + h) * D + col;
            *reinterpret_cast<float2 *>(dst) = make_float2(o[j][0] * inv0, o[j][1] * inv0);
        }
        if (r0 + 8 < rows) {
            float *dst = p.out + ((int64_t)(q0 + qt * BQ + r0 + 8) * p.num_q_heads + h) * D + col;
            *reinterpret_cast<float2 *>(dst) = make_float2(o[j][2] * inv1, o[j][3] * inv1);
        }
    }
}

template <int D, typename T>
int launch_prefill_t(const pkv_pool *pool, const PrefillParams &prm, int max_q_len,
                     cudaStream_t s)
{
    using C = PCfg<D>;
    static bool configured = false;
    if (!configured) {
        if (cudaFuncSetAttribute(paged_prefill_kernel<D, T>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::SMEM_BYTES) != cudaSuccess)
            return PKV_ERR_CUDA;
        configured = true;
    }
    const dim3 grid((unsigned)((max_q_len + BQ - 1) / BQ), (unsigned)prm.num_q_heads,
                    (unsigned)prm.batch);
    if (launch_pdl(paged_prefill_kernel<D, T>, grid, dim3(NWARP * 32), (size_t)C::SMEM_BYTES, s,
                   prm) != cudaSuccess)
        return PKV_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace

int launch_prefill(const pkv_pool *pool, const void *q, int num_q_heads, const void *k_cache,
                   const void *v_cache, const int32_t *block_tables, int max_blocks_per_seq,
                   const int32_t *q_start, const int32_t *seq_lens, int batch, int max_q_len,
                   float scale, float *out, pkv_stream_t stream)
{
    PrefillParams prm{};
    prm.q = q;
    prm.k_cache = k_cache;
    prm.v_cache = v_cache;
    prm.block_tables = block_tables;
    prm.q_start = q_start;
    prm.seq_lens = seq_lens;
    prm.out = out;
    prm.err = pool->d_err;
    prm.batch = batch;
    prm.num_q_heads = num_q_heads;
    prm.num_kv_heads = pool->num_kv_heads;
    prm.block_size = pool->block_size;
    prm.max_blocks_per_seq = max_blocks_per_seq;
    prm.num_blocks = pool->num_blocks;
    prm.scale_log2 = (float)((double)scale * 1.4426950408889634);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool bf = pool->kv_dtype == PKV_BF16;
    if (pool->head_dim == 64)
        return bf ? launch_prefill_t<64, __nv_bfloat16>(pool, prm, max_q_len, s)
                  : launch_prefill_t<64, __half>(pool, prm, max_q_len, s);
    return bf ? launch_prefill_t<128, __nv_bfloat16>(pool, prm, max_q_len, s)
              : launch_prefill_t<128, __half>(pool, prm, max_q_len, s);
}

}  // namespace pkv
