// paged_prefill_attention: causal attention of a batch of new tokens over the
// paged cache (the new tokens' K and V already appended).
//
// KV cache visualization page, "Prefill and decode feel different": prefill
// handles all prompt tokens at once and is bound by arithmetic, not by bytes,
// so it runs on the fifth-generation tensor cores.  Token i of the n_b new
// tokens of sequence b sits at position p = seq_lens[b] - n_b + i and attends
// over positions 0..p ("KV cache: the engine behind fast LLM inference",
// "Concept"), in FlashAttention-style tiles that never hold the whole score
// matrix ("Flash attention: don't build the giant matrix" in the guide).

#include <cuda_runtime.h>

#include "device_common.cuh"

namespace pkv {
namespace {

using namespace dev;

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
    int batch, num_q_heads, num_kv_heads, block_size, bs_log2, max_blocks_per_seq, num_blocks;
    float scale_log2;
};

// ---- tcgen05: 128 queries x 64 keys per step
//
// A CTA of 4 warps takes 128 queries of one (sequence, query head); thread
// t owns query row t; two CTAs share an SM.  Q, K and V tiles are brought
// by 16-byte cp.async copies (each key row located through the block table)
// into shared memory in the tensor cores' core-matrix layout (8 rows x 16
// bytes per 128-byte core matrix, no swizzle), K/V double buffered.  S = Q K^T
// (M 128, N 64, K = D) and O += P V (M 128, N = D, K 64) are single-thread
// tcgen05.mma issues with fp32 accumulators in tensor memory: S in columns
// [0, 64), O in [64, 64 + D).  Each thread reads its S row with tcgen05.ld,
// does the online softmax for it, writes its P row (fp16/bf16) back to
// shared memory as the next A operand, and rescales its O row in tensor
// memory when its maximum moved by more than 2^8.

constexpr int TBQ = 128, TBK = 64;

template <int D>
struct TcCfg {
    static constexpr int Q_BYTES = TBQ * D * 2;
    static constexpr int KV_BYTES = TBK * D * 2;
    static constexpr int P_BYTES = TBQ * TBK * 2;
    static constexpr int SMEM_BYTES = Q_BYTES + 4 * KV_BYTES + P_BYTES + 64;
    static constexpr int TMEM_COLS = 256;          // S: 64 columns, O: D <= 128 columns
};

// Byte offset of the 16-byte chunk c (8 elements along the contiguous
// dimension) of row r in a core-matrix tile whose rows hold `chunks` chunks.
__device__ __forceinline__ uint32_t core_off(int r, int c, int chunks)
{
    return (uint32_t)(((r >> 3) * chunks + c) * 128 + (r & 7) * 16);
}

// Shared-memory matrix descriptor: start, stride between core matrices along
// K (lbo) and along M/N (sbo), descriptor version 1, no swizzle.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46);
}

// Instruction descriptor of kind::f16: fp32 accumulate, A/B fp16 (0) or
// bf16 (1), A K-major, B K-major (b_mn = 0) or MN-major (1), N, M = 128.
__device__ __forceinline__ uint32_t umma_idesc(uint32_t ab, uint32_t b_mn, uint32_t n)
{
    return (1u << 4) | (ab << 7) | (ab << 10) | (b_mn << 16) | ((n >> 3) << 17) |
           ((uint32_t)(TBQ >> 4) << 24);
}

__device__ __forceinline__ void umma_f16(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t idesc,
                                         uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
                 "l"(da), "l"(db), "r"(idesc), "r"(accumulate)
                 : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(bar))
                 : "memory");
}

// 2^x with the hardware approximation (-inf -> +0).
__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
                 "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
                   "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
                   "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
                   "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
                   "=r"(r[31])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 32; ++j)
        v[j] = __uint_as_float(r[j]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
                 "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
                 "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
                 "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                 "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
                 "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
                 "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
                 "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
                 "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
                 "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
                 "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
                 "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
                 "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
                 : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// One fp32 column of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st1(uint32_t taddr, float x)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr),
                 "r"(__float_as_uint(x))
                 : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ float tmem_ld1(uint32_t taddr)
{
    uint32_t r;
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    return __uint_as_float(r);
}

constexpr int TNT = 256;      // threads: two per query row, each with half the columns

template <int D, typename T>
__global__ void __launch_bounds__(TNT, 2) paged_prefill_tc_kernel(const PrefillParams p)
{
    using C = TcCfg<D>;
    constexpr uint32_t AB = MmaType<T>::bf16 ? 1u : 0u;
    constexpr int DCH = D / 8;                    // 16-byte chunks of a D-wide row
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sQ = smem_raw;
    unsigned char *sK = sQ + C::Q_BYTES;          // two buffers
    unsigned char *sV = sK + 2 * C::KV_BYTES;     // two buffers
    unsigned char *sP = sV + 2 * C::KV_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sP + C::P_BYTES);   // [0] S done, [2] O done
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 3);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    grid_dependency_wait();
    grid_dependents_launch();

    const int b = blockIdx.z;
    const int h = blockIdx.y;
    const int qt = gridDim.x - 1 - blockIdx.x;    // long (late) query tiles first
    const int q0 = __ldg(p.q_start + b);
    const int n = __ldg(p.q_start + b + 1) - q0;
    const int L = __ldg(p.seq_lens + b);
    if (qt * TBQ >= n)
        return;
    if (L < n || L > p.max_blocks_per_seq * p.block_size) {
        if (threadIdx.x == 0 && qt == 0 && h == 0)
            atomicOr(p.err, PKV_EBIT_SEQLEN);
        return;
    }
    const int G = p.num_q_heads / p.num_kv_heads;
    const int kvh = h / G;
    const int base = L - n;
    const int rows = min(TBQ, n - qt * TBQ);
    const int first_pos = base + qt * TBQ;        // position of this CTA's first query
    const int last_pos = first_pos + rows - 1;
    const int ntiles = last_pos / TBK + 1;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int quad = warp & 3;                     // TMEM lanes 32*quad .. 32*quad+31
    const int hf = warp >> 2;                      // which half of the columns
    const int32_t *table = p.block_tables + (int64_t)b * p.max_blocks_per_seq;
    const T *qg = static_cast<const T *>(p.q);
    const T *kg = static_cast<const T *>(p.k_cache);
    const T *vg = static_cast<const T *>(p.v_cache);

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        mbar_init(&bars[2], 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(tmem_slot)),
                     "n"(C::TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }

    // ---- async loads into the core-matrix layout
    for (int idx = tid; idx < TBQ * DCH; idx += TNT) {
        const int r = idx / DCH, c = idx % DCH;
        const bool ok = r < rows;
        const T *src = qg + ((int64_t)(q0 + qt * TBQ + (ok ? r : 0)) * p.num_q_heads + h) * D + c * 8;
        cp_async16(sQ + core_off(r, c, DCH), src, ok);
    }
    // K and V rows of key tile kt into buffer buf: thread t copies chunk
    // t % DCH of rows t / DCH, t / DCH + TNT / DCH, ... of both (block sizes
    // are powers of two: shifts, no divisions)
    auto load_kv = [&](int kt, int buf) {
        const int c = tid % DCH;
#pragma unroll 4
        for (int r = tid / DCH; r < TBK; r += TNT / DCH) {
            const int pos = kt * TBK + r;
            bool ok = pos <= last_pos;
            int64_t row = 0;
            if (ok) {
                const int32_t blk = __ldg(table + (pos >> p.bs_log2));
                if (blk < 0 || blk >= p.num_blocks) {
                    atomicOr(p.err, PKV_EBIT_BLOCK);
                    ok = false;
                } else {
                    row = (((int64_t)blk * p.num_kv_heads + kvh) << p.bs_log2) +
                          (pos & (p.block_size - 1));
                }
            }
            const uint32_t o = core_off(r, c, DCH);
            cp_async16(sK + buf * C::KV_BYTES + o, kg + row * D + c * 8, ok);
            cp_async16(sV + buf * C::KV_BYTES + o, vg + row * D + c * 8, ok);
        }
    };
    load_kv(0, 0);
    cp_async_commit();                            // group: Q, K0, V0
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tmem_s = tmem;                 // S: columns [0, 64)
    const uint32_t tmem_o = tmem + TBK;           // O: columns [64, 64 + D)
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const uint32_t tmem_x = tmem + TBK + D;       // exchange columns between the two halves
    const uint32_t idesc_s = umma_idesc(AB, 0u, TBK);
    const uint32_t idesc_o = umma_idesc(AB, 1u, D);
    const uint32_t sQa = smem_addr(sQ), sKa = smem_addr(sK), sVa = smem_addr(sV), sPa = smem_addr(sP);

    const int r = tid & (TBQ - 1);                 // this thread's query row
    const int qpos = first_pos + min(r, rows - 1);
    // The two threads of a row (warps quad and quad + 4) swap one value
    // through a spare TMEM column; a named barrier per warp pair orders it.
    auto swap_with_partner = [&](float mine, int slot) {
        tmem_st1(tmem_x + lane_base + 2 * slot + hf, mine);
        tc_fence_before();
        named_bar_sync(1 + quad, 64);
        tc_fence_after();
        return tmem_ld1(tmem_x + lane_base + 2 * slot + (hf ^ 1));
    };
    float m_run = -INFINITY, l_run = 0.0f;
    auto wait_bar = [&](uint64_t *bar, uint32_t parity) {
        if (!mbar_wait_bounded(bar, parity, abort_flag) && !*abort_flag) {
            *abort_flag = 1;
            atomicOr(p.err, PKV_EBIT_TIMEOUT);
        }
    };

    for (int kt = 0; kt < ntiles; ++kt) {
        const int buf = kt & 1;
        // K/V of the next tile go to the other buffer, which P.V(kt-1) (waited
        // below in the previous round) was the last to read
        if (kt + 1 < ntiles) {
            load_kv(kt + 1, buf ^ 1);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // S = Q K^T.  Q and K tiles are K-major with DCH chunks a row:
        // K-direction core stride 128 B, row-group stride DCH*128 B; a K = 16
        // step is two chunks.
        if (tid == 0 && !*abort_flag) {
            const uint32_t kb = sKa + buf * C::KV_BYTES;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                umma_f16(tmem_s, umma_desc(sQa + ks * 256, 128, DCH * 128),
                         umma_desc(kb + ks * 256, 128, DCH * 128), idesc_s, ks > 0 ? 1u : 0u);
            umma_commit(&bars[0]);
        }
        wait_bar(&bars[0], (uint32_t)(kt & 1));
        tc_fence_after();

        // ---- this row's scores in the log2 domain, masked where the tile
        // crosses the diagonal
        constexpr int HC = TBK / 2;                // score columns of this thread
        float v[HC];
        tmem_ld32(tmem_s + lane_base + hf * HC, v);
        const bool diag = kt * TBK + TBK - 1 > first_pos;
        if (diag) {
#pragma unroll
            for (int j = 0; j < HC; ++j)
                if (kt * TBK + hf * HC + j > qpos)
                    v[j] = -INFINITY;
        }
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < HC; ++j)
            mx = fmaxf(mx, v[j]);
        mx = fmaxf(mx, swap_with_partner(mx, kt & 1));   // the row's maximum
        mx *= p.scale_log2;                        // scale > 0: the maximum commutes
        // The running maximum moves only when a score exceeds it by more
        // than 2^8 (or on the first tile): below that the weights stay
        // <= 256, exact in fp32 and representable in fp16/bf16, and the
        // final division by the sum of the same weights is unchanged.
        const bool move = kt == 0 || mx > m_run + 8.0f;
        const float m_new = move ? fmaxf(m_run, mx) : m_run;
        const float corr = kt == 0 ? 1.0f : ex2_approx(m_run - m_new);
        m_run = m_new;
        float sum = 0.0f;
#pragma unroll
        for (int j = 0; j < HC; j += 8) {
            uint32_t w[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float p0 = ex2_approx(fmaf(v[j + 2 * u], p.scale_log2, -m_new));
                const float p1 = ex2_approx(fmaf(v[j + 2 * u + 1], p.scale_log2, -m_new));
                sum += p0 + p1;
                w[u] = pack2<T>(p0, p1);
            }
            *reinterpret_cast<uint4 *>(sP + core_off(r, (hf * HC + j) >> 3, TBK / 8)) =
                make_uint4(w[0], w[1], w[2], w[3]);
        }
        l_run = l_run * corr + sum;
        // rescale this warp's half of its O rows when some row maximum moved
        if (kt > 0 && __any_sync(FULL_MASK, move)) {
#pragma unroll
            for (int c0 = 0; c0 < D / 2; c0 += 32) {
                float o[32];
                tmem_ld32(tmem_o + lane_base + hf * (D / 2) + c0, o);
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    o[j] *= corr;
                tmem_st32(tmem_o + lane_base + hf * (D / 2) + c0, o);
            }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // O += P V.  P: K-major, TBK/8 chunks a row.  V is the MN-major B: K
        // (key) direction stride DCH*128 B per group of 8 keys, N (d)
        // direction stride 128 B; a step of 16 keys is two key groups.
        if (tid == 0 && !*abort_flag) {
            const uint32_t vb = sVa + buf * C::KV_BYTES;
#pragma unroll
            for (int ks = 0; ks < TBK / 16; ++ks)
                umma_f16(tmem_o, umma_desc(sPa + ks * 256, 128, (TBK / 8) * 128),
                         umma_desc(vb + ks * 2 * DCH * 128, DCH * 128, 128), idesc_o,
                         (kt > 0 || ks > 0) ? 1u : 0u);
            umma_commit(&bars[2]);
        }
        wait_bar(&bars[2], (uint32_t)(kt & 1));
        tc_fence_after();
    }


    // ---- O / l for this thread's half row (the TMEM loads are warp-wide
    // and run converged; padding rows load without storing)
    {
        const float inv = 1.0f / (l_run + swap_with_partner(l_run, 0));
        float *dst = p.out + ((int64_t)(q0 + qt * TBQ + min(r, rows - 1)) * p.num_q_heads + h) * D +
                     hf * (D / 2);
#pragma unroll
        for (int c0 = 0; c0 < D / 2; c0 += 32) {
            float o[32];
            tmem_ld32(tmem_o + lane_base + hf * (D / 2) + c0, o);
            if (r < rows) {
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    *reinterpret_cast<float4 *>(dst + c0 + j) =
                        make_float4(o[j] * inv, o[j + 1] * inv, o[j + 2] * inv, o[j + 3] * inv);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "n"(C::TMEM_COLS));
}

template <int D, typename T>
int launch_prefill_t(const pkv_pool *pool, const PrefillParams &prm, int max_q_len,
                     cudaStream_t s)
{
    (void)pool;
    using C = TcCfg<D>;
    static bool configured = false;
    if (!configured) {
        if (cudaFuncSetAttribute(paged_prefill_tc_kernel<D, T>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::SMEM_BYTES) != cudaSuccess)
            return PKV_ERR_CUDA;
        configured = true;
    }
    const dim3 grid((unsigned)((max_q_len + TBQ - 1) / TBQ), (unsigned)prm.num_q_heads,
                    (unsigned)prm.batch);
    if (launch_pdl(paged_prefill_tc_kernel<D, T>, grid, dim3(TNT), (size_t)C::SMEM_BYTES, s,
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
    prm.bs_log2 = 0;
    while ((1 << prm.bs_log2) < pool->block_size)
        ++prm.bs_log2;
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
