// paged_prefill_attention: causal attention of a batch of new tokens over the
// paged cache (the new tokens' K and V already appended).
//
// KV cache visualization page, "Prefill and decode feel different": the
// prompt's tokens are processed together in one pass, which makes the work
// limited by arithmetic rather than by memory traffic, so it runs on the
// fifth-generation tensor cores.  Token i of the n_b new
// tokens of sequence b sits at position p = seq_lens[b] - n_b + i and attends
// over positions 0..p ("KV cache: the engine behind fast LLM inference",
// "Concept"), in FlashAttention-style tiles that never hold the whole score
// matrix ("Flash attention: don't build the giant matrix" in the guide).

#include <algorithm>

#include <cuda.h>
#include <cudaTypedefs.h>
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

// A packed pair of the 16-bit type -> two floats (exact).
template <typename T>
__device__ __forceinline__ float2 unpack2(uint32_t w)
{
    if constexpr (MmaType<T>::bf16) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    } else {
        const __half2 h = *reinterpret_cast<const __half2 *>(&w);
        return __half22float2(h);
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
    // K and V caches as 3-D tensors {D, block_size, num_blocks * num_kv_heads}
    // for the tensor-memory-access unit: boxes of 64 x min(block_size, 128)
    // rows, 128-byte swizzle
    CUtensorMap tm_k, tm_v;
    const void *q;
    const void *k_cache;
    const void *v_cache;
    const int32_t *block_tables;
    const int32_t *q_start;
    const int32_t *seq_lens;
    float *out;
    unsigned int *err;
    int batch, num_q_heads, num_kv_heads, block_size, bs_log2, max_blocks_per_seq, num_blocks;
    int box_rows;       // min(block_size, 128)
    int nqt;            // query tiles of 256 per sequence: ceil(max_q_len / 256)
    int nitems;         // work items (see make_item / make_prefix_item)
    float scale_log2;
    // Shared-prefix pass (cascade): instead of a prompt's causal queries, the
    // rows of an item are the q heads of the sequences of one group that
    // share a prefix (member-major: row m G + g is member m's head kvh G + g),
    // over one chunk of the prefix's keys, with no causal mask; the result is
    // a partial (unnormalised O, running maximum, sum) per row.
    int cascade;
    const int32_t *grp_start;   // [ngroups + 1]: the group's members in grp_seqs
    const int32_t *grp_seqs;    // member sequences; the first one's table is read
    const int32_t *grp_len;     // [ngroups]: tokens of the shared prefix
    int ngroups, group_q;       // groups; query heads per KV head
    int kc_tiles, nkc;          // key tiles (of 128) per chunk; chunks per group at most
    float *part;                // [nkc][batch][num_q_heads][D + 4]
};

// ---- tcgen05: 2 x 128 queries x 128 keys per step, warp-specialised,
// persistent
//
// One CTA per SM walks work items: 256 queries of one (sequence, query head)
// as two 128-row halves A and B that share every K/V tile.  Items are
// numbered longest first and dealt to the CTAs in an order that alternates
// direction each round.  Three roles:
//  * four producer warps copy a quarter of each item's Q with 16-byte
//    cp.async copies into the tensor cores' core-matrix layout (8 rows x 16
//    bytes per 128-byte core matrix, no swizzle); then warps 0, 1 bring K
//    tiles and warps 2, 3 V tiles into two-slot rings, 128-byte swizzled
//    (row r of a 64-column panel at 128 r, its 16-byte chunks permuted by
//    r mod 8): one tensor-memory-access copy per cache block and panel (lane
//    j takes the j-th block of the tile), 16-byte cp.async copies for blocks
//    of 4 rows and for the block where the sequence ends;
//  * one thread issues the tcgen05.mma: S = Q K^T (M 128, N 128, K = D, both
//    operands in shared memory) and O += P V (M 128, N = D, K 128, P read
//    from tensor memory, as a high and a low part: two MMAs per K step)
//    per half, fp32 accumulators in tensor memory (half h: S in columns
//    [256 h, 256 h + 128), O in the next D);
//  * one warpgroup per half, one thread per query row, reads its S row with
//    tcgen05.ld, does the online softmax, writes P as high and low
//    fp16/bf16 parts (p = hi + lo to ~2^-16) over the S columns it has
//    read, rescales its O row in tensor memory when the
//    row maximum moved by more than 2^8, and at the end of an item writes
//    O / l out through shared-memory staging.
// The issue order PV_A(j), S_A(j+1), PV_B(j), S_B(j+1) lets one half's
// softmax run while the tensor cores work on the other half; tcgen05.mma
// runs in issue order, so S_h(j+1) overwrites P_h(j) only after P_h(j) V
// has read it.  mbarriers hand the work over: k_full / k_empty and v_full /
// v_empty per slot (tiles counted across items), s_full (tcgen05.commit
// after S_h, which also covers the P V issued before it, so O_h is idle),
// p_full (the half's 128 softmax threads), o_done (after an item's last
// P V), o_free (the softmax threads have read O out: the next item's first
// P V may overwrite it) and q_full / q_empty (the next item's Q loads once
// the current item's last S has read Q).

constexpr int TBQ = 128, TBK = 128, NQH = 2, NSLOT = 2;
constexpr int SOFT_WARPS = 4 * NQH, PROD_WARPS = 2 * NSLOT;   // K slots, then V slots
constexpr int MMA_WARP = SOFT_WARPS + PROD_WARPS;
constexpr int TNT = (MMA_WARP + 1) * 32;

template <int D>
struct TcCfg {
    static constexpr int Q_BYTES = TBQ * D * 2;          // one half
    static constexpr int KV_BYTES = TBK * D * 2;          // one K or V tile
    // output staging: 32 rows x 32 fp32 per softmax warp
    static constexpr int STG_OFF = NQH * Q_BYTES + 2 * NSLOT * KV_BYTES;
    static constexpr int BAR_OFF = STG_OFF + SOFT_WARPS * 32 * 32 * 4;
    static constexpr int NBARS = 4 * NSLOT + 4 * NQH + 3;
    static constexpr int SMEM_BYTES = BAR_OFF + NBARS * 8 + 16;
    static constexpr int TMEM_COLS = 512;
    static constexpr int HALF_COLS = 256;                 // >= TBK + D
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

// The same for a 128-byte swizzled operand (layout type 2 in bits 61-63).
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    return umma_desc(saddr, lbo, sbo) | ((uint64_t)2 << 61);
}

// One box of a 3-D tensor map into shared memory, completion counted in bytes
// on an mbarrier.  Coordinates past the tensor's end read zeros.
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int x, int y, int z,
                                            uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
        : "memory");
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

// The same with A (M rows in TMEM lanes, K as 16-bit pairs along columns) read
// from tensor memory.
__device__ __forceinline__ void umma_f16_ta(uint32_t tmem_d, uint32_t tmem_a, uint64_t db,
                                            uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
                 "r"(tmem_a), "l"(db), "r"(idesc), "r"(accumulate)
                 : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(bar))
                 : "memory");
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float max3f(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// (a0, a1) = (a0, a1) * s + c as one packed fp32x2 FMA.
__device__ __forceinline__ void fma2_bc(float &a0, float &a1, float s, float c)
{
    asm("{\n\t.reg .b64 x, y, z;\n\tmov.b64 x, {%0, %1};\n\tmov.b64 y, {%2, %2};\n\t"
        "mov.b64 z, {%3, %3};\n\tfma.rn.f32x2 x, x, y, z;\n\tmov.b64 {%0, %1}, x;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(s), "f"(c));
}

// (a0, a1) += (b0, b1) as one packed fp32x2 add.
__device__ __forceinline__ void add2(float &a0, float &a1, float b0, float b1)
{
    asm("{\n\t.reg .b64 x, y;\n\tmov.b64 x, {%0, %1};\n\tmov.b64 y, {%2, %3};\n\t"
        "add.rn.f32x2 x, x, y;\n\tmov.b64 {%0, %1}, x;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(b0), "f"(b1));
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

// 16 consecutive 32-bit columns of this thread's TMEM lane (no wait).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&w)[16])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,"
                 "%12,%13,%14,%15,%16};" ::"r"(taddr),
                 "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]),
                 "r"(w[7]), "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]),
                 "r"(w[14]), "r"(w[15])
                 : "memory");
}

// One unit of work: 256 queries (two halves of 128) of sequence b, query
// head h, query tile qt.  Items are numbered longest (latest) tiles first;
// every role of a CTA derives the same items in the same order.
struct Item {
    int b, h, qt, q0, kvh, rows_all, first_pos, last_pos, ntiles;
    int rows_h[NQH], tiles_h[NQH];
    int kt0;         // first key tile (a prefix chunk's offset; 0 for prefill)
    int g, c;        // prefix pass: group and key chunk
    bool live;       // has rows and valid lengths
    bool bad_len;    // has rows but its length fields are inconsistent
};

// Prefix-pass item i: (row tile qt, group g, KV head kvh, key chunk c).  The
// rows are the group's members' q heads of kvh; the keys, tiles [kt0, kt0 +
// ntiles) of the prefix (every row sees every prefix key: first_pos =
// last_pos = prefix length - 1).
__device__ __forceinline__ Item make_prefix_item(const PrefillParams &p, int i)
{
    constexpr int QT = NQH * TBQ;
    Item it;
    const int per = p.ngroups * p.num_kv_heads * p.nkc;
    it.qt = i / per;
    int rem = i - it.qt * per;
    it.g = rem / (p.num_kv_heads * p.nkc);
    rem -= it.g * (p.num_kv_heads * p.nkc);
    it.kvh = rem / p.nkc;
    it.c = rem - it.kvh * p.nkc;
    it.h = it.kvh * p.group_q;
    it.q0 = __ldg(p.grp_start + it.g);
    const int members = __ldg(p.grp_start + it.g + 1) - it.q0;
    const int P = __ldg(p.grp_len + it.g);
    it.b = members > 0 ? __ldg(p.grp_seqs + it.q0) : 0;
    const int L = members > 0 ? __ldg(p.seq_lens + it.b) : 0;
    it.kt0 = it.c * p.kc_tiles;
    const int rows_total = members * p.group_q;
    const bool rows = it.qt * QT < rows_total && P > 0 && it.kt0 * TBK < P;
    it.bad_len = rows && (P > L || L > p.max_blocks_per_seq * p.block_size);
    it.live = rows && !it.bad_len;
    it.rows_all = it.live ? min(QT, rows_total - it.qt * QT) : 0;
    it.first_pos = P - 1;
    it.last_pos = P - 1;
    it.ntiles = it.live ? min(p.kc_tiles, (P + TBK - 1) / TBK - it.kt0) : 0;
    it.rows_h[0] = min(TBQ, it.rows_all);
    it.rows_h[1] = max(0, it.rows_all - TBQ);
    it.tiles_h[0] = it.rows_h[0] > 0 ? it.ntiles : 0;
    it.tiles_h[1] = it.rows_h[1] > 0 ? it.ntiles : 0;
    return it;
}

__device__ __forceinline__ Item make_item(const PrefillParams &p, int i)
{
    constexpr int QT = NQH * TBQ;
    if (p.cascade)
        return make_prefix_item(p, i);
    Item it;
    it.kt0 = 0;
    it.g = it.c = 0;
    const int per = p.num_q_heads * p.batch;
    const int qt_rev = i / per, rem = i - qt_rev * per;
    it.qt = p.nqt - 1 - qt_rev;
    it.b = rem % p.batch;
    it.h = rem / p.batch;
    it.q0 = __ldg(p.q_start + it.b);
    const int n = __ldg(p.q_start + it.b + 1) - it.q0;
    const int L = __ldg(p.seq_lens + it.b);
    const bool rows = it.qt * QT < n;
    it.bad_len = rows && (L < n || L > p.max_blocks_per_seq * p.block_size);
    it.live = rows && !it.bad_len;
    it.kvh = it.h / (p.num_q_heads / p.num_kv_heads);
    it.rows_all = it.live ? min(QT, n - it.qt * QT) : 0;
    it.first_pos = L - n + it.qt * QT;              // position of the item's first query
    it.last_pos = it.first_pos + it.rows_all - 1;
    it.ntiles = it.live ? it.last_pos / TBK + 1 : 0;
    it.rows_h[0] = min(TBQ, it.rows_all);
    it.rows_h[1] = max(0, it.rows_all - TBQ);
    it.tiles_h[0] = it.live ? (it.first_pos + it.rows_h[0] - 1) / TBK + 1 : 0;
    it.tiles_h[1] = it.rows_h[1] > 0 ? it.ntiles : 0;
    return it;
}

// This CTA's item in round rnd (-1: none): items are numbered longest
// first, and the rounds alternate direction over the CTAs so that every CTA
// gets a mix of long and short items.
__device__ __forceinline__ int item_of(int rnd, int nitems)
{
    const int c = (rnd & 1) ? (int)(gridDim.x - 1 - blockIdx.x) : (int)blockIdx.x;
    const int i = rnd * (int)gridDim.x + c;
    return i < nitems ? i : -1;
}

template <int D, typename T>
__global__ void __launch_bounds__(TNT, 1) paged_prefill_tc_kernel(const __grid_constant__ PrefillParams p)
{
    using C = TcCfg<D>;
    constexpr uint32_t AB = MmaType<T>::bf16 ? 1u : 0u;
    constexpr int DCH = D / 8;                    // 16-byte chunks of a D-wide row
    constexpr int QT = NQH * TBQ;                 // queries of an item
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sQ = smem_raw;                              // NQH halves
    unsigned char *sK = sQ + NQH * C::Q_BYTES;                 // NSLOT K tiles
    unsigned char *sV = sK + NSLOT * C::KV_BYTES;              // NSLOT V tiles
    float4 *stg_all = reinterpret_cast<float4 *>(smem_raw + C::STG_OFF);
    uint64_t *k_full = reinterpret_cast<uint64_t *>(smem_raw + C::BAR_OFF);
    uint64_t *k_empty = k_full + NSLOT;
    uint64_t *v_full = k_empty + NSLOT;
    uint64_t *v_empty = v_full + NSLOT;
    uint64_t *s_full = v_empty + NSLOT;
    uint64_t *p_full = s_full + NQH;
    uint64_t *o_done = p_full + NQH;
    uint64_t *o_free = o_done + NQH;
    uint64_t *q_full = o_free + NQH;
    uint64_t *q_empty = q_full + 1;
    uint64_t *drain = q_empty + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    grid_dependency_wait();
    grid_dependents_launch();

    const int nitems = p.nitems;
    const int tid = threadIdx.x, warp = tid >> 5;

    if (tid == 0) {
        for (int i = 0; i < NSLOT; ++i) {
            mbar_init(&k_full[i], 2);              // tensor-copy bytes + the 16-byte copies
            mbar_init(&k_empty[i], 1);
            mbar_init(&v_full[i], 2);
            mbar_init(&v_empty[i], 1);
        }
        for (int i = 0; i < NQH; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], TBQ);
            mbar_init(&o_done[i], 1);
            mbar_init(&o_free[i], TBQ);
        }
        mbar_init(q_full, PROD_WARPS * 32);
        mbar_init(q_empty, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == MMA_WARP) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(tmem_slot)),
                     "n"(C::TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // A timed-out wait raises the error bit once and makes every role stop.
    auto wait = [&](uint64_t *bar, uint32_t parity) -> bool {
        if (mbar_wait_bounded(bar, parity, abort_flag))
            return true;
        if (!*abort_flag) {
            *abort_flag = 1;
            atomicOr(p.err, PKV_EBIT_TIMEOUT);
        }
        return false;
    };

    if (warp < SOFT_WARPS) {
        // ================= softmax: one thread per query row of half hh
        const int hh = warp >> 2, quad = warp & 3;
        const int r = quad * 32 + (tid & 31);
        const uint32_t t_s = tmem + hh * C::HALF_COLS + ((uint32_t)(quad * 32) << 16);
        const uint32_t t_o = t_s + TBK;
        uint32_t sc = 0, od = 0;                   // phases used of s_full[hh], o_done[hh]
        for (int rnd = 0; rnd * (int)gridDim.x < nitems; ++rnd) {
            const int i = item_of(rnd, nitems);
            if (i < 0)
                continue;
            const Item it = make_item(p, i);
            const int rows = it.rows_h[hh], my_tiles = it.tiles_h[hh];
            if (my_tiles == 0)
                continue;
            // the row's position: causal rows step along the prompt; prefix
            // rows all stand after the whole prefix
            const int qpos = p.cascade ? it.first_pos
                                       : it.first_pos + hh * TBQ + min(r, max(rows, 1) - 1);
            float m_run = -INFINITY, l_run = 0.0f;
            for (int kt = 0; kt < my_tiles; ++kt) {
                if (!__all_sync(FULL_MASK, wait(&s_full[hh], sc & 1)))
                    goto softmax_done;
                ++sc;
                tc_fence_after();
                // keys past this row's position (the tile crosses the
                // diagonal) drop out
                const int kpos = (it.kt0 + kt) * TBK;     // the tile's first key
                const bool diag = kpos + TBK - 1 > (p.cascade ? it.first_pos
                                                              : it.first_pos + hh * TBQ);
                const int lim = qpos - kpos;       // last unmasked column
                // pass 1: the row maximum, 32 columns at a time (chunk loops
                // stay rolled: the three roles share the instruction cache)
                float mx = -INFINITY;
#pragma unroll 1
                for (int c0 = 0; c0 < TBK; c0 += 32) {
                    float v[32];
                    tmem_ld32(t_s + c0, v);
                    if (diag) {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (c0 + j > lim)
                                v[j] = -INFINITY;
                    }
                    // three-input maxima: 32 -> 11 -> 4 -> 1
                    float t[11];
#pragma unroll
                    for (int j = 0; j < 10; ++j)
                        t[j] = max3f(v[3 * j], v[3 * j + 1], v[3 * j + 2]);
                    t[10] = fmaxf(v[30], v[31]);
                    mx = max3f(mx, max3f(t[0], t[1], t[2]), max3f(t[3], t[4], t[5]));
                    mx = max3f(mx, max3f(t[6], t[7], t[8]), fmaxf(t[9], t[10]));
                }
                mx *= p.scale_log2;                // scale > 0: the maximum commutes
                // The running maximum moves only when a score exceeds it by
                // more than 2^8 (or on the first tile): below that the weights
                // stay <= 256, exact in fp32 and representable in fp16/bf16,
                // and the final division by the sum of the same weights is
                // unchanged.
                const bool move = kt == 0 || mx > m_run + 8.0f;
                const float m_new = move ? fmaxf(m_run, mx) : m_run;
                const float corr = kt == 0 ? 1.0f : ex2_approx(m_run - m_new);
                m_run = m_new;
                // O_h is idle here: the P V of the previous tile finished
                // before S_h(kt) did, the next one waits for p_full
                if (kt > 0 && __any_sync(FULL_MASK, move)) {
#pragma unroll 1
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        float o[32];
                        tmem_ld32(t_o + c0, o);
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            o[j] *= corr;
                        tmem_st32(t_o + c0, o);
                    }
                }
                // pass 2: weights, their sum, and P (keys 32c..32c+31 as
                // 16-bit pairs, high parts in columns 32c..32c+15, low parts
                // in 32c+16..32c+31: the S columns of this chunk, already
                // read)
                float sum = 0.0f;
#pragma unroll 1
                for (int c0 = 0; c0 < TBK; c0 += 32) {
                    float v[32];
                    tmem_ld32(t_s + c0, v);
                    if (diag) {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (c0 + j > lim)
                                v[j] = -INFINITY;
                    }
#pragma unroll
                    for (int j = 0; j < 32; j += 2)        // the exponent, two a step
                        fma2_bc(v[j], v[j + 1], p.scale_log2, -m_new);
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        v[j] = ex2_approx(v[j]);
                    // P in two parts of the 16-bit type, hi + lo = p to
                    // ~2^-16 relative (rounded once, p alone would carry up
                    // to 2^-9 (bf16) or 2^-12 (fp16) of error into P.V)
                    uint32_t w[16], wl[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        w[j] = pack2<T>(v[2 * j], v[2 * j + 1]);
                        const float2 h = unpack2<T>(w[j]);
                        float r0 = v[2 * j], r1 = v[2 * j + 1];
                        add2(r0, r1, -h.x, -h.y);
                        wl[j] = pack2<T>(r0, r1);
                    }
                    tmem_st16(t_s + c0, w);
                    tmem_st16(t_s + c0 + 16, wl);
#pragma unroll
                    for (int k = 16; k > 1; k >>= 1)       // tree sum over pairs
#pragma unroll
                        for (int j = 0; j < k; j += 2)
                            add2(v[j], v[j + 1], v[j + k], v[j + k + 1]);
                    sum += v[0] + v[1];
                }
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                l_run = l_run * corr + sum;
                tc_fence_before();
                mbar_arrive(&p_full[hh]);
            }
            // ---- O / l (warp-uniform: the TMEM loads run converged; padding
            // rows load without storing), then O_h is free for the next item
            if (!__all_sync(FULL_MASK, wait(&o_done[hh], od & 1)))
                goto softmax_done;
            ++od;
            tc_fence_after();
            {
                // 32 columns at a time through the warp's staging rows (16-byte
                // slot j of row x at j xor (x mod 8): conflict-free both
                // ways), then out as 128-byte row segments, four rows a store
                // (prefix pass: O unnormalised, with the row's running
                // maximum and sum beside it)
                const float inv = p.cascade ? 1.0f : 1.0f / l_run;
                const int lane = tid & 31;
                float4 *stg = stg_all + warp * 32 * 8;
                const int xr = lane >> 3, xj = lane & 7;   // store: rows xr, xr + 4, ...
                const int64_t row0 = (int64_t)it.q0 + it.qt * QT + hh * TBQ + quad * 32;
                // output row of the item's row x of this warp's 32
                auto out_row = [&](int x) -> float * {
                    if (!p.cascade)
                        return p.out + ((row0 + x) * p.num_q_heads + it.h) * D;
                    const int mr = it.qt * QT + hh * TBQ + quad * 32 + x;   // member row
                    const int mem = mr / p.group_q;
                    const int seq = __ldg(p.grp_seqs + it.q0 + mem);
                    return p.part + (((int64_t)it.c * p.batch + seq) * p.num_q_heads +
                                     it.kvh * p.group_q + (mr - mem * p.group_q)) * (D + 4);
                };
                // each lane finds its own row once; a store of row x takes
                // lane x's pointer
                float *const my_row = r < rows ? out_row(lane) : nullptr;
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    float o[32];
                    tmem_ld32(t_o + c0, o);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        stg[lane * 8 + (j ^ (lane & 7))] = make_float4(
                            o[4 * j] * inv, o[4 * j + 1] * inv, o[4 * j + 2] * inv, o[4 * j + 3] * inv);
                    __syncwarp();
#pragma unroll
                    for (int x = xr; x < 32; x += 4) {
                        const float4 v = stg[x * 8 + (xj ^ (x & 7))];
                        float *const rp = reinterpret_cast<float *>(__shfl_sync(
                            0xffffffffu, reinterpret_cast<unsigned long long>(my_row), x));
                        if (quad * 32 + x < rows)
                            *reinterpret_cast<float4 *>(rp + c0 + 4 * xj) = v;
                    }
                    __syncwarp();
                }
                if (p.cascade && r < rows) {
                    my_row[D] = m_run;
                    my_row[D + 1] = l_run;
                }
            }
            tc_fence_before();
            mbar_arrive(&o_free[hh]);
        }
    softmax_done:;
    } else if (warp < MMA_WARP) {
        // ================= producer warp pw: per item, rows pw*64 .. pw*64+63
        // of Q (once the previous item's last S has read Q), then K (pw <
        // NSLOT) or V tiles into slot pw % NSLOT: the CTA's tiles are counted
        // across items, tile g in slot g % NSLOT.  Q: eight consecutive lanes
        // fill one core matrix (8 rows x 16 B, a conflict-free 128-byte
        // shared-memory write); a warp reads 64 contiguous bytes of 8 rows.
        const int pw = warp - SOFT_WARPS;
        const int slot = pw % NSLOT;
        const bool is_k = pw < NSLOT;
        const int rr = tid & 7, cq = (tid >> 3) & 3;
        const int lane = tid & 31;
        const T *qg = static_cast<const T *>(p.q);
        unsigned char *ring = (is_k ? sK : sV) + slot * C::KV_BYTES;
        uint64_t *full = is_k ? &k_full[slot] : &v_full[slot];
        uint64_t *empty = is_k ? &k_empty[slot] : &v_empty[slot];
        const CUtensorMap *tm = is_k ? &p.tm_k : &p.tm_v;
        const T *cache = static_cast<const T *>(is_k ? p.k_cache : p.v_cache);
        const int R = p.box_rows;                  // rows of one box: min(block size, 128)
        const int nbox = TBK / R;                  // boxes a tile: at most 32 (blocks >= 4 rows)
        const int oob = p.num_blocks * p.num_kv_heads;   // a block index past the end: zero fill
        int gt = 0;                                // the CTA's tiles so far
        uint32_t qc = 0;                           // items so far
        for (int rnd = 0; rnd * (int)gridDim.x < nitems; ++rnd) {
            const int i = item_of(rnd, nitems);
            if (i < 0)
                continue;
            const Item it = make_item(p, i);
            if (!it.live)
                continue;
            const int32_t *table = p.block_tables + (int64_t)it.b * p.max_blocks_per_seq;
            if (qc > 0 && !wait(q_empty, (qc - 1) & 1))
                goto producer_done;
#pragma unroll 1
            for (int g = 0; g < QT / PROD_WARPS / 8; ++g) {
                const int r = pw * (QT / PROD_WARPS) + g * 8 + rr;   // query of the item
                const bool ok = r < it.rows_all;
                const T *src;
                if (p.cascade) {
                    // member row: member mr / G's q head kvh G + mr % G
                    const int mr = it.qt * QT + (ok ? r : 0);
                    const int mem = mr / p.group_q;
                    const int seq = __ldg(p.grp_seqs + it.q0 + mem);
                    src = qg + ((int64_t)seq * p.num_q_heads + it.h + (mr - mem * p.group_q)) * D;
                } else {
                    src = qg + ((int64_t)(it.q0 + it.qt * QT + (ok ? r : 0)) * p.num_q_heads +
                                it.h) * D;
                }
#pragma unroll
                for (int c = cq; c < DCH; c += 4)
                    cp_async16(sQ + (r >> 7) * C::Q_BYTES + core_off(r & (TBQ - 1), c, DCH),
                               src + c * 8, ok);
            }
            cp_async_commit();
            bool q_sent = false;
            for (int kt = 0; kt < it.ntiles; ++kt) {
                const int g = gt + kt;
                if (g % NSLOT != slot)
                    continue;
                // lane j: rows [j R, j R + R) of the tile, one cache block
                // (block sizes are powers of two: shifts, no divisions); the
                // block-id load overlaps the wait for the slot
                const int pos0 = (it.kt0 + kt) * TBK + lane * R;
                const bool inbox = lane < nbox;
                const bool live = inbox && pos0 <= it.last_pos;
                const int32_t blk = live ? __ldg(table + (pos0 >> p.bs_log2)) : 0;
                if (g >= NSLOT && !wait(empty, (uint32_t)(((g / NSLOT) & 1) ^ 1)))
                    goto producer_done;
                int z = oob;
                if (live) {
                    if (blk < 0 || blk >= p.num_blocks)
                        atomicOr(p.err, PKV_EBIT_BLOCK);
                    else
                        z = blk * p.num_kv_heads + it.kvh;
                }
                const int y = pos0 & (p.block_size - 1);
                // A box goes by one tensor copy per 64-column panel when it
                // starts on a 1024-byte boundary (boxes of >= 8 rows) and
                // holds no row past the sequence end (those must be zeros: P
                // is 0 there, but 0 times a stale NaN is not); the other
                // boxes go by 16-byte copies.
                const bool by_tma = inbox && R >= 8 && (z == oob || pos0 + R - 1 <= it.last_pos);
                const unsigned tma_boxes = __popc(__ballot_sync(FULL_MASK, by_tma));
                const unsigned cp_boxes = __ballot_sync(FULL_MASK, inbox && !by_tma);
                if (lane == 0)
                    mbar_arrive_expect_tx(full, tma_boxes * (uint32_t)R * 2u * D);
                __syncwarp();
                if (by_tma) {
#pragma unroll
                    for (int pn = 0; pn < D / 64; ++pn)
                        tma_load_3d(ring + pn * (TBK * 128) + lane * R * 128, tm, pn * 64, y, z,
                                    full);
                }
                if (cp_boxes) {
                    // chunk c of tile row r lands at 128 r + 16 (c mod 8 xor
                    // r mod 8) in panel c / 8 (the 128-byte swizzle pattern)
                    for (unsigned m = cp_boxes; m; m &= m - 1) {
                        const int bx = __ffs(m) - 1;
                        const int zb = __shfl_sync(FULL_MASK, z, bx);
                        const int yb = __shfl_sync(FULL_MASK, y, bx);
                        for (int idx = lane; idx < R * DCH; idx += 32) {
                            const int r = bx * R + idx / DCH, c = idx % DCH;
                            const bool valid =
                                zb != oob && (it.kt0 + kt) * TBK + r <= it.last_pos;
                            const int64_t row =
                                valid ? (int64_t)zb * p.block_size + yb + idx / DCH : 0;
                            cp_async16(ring + (c >> 3) * (TBK * 128) + r * 128 +
                                           (((c & 7) ^ (r & 7)) << 4),
                                       cache + row * D + c * 8, valid);
                        }
                    }
                    cp_async_commit();
                    cp_async_wait<0>();
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                }
                __syncwarp();
                if (lane == 0)                     // the 16-byte copies (if any) have landed
                    mbar_arrive(full);
                if (!q_sent) {                     // Q (this thread's cp.async group) has landed
                    cp_async_wait<0>();
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    mbar_arrive(q_full);
                    q_sent = true;
                }
            }
            if (!q_sent) {
                cp_async_wait<0>();
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                mbar_arrive(q_full);
            }
            gt += it.ntiles;
            ++qc;
        }
    producer_done:
        cp_async_wait<0>();
    } else if ((tid & 31) == 0) {
        // ================= MMA issue (one thread)
        const uint32_t idesc_s = umma_idesc(AB, 0u, TBK);
        const uint32_t idesc_o = umma_idesc(AB, 1u, D);
        const uint32_t sQa = smem_addr(sQ), sKa = smem_addr(sK), sVa = smem_addr(sV);
        int gt = 0;                                // the CTA's tiles so far
        uint32_t qc = 0, pc[NQH] = {0, 0}, ofc[NQH] = {0, 0};
        bool o_used[NQH] = {false, false};         // O_h holds an earlier item's result
        bool ok = true;
        for (int rnd = 0; rnd * (int)gridDim.x < nitems && ok; ++rnd) {
            const int i = item_of(rnd, nitems);
            if (i < 0)
                continue;
            const Item it = make_item(p, i);
            if (it.bad_len)
                atomicOr(p.err, PKV_EBIT_SEQLEN);
            if (!it.live)
                continue;
            const int last_half = it.tiles_h[1] > 0 ? 1 : 0;   // the last reader of each tile
            int s_left = it.tiles_h[0] + it.tiles_h[1];         // S issues until Q is free
            // S_hh = Q_hh K^T, both K-major.  Q: core-matrix layout with DCH
            // chunks a row (K-direction core stride 128 B, row-group stride
            // DCH*128 B; a K = 16 step is two chunks).  K: 128-byte swizzled
            // panels of 64 d (8-row groups 1024 B apart); a K = 16 step is
            // 32 B into the panel's rows.
            auto issue_s = [&](int hh, int g) {
                const uint32_t kb = sKa + (g % NSLOT) * C::KV_BYTES, qb = sQa + hh * C::Q_BYTES;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    umma_f16(tmem + hh * C::HALF_COLS, umma_desc(qb + ks * 256, 128, DCH * 128),
                             umma_desc_sw128(kb + (ks / 4) * (TBK * 128) + (ks % 4) * 32, 16, 1024),
                             idesc_s, ks > 0 ? 1u : 0u);
                if (hh == last_half)
                    umma_commit(&k_empty[g % NSLOT]);
                umma_commit(&s_full[hh]);
                if (--s_left == 0)
                    umma_commit(q_empty);
            };
            // O_hh += P_hh V.  P: in tensor memory over the S columns, keys
            // 32c..32c+31 as 16-bit pairs: the high parts in columns 32c..
            // 32c+15, the low parts in the next 16; a K step (16 keys) reads
            // 8 columns of each, both MMAs accumulating into O_hh.  V is the
            // MN-major B in 128-byte
            // swizzled panels: a key row of 64 d every 128 B, 8-key groups
            // 1024 B apart, the next 64 d a panel (TBK*128 B) on; a step of
            // 16 keys is 2048 B.
            auto issue_pv = [&](int hh, int g, int kt) {
                const uint32_t vb = sVa + (g % NSLOT) * C::KV_BYTES;
#pragma unroll
                for (int ks = 0; ks < TBK / 16; ++ks) {
                    const uint32_t pa = tmem + hh * C::HALF_COLS + 32 * (ks >> 1) + 8 * (ks & 1);
                    const uint64_t vd = umma_desc_sw128(vb + ks * 2048, TBK * 128, 1024);
                    umma_f16_ta(tmem + hh * C::HALF_COLS + TBK, pa, vd, idesc_o,
                                (kt > 0 || ks > 0) ? 1u : 0u);
                    umma_f16_ta(tmem + hh * C::HALF_COLS + TBK, pa + 16, vd, idesc_o, 1u);
                }
                if (hh == last_half)
                    umma_commit(&v_empty[g % NSLOT]);
            };
            if (!(ok = wait(q_full, qc & 1) &&
                       wait(&k_full[gt % NSLOT], (uint32_t)((gt / NSLOT) & 1))))
                break;
            ++qc;
            tc_fence_after();
            for (int hh = 0; hh < NQH; ++hh)
                if (it.tiles_h[hh] > 0)
                    issue_s(hh, gt);
            for (int kt = 0; kt < it.ntiles && ok; ++kt) {
                const int g = gt + kt;
                for (int hh = 0; hh < NQH; ++hh) {
                    if (kt >= it.tiles_h[hh])
                        continue;
                    if (!(ok = wait(&p_full[hh], pc[hh] & 1) &&
                               wait(&v_full[g % NSLOT], (uint32_t)((g / NSLOT) & 1))))
                        break;
                    ++pc[hh];
                    if (kt == 0 && o_used[hh]) {   // the softmax warps have read O_h out
                        if (!(ok = wait(&o_free[hh], ofc[hh] & 1)))
                            break;
                        ++ofc[hh];
                    }
                    tc_fence_after();
                    issue_pv(hh, g, kt);
                    if (kt + 1 < it.tiles_h[hh]) {
                        if (!(ok = wait(&k_full[(g + 1) % NSLOT], (uint32_t)(((g + 1) / NSLOT) & 1))))
                            break;
                        tc_fence_after();
                        issue_s(hh, g + 1);
                    } else {
                        umma_commit(&o_done[hh]);
                        o_used[hh] = true;
                    }
                }
            }
            gt += it.ntiles;
        }
        // every issued MMA has finished before tensor memory is released
        umma_commit(drain);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(drain, 0u) && globaltimer_ns() - t0 < WAIT_LIMIT_NS) {
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "n"(C::TMEM_COLS));
    }
}

template <int D, typename T>
int launch_prefill_t(const pkv_pool *pool, const PrefillParams &prm, int max_q_len,
                     cudaStream_t s)
{
    using C = TcCfg<D>;
    // Set per call (for the current device, from any host thread): a few
    // microseconds against a kernel of hundreds.
    if (cudaFuncSetAttribute(paged_prefill_tc_kernel<D, T>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM_BYTES) != cudaSuccess)
        return PKV_ERR_CUDA;
    // one CTA per SM (of the pool's device), each walking the items c,
    // c + grid, ...
    const int sms = pool->num_sms;
    if (sms < 1)
        return PKV_ERR_CUDA;
    (void)max_q_len;
    const int nitems = prm.nitems;
    if (nitems < 1)
        return PKV_OK;
    const dim3 grid((unsigned)(nitems < sms ? nitems : sms));
    if (launch_pdl(paged_prefill_tc_kernel<D, T>, grid, dim3(TNT), (size_t)C::SMEM_BYTES, s,
                   prm) != cudaSuccess)
        return PKV_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

// A cache [num_blocks][num_kv_heads][block_size][D] of 16-bit elements as the
// 3-D tensor {D, block_size, num_blocks * num_kv_heads}, boxes of 64 x rows x 1.
bool encode_cache_map(CUtensorMap *m, const pkv_pool *pool, const void *base, int rows)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc)
        return false;
    const int D = pool->head_dim, bs = pool->block_size;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)bs,
                                (cuuint64_t)pool->num_blocks * (cuuint64_t)pool->num_kv_heads};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)bs * D * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType dt = pool->kv_dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                              : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    return enc(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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
    prm.box_rows = pool->block_size < TBK ? pool->block_size : TBK;
    constexpr int QT = NQH * TBQ;
    prm.nqt = (max_q_len + QT - 1) / QT;
    if ((int64_t)prm.nqt * num_q_heads * batch >= ((int64_t)1 << 31))
        return PKV_ERR_UNSUPPORTED;
    prm.nitems = prm.nqt * num_q_heads * batch;
    if (!encode_cache_map(&prm.tm_k, pool, k_cache, prm.box_rows) ||
        !encode_cache_map(&prm.tm_v, pool, v_cache, prm.box_rows))
        return PKV_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool bf = pool->kv_dtype == PKV_BF16;
    if (pool->head_dim == 64)
        return bf ? launch_prefill_t<64, __nv_bfloat16>(pool, prm, max_q_len, s)
                  : launch_prefill_t<64, __half>(pool, prm, max_q_len, s);
    return bf ? launch_prefill_t<128, __nv_bfloat16>(pool, prm, max_q_len, s)
              : launch_prefill_t<128, __half>(pool, prm, max_q_len, s);
}

namespace {

// Merge each prefix row's chunk partials (left by the prefix pass) into chunk
// 0: O in columns [0, D), the maximum and the sum in D + 2 and D + 3.  One
// thread per (row, 4 columns), grid-stride over the sequences' q heads; rows
// of sequences without a prefix are skipped.  The chunk loads of a unit are
// independent, and the unit writes only columns it alone reads (chunk 0's
// own maximum stays in D for the row's other units).
template <int D>
__global__ void __launch_bounds__(256) prefix_merge_kernel(const int32_t *seq_prefix,
                                                           float *part, int batch,
                                                           int num_q_heads, int kc_tiles)
{
    grid_dependency_wait();
    grid_dependents_launch();
    const int64_t cstride = (int64_t)batch * num_q_heads * (D + 4);
    const int64_t units = (int64_t)batch * num_q_heads * (D / 4);
    for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < units;
         u += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = u / (D / 4);
        const int d = (int)(u - row * (D / 4)) * 4;
        const int b = (int)(row / num_q_heads);
        const int P = __ldg(seq_prefix + b);
        if (P <= 0)
            continue;
        const int nkc = ((P + TBK - 1) / TBK + kc_tiles - 1) / kc_tiles;
        float *row0 = part + row * (D + 4);
        float mc[16], M = -INFINITY;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            mc[c] = c < nkc ? __ldcg(row0 + c * cstride + D) : -INFINITY;
            M = fmaxf(M, mc[c]);
        }
        float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        float wsum = 0.0f;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            if (c < nkc) {
                const float w = ex2_approx(mc[c] - M);
                const float4 o = __ldcg(reinterpret_cast<const float4 *>(row0 + c * cstride + d));
                acc.x = fmaf(w, o.x, acc.x);
                acc.y = fmaf(w, o.y, acc.y);
                acc.z = fmaf(w, o.z, acc.z);
                acc.w = fmaf(w, o.w, acc.w);
                if (d == 0)
                    wsum = fmaf(w, __ldcg(row0 + c * cstride + D + 1), wsum);
            }
        }
        *reinterpret_cast<float4 *>(row0 + d) = acc;
        if (d == 0) {
            row0[D + 2] = M;
            row0[D + 3] = wsum;
        }
    }
}

}  // namespace

int launch_prefix_merge(const pkv_pool *pool, const int32_t *seq_prefix, float *part, int batch,
                        int num_q_heads, int kc_tiles, pkv_stream_t stream)
{
    const int64_t units = (int64_t)batch * num_q_heads * (pool->head_dim / 4);
    int64_t blocks = (units + 255) / 256;
    const int64_t cap = (int64_t)pool->num_sms * 8;
    if (blocks > cap)
        blocks = cap;
    if (blocks < 1)
        blocks = 1;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const cudaError_t e =
        pool->head_dim == 64
            ? launch_pdl(prefix_merge_kernel<64>, dim3((unsigned)blocks), dim3(256), 0, s,
                         seq_prefix, part, batch, num_q_heads, kc_tiles)
            : launch_pdl(prefix_merge_kernel<128>, dim3((unsigned)blocks), dim3(256), 0, s,
                         seq_prefix, part, batch, num_q_heads, kc_tiles);
    if (e != cudaSuccess)
        return PKV_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

int launch_prefix_pass(const pkv_pool *pool, const void *q, int num_q_heads, const void *k_cache,
                       const void *v_cache, const int32_t *block_tables, int max_blocks_per_seq,
                       const int32_t *seq_lens, int batch, const int32_t *grp_start,
                       const int32_t *grp_seqs, const int32_t *grp_len, int ngroups,
                       int max_group_size, int max_prefix_len, float scale, float *part,
                       int *kc_tiles_out, pkv_stream_t stream)
{
    PrefillParams prm{};
    prm.q = q;
    prm.k_cache = k_cache;
    prm.v_cache = v_cache;
    prm.block_tables = block_tables;
    prm.seq_lens = seq_lens;
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
    prm.box_rows = pool->block_size < TBK ? pool->block_size : TBK;
    prm.cascade = 1;
    prm.grp_start = grp_start;
    prm.grp_seqs = grp_seqs;
    prm.grp_len = grp_len;
    prm.ngroups = ngroups;
    prm.group_q = num_q_heads / pool->num_kv_heads;
    prm.part = part;
    constexpr int QT = NQH * TBQ;
    prm.nqt = ((int64_t)max_group_size * prm.group_q + QT - 1) / QT;
    // Key chunks of kc_tiles tiles each (the chunks of a row are merged at
    // the end; at most 16, the partials' room): the persistent CTAs take the
    // items in waves of num_sms, so the pass lasts about waves x (kc_tiles
    // + one tile's worth of item setup and output); the chunk size with the
    // least such time wins, the larger on ties (fewer partials to merge).
    const int tiles = std::max(1, (max_prefix_len + TBK - 1) / TBK);
    const int64_t base = (int64_t)prm.nqt * ngroups * pool->num_kv_heads;
    const int64_t sms = std::max(1, pool->num_sms);
    int64_t best_cost = INT64_MAX;
    prm.kc_tiles = tiles;
    for (int kc = tiles; kc >= 1; --kc) {
        const int64_t nkc = (tiles + kc - 1) / kc;
        if (nkc > 16)
            break;
        const int64_t waves = (base * nkc + sms - 1) / sms;
        const int64_t cost = waves * (kc + 1);
        if (cost < best_cost) {
            best_cost = cost;
            prm.kc_tiles = kc;
        }
    }
    prm.nkc = (tiles + prm.kc_tiles - 1) / prm.kc_tiles;
    *kc_tiles_out = prm.kc_tiles;
    const int64_t nitems = (int64_t)prm.nqt * ngroups * pool->num_kv_heads * prm.nkc;
    if (nitems >= ((int64_t)1 << 31))
        return PKV_ERR_UNSUPPORTED;
    prm.nitems = (int)nitems;
    if (!encode_cache_map(&prm.tm_k, pool, k_cache, prm.box_rows) ||
        !encode_cache_map(&prm.tm_v, pool, v_cache, prm.box_rows))
        return PKV_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool bf = pool->kv_dtype == PKV_BF16;
    if (pool->head_dim == 64)
        return bf ? launch_prefill_t<64, __nv_bfloat16>(pool, prm, 0, s)
                  : launch_prefill_t<64, __half>(pool, prm, 0, s);
    return bf ? launch_prefill_t<128, __nv_bfloat16>(pool, prm, 0, s)
              : launch_prefill_t<128, __half>(pool, prm, 0, s);
}

}  // namespace pkv
