// paged_decode_attention: one decode step of attention over a paged KV cache.
//
// What it computes ("KV cache: the engine behind fast LLM inference",
// "Concept" and step 3 of "What happens at each decoding step"): for every
// sequence b and query head h, softmax(scale * q . K^T) . V over all cached
// rows of KV head h / G, the rows reached through the sequence's block table
// (KV cache visualization page, "PagedAttention: the cache in blocks"; query
// heads share KV heads as in its "How much memory", GQA).
//
// How (GB300 design; the pages give no kernel):
//  * Decode reads the whole cache once per step and does little arithmetic
//    per byte (KV cache visualization, "Prefill and decode feel different"),
//    so the kernel is built to stream K/V at HBM bandwidth.  G query heads
//    per K/V byte is far below the tensor ridge, but the instructions per
//    byte are not: with G >= 2 the grouped heads make each 16-token tile a
//    small dense contraction (16 tokens x G heads x d), done as warp-level
//    MMAs that serve all heads of the group from one read of the tile, which
//    cuts the instructions per tile several-fold (fp32 caches and G = 1 stay
//    on the CUDA cores).
//  * The batch's work is a list of work units (1, 2 or 4 16-token tiles of
//    one sequence and KV head, by cache type), ordered by (sequence, KV
//    head, unit).  A persistent grid of one CTA per SM takes a contiguous
//    share of that list (split-K across the sequence axis), the shares
//    balanced by a cost that counts each unit and charges each (sequence,
//    KV head) piece end.
//  * In each CTA one producer warp issues the asynchronous copies of whole
//    K and V units, located through the block table, into a ring of
//    shared-memory stages guarded by mbarriers: 128-byte-swizzled tensor
//    copies for one-tile units, four-row gathers for multi-tile units,
//    plain bulk copies for small blocks (the int8 / int4 scales ride along
//    as 16-byte cp.async copies); 11 consumer warps take units round-robin,
//    each keeping its own online-softmax state (the FlashAttention idea of
//    never materialising the score row, from the guide's "Flash attention:
//    don't build the giant matrix").
//  * At the end of each (sequence, KV head) piece the consumer warps merge
//    their states.  A piece that is the whole sequence is written to `out`;
//    otherwise the CTA stores a partial (max, sum, weighted V) and the last
//    CTA to finish that sequence/head (a counter in the workspace) merges
//    all partials in a fixed order and resets the counter.
//  * Every mbarrier wait is bounded; on timeout the kernel records
//    PKV_EBIT_TIMEOUT, winds down without further waits and lets its own
//    copies drain before exiting.

#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <type_traits>

#include "device_common.cuh"

namespace pkv {
namespace kern {

using namespace dev;

constexpr int TILE = 16;        // tokens per pipeline stage
constexpr int MAX_STAGES = 64;
// misc ints in shared memory: [0] abort flag, [2] a constant zero, [4..6)
// "merge the partials of the first / last piece" flags, [8..32) scan
// scratch, [32..32+MAX_STAGES) last issued round per stage (+1; 0 = never),
// [96..98) q copies issued per slot, [98] number of q copies issued so far
// (they go out in piece order).
constexpr int MISC_ISSUED = 32;
constexpr int MISC_QISSUED = MISC_ISSUED + MAX_STAGES;
constexpr int MISC_QCOUNT = MISC_QISSUED + 2;
constexpr int MISC_INTS = MISC_QCOUNT + 6;

__host__ __device__ constexpr int round_up(int x, int a) { return (x + a - 1) / a * a; }

// Tile math: with G >= 2 query heads per KV head and a 16-bit, 8-bit or
// 4-bit cache, on the tensor cores (warp-level MMA, all heads of the group
// from one read of the tile); with G = 1 (the MMA's head dimension would be
// 1/8 used, and its dependent chain per tile outlasts the CUDA cores' on
// short pieces: 80 against 68 us on the GPT-2-small shape) or an fp32 cache
// (no exact tensor-core type), on the CUDA cores.
__host__ __device__ constexpr bool mma_path(int KV, int G) { return KV != PKV_F32 && G >= 2; }

// Consumer warps per CTA: 11 + the producer.  (The tensor-core tile math
// fits in 128 registers, so 15 consumer warps would fit; measured on the
// workload shapes, 11 are as fast or faster: 52.4 against 56.5 us on the
// Llama-3-8B shape, 120 against 139 us on the Llama-2-70B shape.  The
// CUDA-core tile math takes up to 168 registers.)
__host__ __device__ constexpr int consumer_warps(int G, int KV)
{
    return 11;
}

// Bits of one cached element.
template <int KV>
struct KvBits;
template <> struct KvBits<PKV_F32> { static constexpr int v = 32; };
template <> struct KvBits<PKV_F16> { static constexpr int v = 16; };
template <> struct KvBits<PKV_BF16> { static constexpr int v = 16; };
template <> struct KvBits<PKV_I8> { static constexpr int v = 8; };
template <> struct KvBits<PKV_I4> { static constexpr int v = 4; };

// Quantized caches carry one fp16 scale per cached row.
__host__ __device__ constexpr bool quantized(int KV) { return KV == PKV_I8 || KV == PKV_I4; }

template <int D, int G, int KV>
struct Cfg {
    static constexpr bool MMA = mma_path(KV, G);
    static constexpr int W = consumer_warps(G, KV);
    static constexpr int NTHREADS = (W + 1) * 32;
    static constexpr int ROWB = D * KvBits<KV>::v / 8;   // bytes of one cached row
    static constexpr int NCH = ROWB / 16;          // 16-byte chunks per row
    static constexpr int DS = NCH >= 8 ? 8 : NCH;  // lanes sharing one token's dot product
    static constexpr int TQ = 32 / DS;             // token groups per warp
    static constexpr int TPL = TILE / TQ;          // tokens per lane per tile
    static constexpr int CPL = NCH / DS;           // chunks per lane per token
    static constexpr int NP = TPL * G;             // partial dots per lane
    static constexpr int NF = G >= 2 ? G / 2 : 1;  // scores per lane after reduction
    static constexpr int VE = D / 32;              // V elements per lane
    // A work unit (what a stage holds and a consumer warp takes) is SUB
    // tiles of one (sequence, KV head): on the tensor cores 4 for 4-bit and
    // 2 for 8-bit caches, whose 16-token tiles are only 1 or 2 KB of K (so
    // many small copies are bound by the copy unit's rate per copy and by
    // the producer's work per stage); on the CUDA cores 2 for tiles of at
    // most 2 KB; else 1.
    static constexpr int SUB = mma_path(KV, G) ? (KV == PKV_I4 ? 4 : KV == PKV_I8 ? 2 : 1)
                                               : (KV != PKV_F32 && TILE * ROWB <= 2048 ? 2 : 1);
    static constexpr int TT = TILE * SUB;          // tokens per unit
    static constexpr int KV_BYTES = TT * ROWB;     // one unit of K (or V)
    static constexpr int SC_BYTES = quantized(KV) ? TT * 2 : 0;
    // block-table ids (or gathered rows) a producer lane holds per unit
    static constexpr int NIDS = SUB > 1 ? 8 : 4;
    // a stage: the tile's K then V (the scales ride in a ring of their own,
    // so that every stage starts on a 1024-byte boundary)
    static constexpr int STAGE_BYTES = 2 * KV_BYTES;
    // The tensor-core tile math reads rows of 128 or 256 bytes through the
    // 128-byte swizzle: with blocks of >= 16 rows its one-tile stages come
    // by tensor copies that lay them out swizzled (16-byte chunk j of a
    // 128-byte segment s at j ^ (s mod 8)), which spreads the fragment loads
    // over the banks.  (The units' gathered rows are wider than the
    // swizzle's 128-byte span, so they stay plain.)
    static constexpr bool SWIZZLE_OK = mma_path(KV, G) && (ROWB == 128 || ROWB == 256) && SUB == 1;
    static constexpr int QSLOT = round_up(G * D * 4, 128);   // fits any q dtype
    static constexpr int MERGE_FLOATS = W * G * (D + 2);
    // per warp (CUDA-core tile math only): {p, p} pairs of the tile
    // ([TILE][G] float2) + G rescale factors
    static constexpr int PSW = mma_path(KV, G) ? 0 : round_up(TILE * 2 * G + G, 4);
    static constexpr int PS_FLOATS = W * PSW;
    static_assert(NCH >= 4 && (NCH % DS) == 0, "row must split into 16-byte chunks");
    static_assert(TPL * TQ == TILE, "tile split");
};

struct Params {
    // K and V caches as tensors of rows of 128-byte segments, for the
    // swizzled tensor copies (see Cfg::SWIZZLE_OK): {ROWB / e, bs, NB * Hkv}
    // for 128-byte rows, {128 / e, 2, bs, NB * Hkv} for 256-byte rows
    CUtensorMap tm_k, tm_v;
    int swz;            // tiles come swizzled by tensor copies
    const void *q;
    const unsigned char *k_cache;
    const unsigned char *v_cache;
    const __half *k_scales;
    const __half *v_scales;
    const int32_t *block_tables;
    const int32_t *seq_lens;
    float *out;
    float *partials;
    int *counters;
    unsigned int *err;
    int batch;
    int num_q_heads;
    int num_kv_heads;
    int block_size;
    int bs_log2;
    int max_blocks_per_seq;
    int max_seq_len;
    int len_cap;        // min(max_seq_len, max_blocks_per_seq * block_size)
    int window;         // > 0: attend over the last `window` rows only
    // Shared-prefix (cascade) decode: sequence b attends here only over rows
    // [seq_prefix[b], L) and folds in the partial a prefix pass left for its
    // heads over rows [0, seq_prefix[b]) (null: no prefix)
    const int32_t *seq_prefix;
    const float *prefix_part;   // [batch][num_q_heads][D + 4]: O; maximum, sum at D + 2, D + 3
    int num_blocks;
    int q_dtype;
    int q_bytes;
    int nst;
    float scale_log2;   // scale * log2(e): scores live in the log2 domain
};

// Shared-memory carve-up (dynamic), identical on host and device.
struct Layout {
    int stages, scales, qring, merge, ps, pre, lens, tstart, cstart, bars, misc, total;
};

template <int D, int G, int KV>
__host__ __device__ inline Layout make_layout(int nst, int batch, bool prefix)
{
    using C = Cfg<D, G, KV>;
    Layout L;
    int o = 0;
    L.stages = o; o += nst * C::STAGE_BYTES;
    L.scales = o; o += nst * 2 * C::SC_BYTES;      // K then V scales of each stage
    L.qring = o; o += 2 * C::QSLOT;
    // (every region from here on starts on a 16-byte boundary: the ps and
    // prefix-row regions take 16-byte accesses)
    L.merge = o; o += round_up(C::MERGE_FLOATS * 4, 16);
    L.ps = o; o += round_up(C::PS_FLOATS * 4, 16);
    L.pre = o; o += prefix ? round_up(G * (D + 4) * 4, 16) : 0;   // a piece's merged prefix rows
    L.lens = o; o += 2 * batch * 4;        // lengths, then window starts
    L.tstart = o; o += (batch + 1) * 4;
    L.cstart = o; o += (batch + 1) * 4;
    o = round_up(o, 8);
    L.bars = o; o += (2 * nst + 4) * 8;
    L.misc = o; o += MISC_INTS * 4;
    L.total = round_up(o, 128);
    return L;
}

// The end of a piece (the warps wait for the last of them, merge their
// states and write the result) costs about as much as this many work units;
// the split over CTAs charges it, so that a CTA whose share holds many short
// sequences gets fewer units.  Set from timings on GB300 of the workload
// shapes (one KV head's piece end against its units): about 1.4 us a piece
// at G = 4 and 3 us at G = 8 against 0.15-0.17 us a 16-token tile; more, in
// units, at G = 1 (cheap tiles) and with 64-token units (a warp that ends
// a piece late holds the others back by up to a whole unit).
__host__ __device__ constexpr int piece_cost(int G, int sub = 1)
{
    return sub > 1 ? (sub == 4 ? 12 : 10) + (2 + 2 * G) / sub : (G == 1 ? 16 : 2 + 2 * G);
}

// Owner CTA of global tile x when T tiles are split evenly over P CTAs:
// CTA c owns [floor(c*T/P), floor((c+1)*T/P)).
__device__ __forceinline__ int owner_of(int64_t x, int64_t T, int P)
{
    return (int)(((x + 1) * P - 1) / T);
}

// Largest b with tstart[b] <= x (x < tstart[batch]); never an empty sequence.
__device__ __forceinline__ int find_seq(const int *tstart, int batch, int64_t x)
{
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (tstart[mid] <= x) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// ---- per-dtype tile math ----------------------------------------------------

// q held in registers for the QK product, in the lane's chunk order.
template <int D, int G, int KV>
struct QRegs;

// 16-bit K/V: q stays packed; products use the mixed-precision FMA.
template <int D, int G>
struct QRegs16 {
    using C = Cfg<D, G, PKV_BF16>;
    uint4 w[G][C::CPL];
};
template <int D, int G> struct QRegs<D, G, PKV_BF16> : QRegs16<D, G> {};
template <int D, int G> struct QRegs<D, G, PKV_F16> : QRegs16<D, G> {};
template <int D, int G>
struct QRegs<D, G, PKV_F32> { float4 w[G][Cfg<D, G, PKV_F32>::CPL]; };
template <int D, int G>
struct QRegs<D, G, PKV_I8> { float w[G][Cfg<D, G, PKV_I8>::CPL][16]; };
// 4-bit K: q as fp16 pairs in the order the codes are unpacked (pair 4w+k of
// a 32-code chunk holds elements 8w+k and 8w+k+4).
template <int D, int G>
struct QRegs<D, G, PKV_I4> { uint32_t w[G][Cfg<D, G, PKV_I4>::CPL][16]; };

__device__ __forceinline__ float q_elem(const unsigned char *qs, int idx, int q_dtype)
{
    if (q_dtype == PKV_F16)
        return __half2float(reinterpret_cast<const __half *>(qs)[idx]);
    if (q_dtype == PKV_BF16)
        return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(qs)[idx]);
    return reinterpret_cast<const float *>(qs)[idx];
}

template <int D, int G, int KV>
__device__ __forceinline__ void load_q(QRegs<D, G, KV> &qr, const unsigned char *qs, int ds,
                                       int q_dtype)
{
    using C = Cfg<D, G, KV>;
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int c = 0; c < C::CPL; ++c) {
            const int chunk = ds + C::DS * c;
            if constexpr (KV == PKV_BF16 || KV == PKV_F16) {
                qr.w[g][c] = *reinterpret_cast<const uint4 *>(qs + (g * D + chunk * 8) * 2);
            } else if constexpr (KV == PKV_F32) {
                qr.w[g][c] = *reinterpret_cast<const float4 *>(qs + (g * D + chunk * 4) * 4);
            } else if constexpr (KV == PKV_I4) {
#pragma unroll
                for (int pr = 0; pr < 16; ++pr) {
                    const int e0 = g * D + chunk * 32 + 8 * (pr >> 2) + (pr & 3);
                    const __half2 h = __floats2half2_rn(q_elem(qs, e0, q_dtype),
                                                        q_elem(qs, e0 + 4, q_dtype));
                    qr.w[g][c][pr] = *reinterpret_cast<const uint32_t *>(&h);
                }
            } else {
#pragma unroll
                for (int u = 0; u < 16; ++u)
                    qr.w[g][c][u] = q_elem(qs, g * D + chunk * 16 + u, q_dtype);
            }
        }
}

// (a0, a1) += (b0, b1) * (c0, c1) as one packed fp32x2 FMA.
__device__ __forceinline__ void fma2(float &a0, float &a1, float b0, float b1, float c0, float c1)
{
    asm("{\n\t.reg .b64 x, y, z;\n\t"
        "mov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\tmov.b64 z, {%0, %1};\n\t"
        "fma.rn.f32x2 z, x, y, z;\n\tmov.b64 {%0, %1}, z;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// This lane's K chunks of a tile: chunk ds + DS*c of token tq + TQ*ii.
template <int D, int G, int KV>
__device__ __forceinline__ void load_k(uint4 (&kr)[Cfg<D, G, KV>::TPL][Cfg<D, G, KV>::CPL],
                                       const unsigned char *sK, int tq, int ds)
{
    using C = Cfg<D, G, KV>;
#pragma unroll
    for (int ii = 0; ii < C::TPL; ++ii)
#pragma unroll
        for (int c = 0; c < C::CPL; ++c)
            kr[ii][c] = *reinterpret_cast<const uint4 *>(sK + (tq + C::TQ * ii) * C::ROWB +
                                                         (ds + C::DS * c) * 16);
}

// part[ii*G + g] += q[g] . K[token t_ii] over this lane's chunks (held in kr).
template <int D, int G, int KV>
__device__ __forceinline__ void qk_tile(float (&part)[Cfg<D, G, KV>::NP],
                                        const QRegs<D, G, KV> &qr,
                                        const uint4 (&kr)[Cfg<D, G, KV>::TPL][Cfg<D, G, KV>::CPL])
{
    using C = Cfg<D, G, KV>;
#pragma unroll
    for (int ii = 0; ii < C::TPL; ++ii) {
#pragma unroll
        for (int c = 0; c < C::CPL; ++c) {
            const uint4 kw = kr[ii][c];
            if constexpr (KV == PKV_BF16) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float a = part[ii * G + g];
                    a = fma_bf16x2(qr.w[g][c].x, kw.x, a);
                    a = fma_bf16x2(qr.w[g][c].y, kw.y, a);
                    a = fma_bf16x2(qr.w[g][c].z, kw.z, a);
                    a = fma_bf16x2(qr.w[g][c].w, kw.w, a);
                    part[ii * G + g] = a;
                }
            } else if constexpr (KV == PKV_F16) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float a = part[ii * G + g];
                    a = fma_f16x2(qr.w[g][c].x, kw.x, a);
                    a = fma_f16x2(qr.w[g][c].y, kw.y, a);
                    a = fma_f16x2(qr.w[g][c].z, kw.z, a);
                    a = fma_f16x2(qr.w[g][c].w, kw.w, a);
                    part[ii * G + g] = a;
                }
            } else if constexpr (KV == PKV_F32) {
                const float4 kf = *reinterpret_cast<const float4 *>(&kw);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float a = part[ii * G + g];
                    a = fmaf(qr.w[g][c].x, kf.x, a);
                    a = fmaf(qr.w[g][c].y, kf.y, a);
                    a = fmaf(qr.w[g][c].z, kf.z, a);
                    a = fmaf(qr.w[g][c].w, kf.w, a);
                    part[ii * G + g] = a;
                }
            } else if constexpr (KV == PKV_I4) {
                const uint32_t wds[4] = {kw.x, kw.y, kw.z, kw.w};
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint32_t h = i4pair_to_half2(wds[u], k);   // codes 8u+k, 8u+k+4
#pragma unroll
                        for (int g = 0; g < G; ++g)
                            part[ii * G + g] = fma_f16x2(qr.w[g][c][4 * u + k], h,
                                                         part[ii * G + g]);
                    }
            } else {
                // codes -> exact floats two at a time; the dot products as
                // packed fp32x2 FMAs over element pairs (two partial sums per
                // head, added at the end of the chunk)
                float kf[16];
                const uint32_t wds[4] = {kw.x ^ 0x80808080u, kw.y ^ 0x80808080u,
                                         kw.z ^ 0x80808080u, kw.w ^ 0x80808080u};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    i8pair_to_float2<0>(wds[u], kf[4 * u + 0], kf[4 * u + 1]);
                    i8pair_to_float2<1>(wds[u], kf[4 * u + 2], kf[4 * u + 3]);
                }
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float a0 = part[ii * G + g], a1 = 0.0f;
#pragma unroll
                    for (int u = 0; u < 16; u += 2)
                        fma2(a0, a1, qr.w[g][c][u], qr.w[g][c][u + 1], kf[u], kf[u + 1]);
                    part[ii * G + g] = a0 + a1;
                }
            }
        }
    }
}

// Sum partial dots across the DS lanes that split one token's dot product.
// While more than one value is left, each level halves the vector: the lane
// whose MASK bit is set keeps the upper half and sends the lower one, so after
// all levels lane ds holds entries [NF*ds, NF*ds + NF) of the original vector
// (a reduce-scatter).  Once one value is left the remaining levels are a
// butterfly sum.
template <int N, int MASK, int NP>
__device__ __forceinline__ void reduce_scatter(float (&part)[NP], int ds)
{
    if constexpr (MASK >= 1) {
        if constexpr (N >= 2) {
            const bool upper = (ds & MASK) != 0;
#pragma unroll
            for (int j = 0; j < N / 2; ++j) {
                const float send = upper ? part[j] : part[j + N / 2];
                const float keep = upper ? part[j + N / 2] : part[j];
                part[j] = keep + __shfl_xor_sync(FULL_MASK, send, MASK);
            }
            reduce_scatter<N / 2, MASK / 2, NP>(part, ds);
        } else {
            part[0] += __shfl_xor_sync(FULL_MASK, part[0], MASK);
            reduce_scatter<1, MASK / 2, NP>(part, ds);
        }
    }
}

// The lane's VE elements of V row t, as floats.
template <int D, int KV>
__device__ __forceinline__ void load_v(float (&v)[D / 32], const unsigned char *sV, int t,
                                       int lane)
{
    constexpr int VE = D / 32;
    constexpr int ROWB = D * KvBits<KV>::v / 8;
    const unsigned char *p = sV + t * ROWB + lane * VE * KvBits<KV>::v / 8;
    if constexpr (KV == PKV_BF16) {
        if constexpr (VE == 4) {
            const uint2 w = *reinterpret_cast<const uint2 *>(p);
            v[0] = bf16lo(w.x); v[1] = bf16hi(w.x); v[2] = bf16lo(w.y); v[3] = bf16hi(w.y);
        } else {
            const uint32_t w = *reinterpret_cast<const uint32_t *>(p);
            v[0] = bf16lo(w); v[1] = bf16hi(w);
        }
    } else if constexpr (KV == PKV_F16) {
        if constexpr (VE == 4) {
            const uint2 w = *reinterpret_cast<const uint2 *>(p);
            const float2 a = half2_to_float2(w.x), b = half2_to_float2(w.y);
            v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
        } else {
            const float2 a = half2_to_float2(*reinterpret_cast<const uint32_t *>(p));
            v[0] = a.x; v[1] = a.y;
        }
    } else if constexpr (KV == PKV_F32) {
        if constexpr (VE == 4) {
            const float4 w = *reinterpret_cast<const float4 *>(p);
            v[0] = w.x; v[1] = w.y; v[2] = w.z; v[3] = w.w;
        } else {
            const float2 w = *reinterpret_cast<const float2 *>(p);
            v[0] = w.x; v[1] = w.y;
        }
    } else if constexpr (KV == PKV_I4) {
        static_assert(VE == 4, "4-bit rows are d = 128");
        const uint32_t b = *reinterpret_cast<const uint16_t *>(p);
#pragma unroll
        for (int e = 0; e < 4; ++e)
            v[e] = i4_to_float(b >> (4 * e));
    } else {
        if constexpr (VE == 4) {
            const uint32_t b = *reinterpret_cast<const uint32_t *>(p) ^ 0x80808080u;
            i8pair_to_float2<0>(b, v[0], v[1]);
            i8pair_to_float2<1>(b, v[2], v[3]);
        } else {
            const uint32_t b = (uint32_t)(*reinterpret_cast<const uint16_t *>(p)) ^ 0x8080u;
            i8pair_to_float2<0>(b, v[0], v[1]);
        }
    }
}

// Raw bytes of the lane's VE elements of one V row, when they fit in 8 bytes
// (every case but fp32 with d = 128): a warp copies its V columns of the
// whole tile into registers and releases the stage before the arithmetic.
template <int D, int KV>
struct VRaw {
    static constexpr int BYTES = (D / 32) * KvBits<KV>::v / 8;
    static constexpr bool IN_REGS = BYTES <= 8;
    using type = typename std::conditional<(BYTES <= 4), uint32_t, uint2>::type;
};

template <int D, int KV>
__device__ __forceinline__ typename VRaw<D, KV>::type load_v_raw(const unsigned char *sV, int t,
                                                                 int lane)
{
    constexpr int BYTES = VRaw<D, KV>::BYTES;
    const unsigned char *p = sV + t * (D * KvBits<KV>::v / 8) + lane * BYTES;
    if constexpr (BYTES == 8)
        return *reinterpret_cast<const uint2 *>(p);
    else if constexpr (BYTES == 4)
        return *reinterpret_cast<const uint32_t *>(p);
    else
        return (uint32_t)(*reinterpret_cast<const uint16_t *>(p));
}

template <int D, int KV>
__device__ __forceinline__ void unpack_v(float (&v)[D / 32], typename VRaw<D, KV>::type raw)
{
    constexpr int VE = D / 32;
    if constexpr (KV == PKV_BF16) {
        if constexpr (VE == 4) {
            v[0] = bf16lo(raw.x); v[1] = bf16hi(raw.x); v[2] = bf16lo(raw.y); v[3] = bf16hi(raw.y);
        } else {
            v[0] = bf16lo(raw); v[1] = bf16hi(raw);
        }
    } else if constexpr (KV == PKV_F16) {
        if constexpr (VE == 4) {
            const float2 a = half2_to_float2(raw.x), b = half2_to_float2(raw.y);
            v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
        } else {
            const float2 a = half2_to_float2(raw);
            v[0] = a.x; v[1] = a.y;
        }
    } else if constexpr (KV == PKV_F32) {
        static_assert(VE == 2, "fp32 rows of d = 128 are read from shared memory");
        v[0] = __uint_as_float(raw.x); v[1] = __uint_as_float(raw.y);
    } else if constexpr (KV == PKV_I4) {
        static_assert(VE == 4, "4-bit rows are d = 128");
#pragma unroll
        for (int e = 0; e < 4; ++e)
            v[e] = i4_to_float(raw >> (4 * e));
    } else {
        if constexpr (VE == 4) {
            const uint32_t b = raw ^ 0x80808080u;
            i8pair_to_float2<0>(b, v[0], v[1]);
            i8pair_to_float2<1>(b, v[2], v[3]);
        } else {
            const uint32_t b = raw ^ 0x8080u;
            i8pair_to_float2<0>(b, v[0], v[1]);
        }
    }
}

// 2^x with the hardware approximation (relative error ~2^-22; -inf -> +0).
__device__ __forceinline__ float exp2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The 16 rows at row `y` of (block, head) `z` as one tensor copy with the
// 128-byte swizzle into shared memory at dst (1024-byte aligned): 3-D view
// {128-byte row, bs, NB * Hkv} for 128-byte rows, 4-D {128 bytes, 2, bs,
// NB * Hkv} for 256-byte rows.  Completion is counted in bytes on the
// mbarrier; `policy` is an L2 cache hint.
template <int ROWB>
__device__ __forceinline__ void tma_tile_swz(void *dst, const CUtensorMap *map, int y, int z,
                                             uint64_t *bar, uint64_t policy)
{
    if constexpr (ROWB == 128) {
        asm volatile(
            "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
            ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
            "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(y), "r"(z), "r"(smem_addr(bar)),
            "l"(policy)
            : "memory");
    } else {
        static_assert(ROWB == 256, "swizzled tiles have rows of 128 or 256 bytes");
        asm volatile(
            "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
            ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_addr(dst)),
            "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(0), "r"(y), "r"(z),
            "r"(smem_addr(bar)), "l"(policy)
            : "memory");
    }
}

// Byte offset of a 16-byte chunk inside a tile laid out by the swizzled
// tensor copies (128-byte swizzle: chunk bits 4-6 xor segment bits 7-9), or
// unchanged for a plain tile.
__device__ __forceinline__ uint32_t swz_off(uint32_t off, bool swz)
{
    return swz ? off ^ ((off >> 3) & 0x70u) : off;
}

// Tokens per row of the gather view of the caches for units of tt tokens:
// a block's tokens, at most 16, at most a quarter unit (so that a unit is
// four or eight rows).
__host__ __device__ constexpr int gather_row_tokens(int bs, int tt)
{
    return bs < TILE ? (bs < tt / 4 ? bs : tt / 4) : (TILE < tt / 4 ? TILE : tt / 4);
}

// Four rows of a 2-D view of a cache (x = 0, rows r0..r3) as one gather copy
// into shared memory at dst, laid out one after another; completion is
// counted in bytes on the mbarrier; `policy` is an L2 cache hint.
__device__ __forceinline__ void tma_gather4(void *dst, const CUtensorMap *map, int r0, int r1,
                                            int r2, int r3, uint64_t *bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(r0), "r"(r1), "r"(r2), "r"(r3),
        "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// ---- tile math on the tensor cores (warp-level MMA) --------------------------
//
// For 16-bit, 8-bit and 4-bit caches a warp does a tile's two products as
// m16n8k16 MMAs with fp32 accumulation (the scores and outputs of all G <= 8
// heads of the group at once):
//   S^T = K q^T:   M = the tile's 16 tokens, N = the heads (padded to 8),
//                  K = 16 elements of d per MMA;
//   O^T += V^T P^T: M = 16 output elements, N = the heads, K = the 16 tokens.
// Fragment layout (PTX m16n8k16, .row.col): with gid = lane / 4 and
// tig = lane % 4, A holds (row gid | gid+8, k 2tig..2tig+1 | 2tig+8..2tig+9),
// B holds (k 2tig..2tig+1 | 2tig+8..2tig+9, column gid), C holds (row gid |
// gid+8, columns 2tig, 2tig+1).  Two freedoms keep the shared-memory reads
// plain 16-byte loads of the rows as the bulk copies left them:
//  * the order of d inside q.K is free (the same permutation on both
//    operands): lane tig takes a contiguous quarter of every K row and of q;
//  * the output elements a row of O^T stands for are free: lane gid owns the
//    contiguous eighth [gid D/8, (gid+1) D/8) of d, m-tile j's rows gid and
//    gid+8 being elements gid D/8 + 2j and + 2j + 1.
// S^T comes out with a lane holding two tokens x two heads; one 8x8
// transpose (movmatrix) per half tile turns the packed weights into the B
// fragment of P^T.  Weights are split into a high and a low part of the MMA
// type (p = hi + lo to ~2^-16 relative) and both are multiplied, so that the
// weights' rounding stays far inside the error budget; for the same reason a
// q whose type differs from the cache's is split the same way.  The products
// of 16-bit (or exactly converted int8 / int4) operands are exact in fp32.

// The MMA operand type of a cache: bf16 for bf16 caches, else fp16 (int8 and
// int4 codes are exact in fp16).
template <int KV>
struct MmaBf16 { static constexpr bool v = KV == PKV_BF16; };

template <bool BF>
__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1)
{
    if constexpr (BF)
        asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, "
                     "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                     : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                     : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    else
        asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, "
                     "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                     : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                     : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 matrix of 16-bit values held one pair per lane (lane
// holds row lane/4, columns 2(lane%4), +1), in the same layout.
__device__ __forceinline__ uint32_t transpose8x8(uint32_t x)
{
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// (x, y) -> packed pairs hi and lo of the MMA type with hi + lo = (x, y) up to
// the rounding of lo (relative 2^-16 for bf16, 2^-22 for fp16).
template <bool BF>
__device__ __forceinline__ void split_pair(float x, float y, uint32_t &hi, uint32_t &lo)
{
    if constexpr (BF) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
        const __nv_bfloat162 l = __floats2bfloat162_rn(x - __low2float(h), y - __high2float(h));
        hi = *reinterpret_cast<const uint32_t *>(&h);
        lo = *reinterpret_cast<const uint32_t *>(&l);
    } else {
        const __half2 h = __floats2half2_rn(x, y);
        const __half2 l = __floats2half2_rn(x - __low2float(h), y - __high2float(h));
        hi = *reinterpret_cast<const uint32_t *>(&h);
        lo = *reinterpret_cast<const uint32_t *>(&l);
    }
}

// Two biased int8 codes (code ^ 0x80) picked by SEL from a word -> an exact
// fp16 pair: the biased byte becomes the low mantissa bits of 1024 (0x64 in
// the high byte) and 1152 = 1024 + 128 (0x6480) is subtracted.  SEL 0x4140
// takes bytes 0, 1; 0x4342 bytes 2, 3.
template <uint32_t SEL>
__device__ __forceinline__ uint32_t i8pair_to_half2(uint32_t biased)
{
    const uint32_t t = __byte_perm(biased, 0x64646464u, SEL);
    uint32_t h;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(h) : "r"(t), "r"(0x64806480u));
    return h;
}

template <int D, int KV>
struct MmaCfg {
    static constexpr int ROWB = D * KvBits<KV>::v / 8;   // bytes of one cached row
    static constexpr int KQB = ROWB / 4;                  // a lane's quarter of a K row
    static constexpr int KCH = KQB / 16;                  // its 16-byte chunks
    static constexpr int KS = D / 16;                     // k-steps of q.K (16 elements each)
    static constexpr int VB = ROWB / 8;                   // a lane's eighth of a V row
    static constexpr int MT = D / 16;                     // m-tiles of O^T
    // 16-bit rows of d = 128 are read in a chunk order rotated by lane pairs,
    // which spreads a quarter-warp's 16-byte reads over all banks but the
    // two tokens' (2-way conflict instead of 4-way)
    static constexpr bool ROTATE = KvBits<KV>::v == 16 && KCH == 4;
    static_assert(KCH >= 1 || KV == PKV_I4, "K quarter rows are whole 16-byte chunks");
};

// Element of d (within the lane's quarter of the row, offset tig * D / 4)
// that element u of half h of the q B fragment of k-step ks stands for; the
// same element the K A fragment's pair holds.
template <int D, int KV>
__device__ __forceinline__ int q_elem_index(int ks, int h, int u, int rot)
{
    if constexpr (KvBits<KV>::v == 16) {
        // chunk slot ks / 2 (holding chunk (ks / 2 + rot) mod KCH); words
        // 2 (ks % 2) + h of it
        constexpr int KCH = MmaCfg<D, KV>::KCH;
        const int chunk = ((ks >> 1) + rot) & (KCH - 1);
        return 8 * chunk + 4 * (ks & 1) + 2 * h + u;
    } else if constexpr (KV == PKV_I8) {
        return 4 * ks + 2 * h + u;                       // word ks, bytes 2h + u
    } else {
        // 4-bit: word w = ks / 2 holds codes 8w..8w+7; pair k = 2 (ks % 2) + h
        // is codes (8w + k, 8w + k + 4)
        return 8 * (ks >> 1) + 2 * (ks & 1) + h + 4 * u;
    }
}

template <int D, int G, int KV, bool QS>
struct MmaState {
    uint32_t qh[D / 16][2];                 // q B fragments (high part)
    uint32_t ql[QS ? D / 16 : 1][2];        // low part (q of another type only)
    float acc[D / 16][4];                   // O^T C fragments
    float m[2], l[2];                       // heads 2 tig, 2 tig + 1 (l: this lane's tokens)
};

// q of the piece's G heads (in shared memory, q_dtype) -> B fragments.
// With G < 8 the MMA's 8 head columns repeat the G heads (column n holds
// head n mod G), so that every column's scores, maxima and sums are a real
// head's: the P.V step then carries the weights' low parts in the repeated
// columns (see mma_tile).
template <int D, int G, int KV, bool QS>
__device__ __forceinline__ void load_q_mma(MmaState<D, G, KV, QS> &st, const unsigned char *qs,
                                           int q_dtype, int lane)
{
    constexpr bool BF = MmaBf16<KV>::v;
    const int gid = lane >> 2, tig = lane & 3;
    const int rot = MmaCfg<D, KV>::ROTATE ? (tig >> 1) * 2 : 0;
    const int base = (gid % G) * D + tig * (D / 4);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float x0 = q_elem(qs, base + q_elem_index<D, KV>(ks, h, 0, rot), q_dtype);
            const float x1 = q_elem(qs, base + q_elem_index<D, KV>(ks, h, 1, rot), q_dtype);
            uint32_t hi, lo;
            split_pair<BF>(x0, x1, hi, lo);
            st.qh[ks][h] = hi;
            if constexpr (QS)
                st.ql[ks][h] = lo;
        }
}

// Words of a lane's eighth of a V row (>= 2).
template <int D, int KV>
struct VFrag {
    static constexpr int VW = (MmaCfg<D, KV>::VB + 3) / 4;
};

// S^T = K q^T of one 16-token tile at sK: rows gid, gid + 8 of the tile, the
// lane's quarter of d; accumulated into s (heads 2tig, 2tig + 1).
template <int D, int G, int KV, bool QS>
__device__ __forceinline__ void mma_scores(float (&s)[4], const MmaState<D, G, KV, QS> &st,
                                           const unsigned char *sK, int lane, bool sw)
{
    using M = MmaCfg<D, KV>;
    constexpr bool BF = MmaBf16<KV>::v;
    constexpr int ROWB = M::ROWB;
    const int gid = lane >> 2, tig = lane & 3;
    {
        const uint32_t k0 = gid * ROWB + tig * M::KQB;
        const uint32_t k1 = k0 + 8 * ROWB;
        if constexpr (KvBits<KV>::v == 16) {
            const int rot = M::ROTATE ? (tig >> 1) * 2 : 0;
#pragma unroll
            for (int c = 0; c < M::KCH; ++c) {
                const int ch = (c + rot) & (M::KCH - 1);
                const uint4 x = *reinterpret_cast<const uint4 *>(sK + swz_off(k0 + ch * 16, sw));
                const uint4 y = *reinterpret_cast<const uint4 *>(sK + swz_off(k1 + ch * 16, sw));
                mma_16816<BF>(s, x.x, y.x, x.y, y.y, st.qh[2 * c][0], st.qh[2 * c][1]);
                mma_16816<BF>(s, x.z, y.z, x.w, y.w, st.qh[2 * c + 1][0], st.qh[2 * c + 1][1]);
                if constexpr (QS) {
                    mma_16816<BF>(s, x.x, y.x, x.y, y.y, st.ql[2 * c][0], st.ql[2 * c][1]);
                    mma_16816<BF>(s, x.z, y.z, x.w, y.w, st.ql[2 * c + 1][0],
                                  st.ql[2 * c + 1][1]);
                }
            }
        } else if constexpr (KV == PKV_I8) {
#pragma unroll
            for (int c = 0; c < M::KCH; ++c) {
                const uint4 x = *reinterpret_cast<const uint4 *>(sK + swz_off(k0 + c * 16, sw));
                const uint4 y = *reinterpret_cast<const uint4 *>(sK + swz_off(k1 + c * 16, sw));
                const uint32_t xw[4] = {x.x ^ 0x80808080u, x.y ^ 0x80808080u, x.z ^ 0x80808080u,
                                        x.w ^ 0x80808080u};
                const uint32_t yw[4] = {y.x ^ 0x80808080u, y.y ^ 0x80808080u, y.z ^ 0x80808080u,
                                        y.w ^ 0x80808080u};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int ks = 4 * c + i;
                    const uint32_t a0 = i8pair_to_half2<0x4140u>(xw[i]);
                    const uint32_t a2 = i8pair_to_half2<0x4342u>(xw[i]);
                    const uint32_t a1 = i8pair_to_half2<0x4140u>(yw[i]);
                    const uint32_t a3 = i8pair_to_half2<0x4342u>(yw[i]);
                    mma_16816<BF>(s, a0, a1, a2, a3, st.qh[ks][0], st.qh[ks][1]);
                    if constexpr (QS)
                        mma_16816<BF>(s, a0, a1, a2, a3, st.ql[ks][0], st.ql[ks][1]);
                }
            }
        } else {
            static_assert(KV == PKV_I4 && D == 128, "4-bit rows are d = 128");
            const uint4 x = *reinterpret_cast<const uint4 *>(sK + k0);
            const uint4 y = *reinterpret_cast<const uint4 *>(sK + k1);
            const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
            const uint32_t yw[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                // pair k of word w (codes k, k + 4): k = 0, 1 from the word,
                // k = 2, 3 from the word shifted down a byte
                const int w = ks >> 1;
                const uint32_t xs = (ks & 1) ? xw[w] >> 8 : xw[w];
                const uint32_t ys = (ks & 1) ? yw[w] >> 8 : yw[w];
                const uint32_t a0 = i4pair_lo_to_half2(xs);
                const uint32_t a2 = i4pair_hi_to_half2(xs);
                const uint32_t a1 = i4pair_lo_to_half2(ys);
                const uint32_t a3 = i4pair_hi_to_half2(ys);
                mma_16816<BF>(s, a0, a1, a2, a3, st.qh[ks][0], st.qh[ks][1]);
                if constexpr (QS)
                    mma_16816<BF>(s, a0, a1, a2, a3, st.ql[ks][0], st.ql[ks][1]);
            }
        }
    }
}

// The lane's eighth of the V rows of tokens 2tig, 2tig+1, 2tig+8, 2tig+9 of
// the tile at sV.
template <int D, int KV>
__device__ __forceinline__ void load_v_frag(uint32_t (&vw)[4][VFrag<D, KV>::VW],
                                            const unsigned char *sV, int lane, bool sw)
{
    using M = MmaCfg<D, KV>;
    constexpr int ROWB = M::ROWB;
    const int gid = lane >> 2, tig = lane & 3;
    {
        const int toks[4] = {2 * tig, 2 * tig + 1, 2 * tig + 8, 2 * tig + 9};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t v0 = toks[i] * ROWB + gid * M::VB;
            const unsigned char *p = sV + v0;
            if constexpr (M::VB >= 16) {
#pragma unroll
                for (int c = 0; c < M::VB / 16; ++c) {
                    const uint4 x =
                        *reinterpret_cast<const uint4 *>(sV + swz_off(v0 + 16 * c, sw));
                    vw[i][4 * c] = x.x; vw[i][4 * c + 1] = x.y;
                    vw[i][4 * c + 2] = x.z; vw[i][4 * c + 3] = x.w;
                }
            } else {
                const uint2 x = *reinterpret_cast<const uint2 *>(p);
                vw[i][0] = x.x; vw[i][1] = x.y;
            }
        }
    }
}

// O^T += V^T P^T for one tile: vw from load_v_frag, p0..p3 the weights of
// (token gid, heads 2tig, 2tig+1), (token gid + 8, the same heads).
template <int D, int G, int KV, bool QS>
__device__ __forceinline__ void mma_pv(MmaState<D, G, KV, QS> &st,
                                       const uint32_t (&vw)[4][VFrag<D, KV>::VW], float p0,
                                       float p1, float p2, float p3, int lane)
{
    using M = MmaCfg<D, KV>;
    constexpr bool BF = MmaBf16<KV>::v;
    // P^T as the B fragment: (token gid | gid+8, heads 2tig, 2tig+1) pairs,
    // transposed to (tokens 2tig, 2tig+1 | +8, head gid).  G = 8: the high
    // and the low parts are two B fragments, two MMAs per m-tile.  G < 8:
    // one fragment whose columns [0, G) hold the high parts and [G, 2G) the
    // low parts of the same heads (columns n and n + G hold one head), the
    // rest zero: one MMA per m-tile, the two sums added at the piece's end.
    const int tig = lane & 3;
    uint32_t ph0, pl0, ph1, pl1;
    split_pair<BF>(p0, p1, ph0, pl0);
    split_pair<BF>(p2, p3, ph1, pl1);
    constexpr bool PACK = G < 8;
    uint32_t bh0, bh1, bl0 = 0u, bl1 = 0u;
    if constexpr (PACK) {
        const bool hi_cols = 2 * tig < G, lo_cols = !hi_cols && 2 * tig < 2 * G;
        bh0 = transpose8x8(hi_cols ? ph0 : (lo_cols ? pl0 : 0u));
        bh1 = transpose8x8(hi_cols ? ph1 : (lo_cols ? pl1 : 0u));
    } else {
        bh0 = transpose8x8(ph0);
        bh1 = transpose8x8(ph1);
        bl0 = transpose8x8(pl0);
        bl1 = transpose8x8(pl1);
    }

    // ---- O^T += V^T P^T, m-tile j: rows gid, gid+8 = elements 2j, 2j+1 of
    // the lane's eighth of d
#pragma unroll
    for (int j = 0; j < M::MT; ++j) {
        uint32_t a0, a1, a2, a3;
        if constexpr (KvBits<KV>::v == 16) {
            a0 = __byte_perm(vw[0][j], vw[1][j], 0x5410u);
            a1 = __byte_perm(vw[0][j], vw[1][j], 0x7632u);
            a2 = __byte_perm(vw[2][j], vw[3][j], 0x5410u);
            a3 = __byte_perm(vw[2][j], vw[3][j], 0x7632u);
        } else if constexpr (KV == PKV_I8) {
            // bytes 2j, 2j+1 of the token's eighth: word j / 2
            const int w = j >> 1;
            const uint32_t xa = vw[0][w] ^ 0x80808080u, xb = vw[1][w] ^ 0x80808080u;
            const uint32_t xc = vw[2][w] ^ 0x80808080u, xd = vw[3][w] ^ 0x80808080u;
            // interleave the two tokens' bytes: (A.b, B.b, A.b', B.b')
            const uint32_t tab = (j & 1) ? __byte_perm(xa, xb, 0x7362u) : __byte_perm(xa, xb, 0x5140u);
            const uint32_t tcd = (j & 1) ? __byte_perm(xc, xd, 0x7362u) : __byte_perm(xc, xd, 0x5140u);
            a0 = i8pair_to_half2<0x4140u>(tab);
            a1 = i8pair_to_half2<0x4342u>(tab);
            a2 = i8pair_to_half2<0x4140u>(tcd);
            a3 = i8pair_to_half2<0x4342u>(tcd);
        } else {
            // codes 2j, 2j+1 of the token's eighth (16 codes in two words)
            // are byte j of it: that byte of the two tokens goes to bytes 0
            // and 2 of one word (low nibbles: code 2j; high: code 2j + 1)
            const int w = j >> 2, b = j & 3;
            const uint32_t sel = (uint32_t)b | ((uint32_t)(b + 4) << 8);
            const uint32_t tab = __byte_perm(vw[0][w], vw[1][w], sel);
            const uint32_t tcd = __byte_perm(vw[2][w], vw[3][w], sel);
            a0 = i4pair_lo_to_half2(tab);
            a1 = i4pair_hi_to_half2(tab);
            a2 = i4pair_lo_to_half2(tcd);
            a3 = i4pair_hi_to_half2(tcd);
        }
        mma_16816<BF>(st.acc[j], a0, a1, a2, a3, bh0, bh1);
        if constexpr (!PACK)
            mma_16816<BF>(st.acc[j], a0, a1, a2, a3, bl0, bl1);
    }
}

// One 16-token tile: scores, online softmax, weighted V.  nvalid: tokens of
// the tile inside the sequence; tlo: first token inside the window.  The
// stage is released (empty barrier) as soon as its last byte has been read.
template <int D, int G, int KV, bool QS>
__device__ __forceinline__ void mma_tile(MmaState<D, G, KV, QS> &st, const unsigned char *sK,
                                         const unsigned char *sV, const __half *sKS,
                                         const __half *sVS, int nvalid, int tlo, float scale_log2,
                                         int lane, uint64_t *empty_bar, int swz,
                                         bool release = true)
{
    using M = MmaCfg<D, KV>;
    constexpr int ROWB = M::ROWB;
    constexpr int VW = VFrag<D, KV>::VW;
    const int gid = lane >> 2, tig = lane & 3;

    // (tiles laid out by the swizzled tensor copies: chunk addresses go
    // through swz_off)
    constexpr bool CAN_SWZ = mma_path(KV, G) && (ROWB == 128 || ROWB == 256);
    const bool sw = CAN_SWZ && swz != 0;

    float s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    mma_scores<D, G, KV, QS>(s, st, sK, lane, sw);

    // ---- V and the scales; then the stage goes back to the producer
    uint32_t vw[4][VW];
    load_v_frag<D, KV>(vw, sV, lane, sw);
    if constexpr (KvBits<KV>::v == 16) {
        // rows past the sequence end may hold anything (0 * NaN is NaN)
        if (nvalid < TILE) {
            const int toks[4] = {2 * tig, 2 * tig + 1, 2 * tig + 8, 2 * tig + 9};
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (toks[i] >= nvalid)
#pragma unroll
                    for (int u = 0; u < VW; ++u)
                        vw[i][u] = 0u;
        }
    }
    float ks0 = 1.0f, ks1 = 1.0f, vs0 = 1.0f, vs1 = 1.0f;
    if constexpr (quantized(KV)) {
        ks0 = __half2float(sKS[gid]);
        ks1 = __half2float(sKS[gid + 8]);
        vs0 = __half2float(sVS[gid]);
        vs1 = __half2float(sVS[gid + 8]);
    }
    if (release) {
        __syncwarp();
        if (lane == 0)
            mbar_arrive(empty_bar);
    }

    // ---- online softmax (log2 domain) of heads 2tig, 2tig+1 over tokens
    // gid, gid+8 of this lane; the other lanes of the head differ in gid
    const bool v0 = gid < nvalid && gid >= tlo;
    const bool v1 = gid + 8 < nvalid && gid + 8 >= tlo;
    const float sc0 = scale_log2 * ks0, sc1 = scale_log2 * ks1;
    const float x0 = v0 ? s[0] * sc0 : -INFINITY;   // token gid, head 2tig
    const float x1 = v0 ? s[1] * sc0 : -INFINITY;   // token gid, head 2tig + 1
    const float x2 = v1 ? s[2] * sc1 : -INFINITY;   // token gid + 8, head 2tig
    const float x3 = v1 ? s[3] * sc1 : -INFINITY;   // token gid + 8, head 2tig + 1
    const bool above = fmaxf(x0, x2) > st.m[0] || fmaxf(x1, x3) > st.m[1];
    if (__any_sync(FULL_MASK, above)) {
        // the running maxima move (softmax is shift invariant: any running
        // value that is one of the scores seen is exact)
        float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
        for (int mask = 4; mask < 32; mask <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(FULL_MASK, mx0, mask));
            mx1 = fmaxf(mx1, __shfl_xor_sync(FULL_MASK, mx1, mask));
        }
        const float n0 = fmaxf(st.m[0], mx0), n1 = fmaxf(st.m[1], mx1);
        const float c0 = exp2_approx(st.m[0] - n0), c1 = exp2_approx(st.m[1] - n1);
        st.m[0] = n0;
        st.m[1] = n1;
        st.l[0] *= c0;
        st.l[1] *= c1;
#pragma unroll
        for (int j = 0; j < M::MT; ++j) {
            st.acc[j][0] *= c0;
            st.acc[j][2] *= c0;
            st.acc[j][1] *= c1;
            st.acc[j][3] *= c1;
        }
    }
    float p0 = exp2_approx(x0 - st.m[0]), p1 = exp2_approx(x1 - st.m[1]);
    float p2 = exp2_approx(x2 - st.m[0]), p3 = exp2_approx(x3 - st.m[1]);
    st.l[0] += p0 + p2;
    st.l[1] += p1 + p3;
    if constexpr (quantized(KV)) {
        // V codes are dequantized through the weights: p * s_v of the token
        p0 = v0 ? p0 * vs0 : 0.0f;
        p1 = v0 ? p1 * vs0 : 0.0f;
        p2 = v1 ? p2 * vs1 : 0.0f;
        p3 = v1 ? p3 * vs1 : 0.0f;
    }
    mma_pv<D, G, KV, QS>(st, vw, p0, p1, p2, p3, lane);
}

// A unit of NS 16-token tiles of a quantized cache (the tiles [i0, i1) hold
// attended tokens; the others are neither read nor scored): the scores of
// all its tiles first (NS independent MMA chains), one update of the running
// maxima over the unit, then the weighted V of each tile, its V read from
// the stage just before its MMAs.  The stage goes back to the producer after
// the last V read.  (Used for 2-tile units: with 4-tile units of 4-bit
// codes, and with the units' V taken into registers before the softmax so
// that the stage goes back earlier, it was slower than tile by tile.)
template <int D, int G, int KV, bool QS, int NS>
__device__ __forceinline__ void mma_unit(MmaState<D, G, KV, QS> &st, const unsigned char *sK,
                                         const unsigned char *sV, const __half *sKS,
                                         const __half *sVS, int nvalid, int tlo, float scale_log2,
                                         int lane, uint64_t *empty_bar)
{
    static_assert(quantized(KV), "multi-tile units of the tensor-core path are quantized");
    using M = MmaCfg<D, KV>;
    constexpr int TB = TILE * M::ROWB;
    constexpr int VW = VFrag<D, KV>::VW;
    const int gid = lane >> 2;
    const int i0 = tlo > 0 ? tlo / TILE : 0;
    const int i1 = (nvalid + TILE - 1) / TILE;

    // ---- scores (log2 domain) of tokens gid, gid + 8 of every tile
    float x[NS][4];
    bool above = false;
#pragma unroll
    for (int i = 0; i < NS; ++i) {
        float s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if (i >= i0 && i < i1)
            mma_scores<D, G, KV, QS>(s, st, sK + i * TB, lane, false);
        const int t0 = i * TILE + gid, t1 = t0 + 8;
        const bool v0 = t0 < nvalid && t0 >= tlo;
        const bool v1 = t1 < nvalid && t1 >= tlo;
        const float sc0 = scale_log2 * __half2float(sKS[t0]);
        const float sc1 = scale_log2 * __half2float(sKS[t1]);
        x[i][0] = v0 ? s[0] * sc0 : -INFINITY;   // token t0, head 2tig
        x[i][1] = v0 ? s[1] * sc0 : -INFINITY;   // token t0, head 2tig + 1
        x[i][2] = v1 ? s[2] * sc1 : -INFINITY;   // token t1, head 2tig
        x[i][3] = v1 ? s[3] * sc1 : -INFINITY;   // token t1, head 2tig + 1
        above |= fmaxf(x[i][0], x[i][2]) > st.m[0] || fmaxf(x[i][1], x[i][3]) > st.m[1];
    }
    if (__any_sync(FULL_MASK, above)) {
        // the running maxima move (softmax is shift invariant: any running
        // value that is one of the scores seen is exact)
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int i = 0; i < NS; ++i) {
            mx0 = fmaxf(mx0, fmaxf(x[i][0], x[i][2]));
            mx1 = fmaxf(mx1, fmaxf(x[i][1], x[i][3]));
        }
#pragma unroll
        for (int mask = 4; mask < 32; mask <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(FULL_MASK, mx0, mask));
            mx1 = fmaxf(mx1, __shfl_xor_sync(FULL_MASK, mx1, mask));
        }
        const float n0 = fmaxf(st.m[0], mx0), n1 = fmaxf(st.m[1], mx1);
        const float c0 = exp2_approx(st.m[0] - n0), c1 = exp2_approx(st.m[1] - n1);
        st.m[0] = n0;
        st.m[1] = n1;
        st.l[0] *= c0;
        st.l[1] *= c1;
#pragma unroll
        for (int j = 0; j < M::MT; ++j) {
            st.acc[j][0] *= c0;
            st.acc[j][2] *= c0;
            st.acc[j][1] *= c1;
            st.acc[j][3] *= c1;
        }
    }

    // ---- weights and weighted V, tile by tile
#pragma unroll
    for (int i = 0; i < NS; ++i) {
        if (i >= i0 && i < i1) {
            uint32_t vw[4][VW];
            load_v_frag<D, KV>(vw, sV + i * TB, lane, false);
            const int t0 = i * TILE + gid, t1 = t0 + 8;
            const bool v0 = t0 < nvalid && t0 >= tlo;
            const bool v1 = t1 < nvalid && t1 >= tlo;
            float p0 = exp2_approx(x[i][0] - st.m[0]), p1 = exp2_approx(x[i][1] - st.m[1]);
            float p2 = exp2_approx(x[i][2] - st.m[0]), p3 = exp2_approx(x[i][3] - st.m[1]);
            st.l[0] += p0 + p2;
            st.l[1] += p1 + p3;
            // V codes are dequantized through the weights: p * s_v of the
            // token (rows outside the attended range may hold any scale)
            const float vs0 = __half2float(sVS[t0]), vs1 = __half2float(sVS[t1]);
            p0 = v0 ? p0 * vs0 : 0.0f;
            p1 = v0 ? p1 * vs0 : 0.0f;
            p2 = v1 ? p2 * vs1 : 0.0f;
            p3 = v1 ? p3 * vs1 : 0.0f;
            mma_pv<D, G, KV, QS>(st, vw, p0, p1, p2, p3, lane);
        }
    }
    __syncwarp();
    if (lane == 0)
        mbar_arrive(empty_bar);
}

// ---- the kernel ---------------------------------------------------------------

// QS: q's type differs from the MMA operand type, so q is split into a high
// and a low part (tensor-core tile math only).
template <int D, int G, int KV, bool QS>
__global__ void __launch_bounds__(Cfg<D, G, KV>::NTHREADS, 1) paged_decode_kernel(const __grid_constant__ Params p)
{
    using C = Cfg<D, G, KV>;
    constexpr int W = C::W;
    constexpr int NTHREADS = C::NTHREADS;
    extern __shared__ __align__(1024) unsigned char smem[];
    const Layout lay = make_layout<D, G, KV>(p.nst, p.batch, p.seq_prefix != nullptr);
    unsigned char *stages = smem + lay.stages;
    unsigned char *scale_ring = smem + lay.scales;
    unsigned char *qring = smem + lay.qring;
    float *merge = reinterpret_cast<float *>(smem + lay.merge);
    float *psbuf = reinterpret_cast<float *>(smem + lay.ps);
    float *s_pre = reinterpret_cast<float *>(smem + lay.pre);
    int *s_len = reinterpret_cast<int *>(smem + lay.lens);
    int *s_lo = s_len + p.batch;   // first attended position (sliding window)
    int *s_tstart = reinterpret_cast<int *>(smem + lay.tstart);
    int *s_cstart = reinterpret_cast<int *>(smem + lay.cstart);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + lay.bars);
    uint64_t *empty = full + p.nst;
    uint64_t *qfull = empty + p.nst;
    uint64_t *qempty = qfull + 2;
    int *misc = reinterpret_cast<int *>(smem + lay.misc);
    volatile int *abort_flag = misc + 0;  // set on any timeout
    // The 128-byte swizzle repeats every 1024 bytes of shared address, and the
    // tile reads assume it starts at a stage's start: without that alignment
    // the tiles come by plain bulk copies instead.
    const int swz = (C::SWIZZLE_OK && p.swz && (smem_addr(smem) & 1023u) == 0) ? 1 : 0;
    // misc[2]: zero word; misc[4..6): "this CTA merges the partials of its
    // first / last piece"; misc[8..]: scan scratch

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int Hkv = p.num_kv_heads;
    const int B = p.batch;

    if (tid == 0) {
        // full: the producer's expect-tx arrival, plus (quantized caches) the
        // arrival that tracks the scales' cp.async copies
        for (int s = 0; s < p.nst; ++s) {
            mbar_init(&full[s], quantized(KV) ? 2 : 1);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&qfull[s], 1);
            mbar_init(&qempty[s], W);
        }
        for (int i = 0; i < MISC_INTS; ++i)
            misc[i] = 0;
        mbar_fence_init();
    }

    // Everything above touched shared memory only; global inputs may come
    // from the previous kernel in the stream.
    grid_dependency_wait();
    grid_dependents_launch();

    // Sequence lengths (validated) and the exclusive prefix of tiles.
    for (int b = tid; b < B; b += NTHREADS) {
        int L = __ldg(p.seq_lens + b);
        if (L < 0 || L > p.len_cap) {
            if (blockIdx.x == 0)
                atomicOr(p.err, PKV_EBIT_SEQLEN);
            L = 0;
        }
        s_len[b] = L;
        int lo = (p.window > 0 && L > p.window) ? L - p.window : 0;
        if (p.seq_prefix) {
            // the rows after the shared prefix (none if the prefix is all)
            lo = __ldg(p.seq_prefix + b);
            if (lo < 0 || lo > L) {
                if (blockIdx.x == 0)
                    atomicOr(p.err, PKV_EBIT_SEQLEN);
                lo = 0;
            }
        }
        s_lo[b] = lo;
    }
    __syncthreads();
    // Tiles of sequence b: from the one holding its first attended row to the
    // one holding its last (none when no row is left to attend).
    auto seq_tiles = [&](int b) {
        return s_len[b] > s_lo[b] ? (s_len[b] + C::TT - 1) / C::TT - s_lo[b] / C::TT : 0;
    };
    // One pass over the sequences (thread t takes a contiguous run, then
    // warp and block scans): the exclusive prefixes of tiles (s_tstart) and
    // of cost (s_cstart), where each (sequence, KV head) segment costs PC
    // units for its piece end, then one per tile; and this CTA's tiles.
    //
    // The cost is split evenly over P = min(grid, cost) CTAs; a CTA owns
    // the tiles whose cost position (segment start + PC + tile) falls in
    // its share.  The CTAs holding pieces of one sequence/head are
    // consecutive, and each CTA between the owners of a segment's first and
    // last tile owns a tile of it (tile positions are consecutive there), as
    // the merge counts on.
    constexpr int PC = piece_cost(G, C::SUB);
    constexpr int NW = NTHREADS / 32;
    static_assert(NW <= 12, "scan scratch: misc[8, 32)");
    int *s_range = reinterpret_cast<int *>(smem + lay.merge);   // free until the first merge
    {
        const int per = (B + NTHREADS - 1) / NTHREADS;
        const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
        int st = 0, sc = 0;
        for (int b = b0; b < b1; ++b) {
            const int nt = seq_tiles(b);
            st += nt * Hkv;
            sc += nt > 0 ? (nt + PC) * Hkv : 0;
        }
        int it = st, ic = sc;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(FULL_MASK, it, off);
            const int z = __shfl_up_sync(FULL_MASK, ic, off);
            if (lane >= off) {
                it += y;
                ic += z;
            }
        }
        int *wsum = misc + 8;            // [8, 8 + NW) tiles, [20, 20 + NW) cost
        if (lane == 31) {
            wsum[warp] = it;
            wsum[12 + warp] = ic;
        }
        __syncthreads();
        if (warp == 0) {
            int v = lane < NW ? wsum[lane] : 0;
            int u = lane < NW ? wsum[12 + lane] : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(FULL_MASK, v, off);
                const int z = __shfl_up_sync(FULL_MASK, u, off);
                if (lane >= off) {
                    v += y;
                    u += z;
                }
            }
            if (lane < NW) {
                wsum[lane] = v;
                wsum[12 + lane] = u;
            }
        }
        __syncthreads();
        int bt = (warp > 0 ? wsum[warp - 1] : 0) + it - st;
        int bc = (warp > 0 ? wsum[12 + warp - 1] : 0) + ic - sc;
        const int t_all = wsum[NW - 1], c_all = wsum[12 + NW - 1];
        const int p_all = (int)min((int64_t)gridDim.x, (int64_t)c_all);
        // the cost positions where this CTA's share begins and ends
        const int64_t cb[2] = {
            blockIdx.x < p_all ? (int64_t)blockIdx.x * c_all / p_all : c_all,
            blockIdx.x < p_all ? (int64_t)(blockIdx.x + 1) * c_all / p_all : c_all};
        for (int b = b0; b < b1; ++b) {
            const int nt = seq_tiles(b);
            const int cost = nt > 0 ? (nt + PC) * Hkv : 0;
            s_tstart[b] = bt;
            s_cstart[b] = bc;
            // a share boundary inside this sequence's cost -> tiles below it
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                if (cb[e] >= bc && cb[e] < bc + cost) {
                    const int rem = (int)(cb[e] - bc);
                    const int kvh = rem / (nt + PC);
                    const int in = rem - kvh * (nt + PC) - PC;
                    s_range[e] = bt + kvh * nt + (in < 0 ? 0 : (in > nt ? nt : in));
                }
            }
            bt += nt * Hkv;
            bc += cost;
        }
        if (tid == 0) {
            s_tstart[B] = t_all;
            s_cstart[B] = c_all;
            if (cb[0] >= c_all)
                s_range[0] = t_all;
            if (cb[1] >= c_all)
                s_range[1] = t_all;
        }
        __syncthreads();
    }
    const int64_t CT = s_cstart[B];
    const int P = (int)min((int64_t)gridDim.x, CT);
    const int cta = blockIdx.x;
    // cost position of tile i of segment (b, kvh)
    auto tile_cost = [&](int b, int kvh, int i) -> int64_t {
        return (int64_t)s_cstart[b] + (int64_t)kvh * (seq_tiles(b) + PC) + PC + i;
    };
    const int64_t R0 = s_range[0];
    const int64_t R1 = s_range[1];
    const int Hq = p.num_q_heads;

    if (warp == W) {
        // ================= producer warp =================
        // The warp issues tiles in groups of GRP = min(32, stages): lane j
        // copies tile k0 + j into its own stage, so the lanes of a group wait
        // for their stages and issue their copies in parallel (a stage is free
        // again only after its tile of an earlier group was consumed).  The
        // next group's block ids are fetched while this group is issued.
        const int n_local = (int)(R1 - R0);
        const int bs = p.block_size;
        const int GRP = min(32, p.nst);
        const uint64_t policy = policy_evict_first();
        // (with units of several tiles, id[] holds the unit's rows in the
        // gather view of the caches, and nblk the rows holding tokens)
        struct Desc { int b, kvh, ti, nblk; int32_t id[C::NIDS]; };
        // Tile -> (sequence, KV head, tile of the sequence) for the group's
        // consecutive tiles at once.  bh is a sequence at or before the
        // group's first tile; lane j holds the j-th sequence boundary after
        // it, and each lane counts the boundaries at or below its tile by a
        // search over the lanes (shuffles, rather than a binary search whose
        // every step waits on a shared-memory load).  More than 31
        // boundaries in reach (runs of empty sequences) fall back to the
        // binary search.
        auto describe = [&](int k0, int bh) {
            Desc d;
            d.b = d.kvh = d.ti = d.nblk = 0;
#pragma unroll
            for (int i = 0; i < C::NIDS; ++i)
                d.id[i] = -1;
            const int x = (int)(R0 + k0) + lane;
            const int jb = bh + 1 + lane;
            const int tj = jb <= B ? s_tstart[jb] : INT_MAX;
            const int t_bh = s_tstart[bh];
            int pos = 0;
#pragma unroll
            for (int step = 16; step >= 1; step >>= 1) {
                const int t = __shfl_sync(FULL_MASK, tj, pos + step - 1);
                if (t <= x)
                    pos += step;
            }
            const int t_hi = __shfl_sync(FULL_MASK, tj, pos);
            const int t_lo = __shfl_sync(FULL_MASK, tj, pos > 0 ? pos - 1 : 0);
            const bool over = __shfl_sync(FULL_MASK, tj, 31) <= x;
            if (lane < GRP && k0 + lane < n_local) {
                int tb, tb1;
                if (!over) {
                    d.b = bh + pos;
                    tb = pos > 0 ? t_lo : t_bh;
                    tb1 = t_hi;
                } else {
                    d.b = find_seq(s_tstart, B, x);
                    tb = s_tstart[d.b];
                    tb1 = s_tstart[d.b + 1];
                }
                const int nt = (tb1 - tb) / Hkv;
                const int off = x - tb;
                d.kvh = off / nt;
                d.ti = off - d.kvh * nt + s_lo[d.b] / C::TT;
                const int nvalid = min(C::TT, s_len[d.b] - C::TT * d.ti);
                const int32_t *row = p.block_tables + (int64_t)d.b * p.max_blocks_per_seq;
                if constexpr (C::SUB > 1) {
                    // rows of rt tokens; rows before the first attended
                    // token (a window's or a suffix's start) and past the
                    // last token repeat the nearest row with attended tokens,
                    // so that no other block is looked up; a block id out of
                    // range gives -1 (read as row 0, the error word set)
                    const int rt = gather_row_tokens(bs, C::TT);
                    const int nr = C::TT / rt;
                    d.nblk = (nvalid + rt - 1) / rt;
                    const int lead = s_lo[d.b] - C::TT * d.ti;
                    const int r_lo = lead > 0 ? lead / rt : 0;
#pragma unroll
                    for (int r = 0; r < C::NIDS; ++r) {
                        if (r < nr) {
                            const int rr = r < r_lo ? r_lo : (r < d.nblk ? r : d.nblk - 1);
                            const int tok = C::TT * d.ti + rr * rt;
                            const int blk = __ldg(row + (tok >> p.bs_log2));
                            d.id[r] = (blk >= 0 && blk < p.num_blocks)
                                          ? (blk * Hkv + d.kvh) * (bs / rt) + (tok & (bs - 1)) / rt
                                          : -1;
                        }
                    }
                } else {
                    const int first = (TILE * d.ti) >> p.bs_log2;
                    d.nblk = bs >= TILE ? 1 : (nvalid + bs - 1) >> p.bs_log2;   // 1..4 (bs >= 4)
                    d.id[0] = __ldg(row + first);
                    if (d.nblk > 1) d.id[1] = __ldg(row + first + 1);
                    if (d.nblk > 2) d.id[2] = __ldg(row + first + 2);
                    if (d.nblk > 3) d.id[3] = __ldg(row + first + 3);
                }
            }
            return d;
        };
        long long seg_last = -1;                // (sequence, KV head) of the previous tile
        int qn_base = 0;                        // q copies issued before this group
        int st_base = 0, rnd_base = 0;          // stage and ring round of tile k0
        Desc cur = describe(0, n_local > 0 ? find_seq(s_tstart, B, R0) : 0);
        for (int k0 = 0; k0 < n_local; k0 += GRP) {
            const int n = min(GRP, n_local - k0);
            const Desc nxt = describe(k0 + GRP, __shfl_sync(FULL_MASK, cur.b, n - 1));
            const bool active = lane < n;
            const long long seg = active ? (long long)cur.b * Hkv + cur.kvh : -1;
            long long prev = __shfl_up_sync(FULL_MASK, seg, 1);
            if (lane == 0)
                prev = seg_last;
            const bool starts = active && seg != prev;      // first tile of a piece
            const unsigned start_mask = __ballot_sync(FULL_MASK, starts);
            const int qn = qn_base + __popc(start_mask & ((1u << lane) - 1u));
            int st = st_base + lane, rnd = rnd_base;
            if (st >= p.nst) {
                st -= p.nst;
                ++rnd;
            }
            {
                // One convergent polling loop: each round every lane tests,
                // without blocking, its q slot (if its tile starts a piece) and
                // its stage, and issues the copies as soon as they are free; the
                // warp leaves when all lanes are done.  (A blocking wait in a
                // divergent lane would hold up lanes whose stages are already
                // free.)  q copies leave in piece order: the q ring has two slots
                // and a parity test only tells one phase from the next, so copy
                // qn may test its slot only after copy qn - 1 has gone.
                volatile int *qcount = misc + MISC_QCOUNT;
                const int slot = qn & 1;
                bool q_done = !starts;
                bool t_done = !active;
                uint64_t t0 = 0;
                for (uint32_t it = 0;; ++it) {
                    if (!q_done && *qcount == qn &&
                        mbar_test_wait(&qempty[slot], ((qn >> 1) & 1) ^ 1)) {
                        const uint32_t qbytes = (uint32_t)(G * D * p.q_bytes);
                        mbar_arrive_expect_tx(&qfull[slot], qbytes);
                        const unsigned char *qsrc = static_cast<const unsigned char *>(p.q) +
                                                    ((int64_t)cur.b * Hq + cur.kvh * G) * D * p.q_bytes;
                        bulk_g2s(qring + slot * C::QSLOT, qsrc, qbytes, &qfull[slot]);
                        atomicMax(&misc[MISC_QISSUED + slot], (qn >> 1) + 1);
                        __threadfence_block();
                        *qcount = qn + 1;
                        q_done = true;
                    }
                    // Staggered start: the first group's tiles beyond the first W
                    // (one per consumer warp) go out once tile 0 has landed, so
                    // the first tiles are not queued behind the whole ring's
                    // burst and the consumers start earlier.
                    const bool hold = k0 == 0 && lane >= W && !mbar_test_wait(&full[0], 0u);
                    if (!t_done && !hold && mbar_test_wait(&empty[st], (uint32_t)(rnd & 1) ^ 1u)) {
                    unsigned char *sK = stages + st * C::STAGE_BYTES;
                    unsigned char *sV = sK + C::KV_BYTES;
                    unsigned char *sKS = scale_ring + st * 2 * C::SC_BYTES;
                    unsigned char *sVS = sKS + C::SC_BYTES;
                    if constexpr (C::SUB > 1) {
                    // A unit: its rows of rt tokens gathered four at a time
                    // from the 2-D views of the caches (rows of rt * ROWB
                    // bytes), the scales of the rows with tokens by cp.async.
                    const int rt = gather_row_tokens(bs, C::TT);
                    const int nr = C::TT / rt;
                    bool bad = false;
#pragma unroll
                    for (int r = 0; r < C::NIDS; ++r)
                        bad |= r < nr && cur.id[r] < 0;
                    if (bad)
                        atomicOr(p.err, PKV_EBIT_BLOCK);
                    mbar_arrive_expect_tx(&full[st], (uint32_t)(2 * C::KV_BYTES));
                    reinterpret_cast<volatile int *>(misc)[MISC_ISSUED + st] = rnd + 1;
                    const int rb = rt * C::ROWB;
#pragma unroll
                    for (int g4 = 0; g4 < C::NIDS / 4; ++g4) {
                        if (4 * g4 < nr) {
                            const int r0 = max(cur.id[4 * g4], 0), r1 = max(cur.id[4 * g4 + 1], 0);
                            const int r2 = max(cur.id[4 * g4 + 2], 0), r3 = max(cur.id[4 * g4 + 3], 0);
                            tma_gather4(sK + 4 * g4 * rb, &p.tm_k, r0, r1, r2, r3, &full[st],
                                        policy);
                            tma_gather4(sV + 4 * g4 * rb, &p.tm_v, r0, r1, r2, r3, &full[st],
                                        policy);
                        }
                    }
                    if constexpr (quantized(KV)) {
#pragma unroll
                        for (int r = 0; r < C::NIDS; ++r) {
                            if (r < cur.nblk && cur.id[r] >= 0) {
                                // scales of row r: rt halves at element id * rt
                                const unsigned char *ksrc = reinterpret_cast<const unsigned char *>(
                                    p.k_scales + (int64_t)cur.id[r] * rt);
                                const unsigned char *vsrc = reinterpret_cast<const unsigned char *>(
                                    p.v_scales + (int64_t)cur.id[r] * rt);
                                for (int o = 0; o < rt * 2; o += 16) {
                                    cp_async_16b(sKS + r * rt * 2 + o, ksrc + o);
                                    cp_async_16b(sVS + r * rt * 2 + o, vsrc + o);
                                }
                            }
                        }
                        cp_async_mbar_arrive(&full[st]);
                    }
                    } else {
                    const int rows_per_copy = bs >= TILE ? TILE : bs;
                    const uint32_t kv_copy = (uint32_t)(rows_per_copy * C::ROWB);
                    const int sc_copy = rows_per_copy * 2;
                    // Count the bytes of the bulk copies that will be issued.
                    uint32_t total = 0;
                    bool bad = false;
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        if (u < cur.nblk) {
                            if (cur.id[u] >= 0 && cur.id[u] < p.num_blocks)
                                total += 2 * kv_copy;
                            else
                                bad = true;
                        }
                    }
                    if (bad)
                        atomicOr(p.err, PKV_EBIT_BLOCK);
                    mbar_arrive_expect_tx(&full[st], total);
                    // Tell the consumers that this round of the stage is armed.
                    reinterpret_cast<volatile int *>(misc)[MISC_ISSUED + st] = rnd + 1;
                    const int in_block = (TILE * cur.ti) & (bs - 1);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        if (u < cur.nblk && cur.id[u] >= 0 && cur.id[u] < p.num_blocks) {
                            const int64_t row0 = ((int64_t)cur.id[u] * Hkv + cur.kvh) * bs +
                                                 (bs >= TILE ? in_block : 0);
                            const int dst_row = u * rows_per_copy;
                            if constexpr (C::SWIZZLE_OK) {
                                if (swz) {
                                    // 16 rows of the (block, head) as one
                                    // swizzled tensor copy each
                                    const int z = cur.id[u] * Hkv + cur.kvh;
                                    tma_tile_swz<C::ROWB>(sK, &p.tm_k, in_block, z, &full[st],
                                                          policy);
                                    tma_tile_swz<C::ROWB>(sV, &p.tm_v, in_block, z, &full[st],
                                                          policy);
                                } else {
                                    bulk_g2s_hint(sK + dst_row * C::ROWB,
                                                  p.k_cache + row0 * C::ROWB, kv_copy, &full[st],
                                                  policy);
                                    bulk_g2s_hint(sV + dst_row * C::ROWB,
                                                  p.v_cache + row0 * C::ROWB, kv_copy, &full[st],
                                                  policy);
                                }
                            } else {
                                bulk_g2s_hint(sK + dst_row * C::ROWB, p.k_cache + row0 * C::ROWB,
                                              kv_copy, &full[st], policy);
                                bulk_g2s_hint(sV + dst_row * C::ROWB, p.v_cache + row0 * C::ROWB,
                                              kv_copy, &full[st], policy);
                            }
                            if constexpr (quantized(KV)) {
                                // The scales (32 bytes of each array per 16
                                // rows) go by 16-byte (8-byte for 4-row
                                // blocks) cp.async copies: as two more bulk
                                // copies they would double the tile's copy
                                // count, and small tiles are bound by the
                                // bulk-copy unit's rate per copy, not bytes.
                                const unsigned char *ksrc =
                                    reinterpret_cast<const unsigned char *>(p.k_scales + row0);
                                const unsigned char *vsrc =
                                    reinterpret_cast<const unsigned char *>(p.v_scales + row0);
                                if (sc_copy >= 16) {
                                    for (int o = 0; o < sc_copy; o += 16) {
                                        cp_async_16b(sKS + dst_row * 2 + o, ksrc + o);
                                        cp_async_16b(sVS + dst_row * 2 + o, vsrc + o);
                                    }
                                } else {
                                    cp_async_8b(sKS + dst_row * 2, ksrc);
                                    cp_async_8b(sVS + dst_row * 2, vsrc);
                                }
                            }
                        }
                    }
                    if constexpr (quantized(KV))
                        cp_async_mbar_arrive(&full[st]);
                    }
                        t_done = true;
                    }
                    if (__all_sync(FULL_MASK, q_done && t_done))
                        break;
                    if ((it & 63u) == 63u) {
                        // bounded: give up after WAIT_LIMIT_NS (decided by lane 0
                        // so that the whole warp leaves together)
                        int stop = 0;
                        if (lane == 0) {
                            const uint64_t now = globaltimer_ns();
                            if (it == 63u)
                                t0 = now;
                            else if (now - t0 > WAIT_LIMIT_NS || *abort_flag)
                                stop = 1;
                        }
                        if (__shfl_sync(FULL_MASK, stop, 0)) {
                            if (lane == 0 && !*abort_flag) {
                                *abort_flag = 1;
                                atomicOr(p.err, PKV_EBIT_TIMEOUT);
                            }
                            break;
                        }
                    }
                }
            }
            __syncwarp();
            seg_last = __shfl_sync(FULL_MASK, seg, n - 1);
            qn_base += __popc(start_mask);
            st_base += n;
            if (st_base >= p.nst) {
                st_base -= p.nst;
                ++rnd_base;
            }
            cur = nxt;
        }
    } else {
        // ================= consumer warps =================
        const int w = warp;
        const int ds = lane % C::DS;
        const int tq = lane / C::DS;
        const int ctid = tid;                  // 0 .. W*32-1
        float *ps = psbuf + w * C::PSW;
        float *mw = merge + w * G * (D + 2);

        // Fold the shared-prefix partial of (sequence b, query head h,
        // element d) into (m, num, den) (the prefix pass merged its chunks).
        auto fold_prefix = [&](int b, int h, int d, float &m, float &num, float &den) {
            if (p.seq_prefix == nullptr || s_lo[b] == 0)
                return;
            const float *row = p.prefix_part + ((int64_t)b * Hq + h) * (D + 4);
            const float mp = __ldcg(row + D + 2), lp = __ldcg(row + D + 3), op = __ldcg(row + d);
            const float mn = fmaxf(m, mp);
            const float fo = exp2_approx(m - mn), fp = exp2_approx(mp - mn);
            num = fmaf(num, fo, op * fp);
            den = fmaf(den, fo, lp * fp);
            m = mn;
        };
        // The same from the piece's prefix rows staged in shared memory.
        auto fold_prefix_staged = [&](int b, int g, int d, float &m, float &num, float &den) {
            if (p.seq_prefix == nullptr || s_lo[b] == 0)
                return;
            const float *row = s_pre + g * (D + 4);
            const float mp = row[D + 2], lp = row[D + 3], op = row[d];
            const float mn = fmaxf(m, mp);
            const float fo = exp2_approx(m - mn), fp = exp2_approx(mp - mn);
            num = fmaf(num, fo, op * fp);
            den = fmaf(den, fo, lp * fp);
            m = mn;
        };
        // Rows of sequences with no tile here: zeros for empty sequences, the
        // prefix alone for a sequence whose rows are all shared; sequence b
        // is CTA (b % grid)'s job.
        for (int b = cta; b < B; b += gridDim.x) {
            if (seq_tiles(b) == 0)
                for (int idx = ctid; idx < Hq * D; idx += W * 32) {
                    float m = -INFINITY, num = 0.0f, den = 0.0f;
                    fold_prefix(b, idx / D, idx % D, m, num, den);
                    p.out[(int64_t)b * Hq * D + idx] = den > 0.0f ? num / den : 0.0f;
                }
        }

        const int stride = G * (D + 2);   // floats of one partial
        // The CTAs that own the first and last tile of a (sequence, KV
        // head).
        struct SegSpan { int c_first, c_last; };
        auto seg_span = [&](int seg) {
            const int bq = seg / Hkv, kq = seg - (seg / Hkv) * Hkv;
            const int nt = seq_tiles(bq);
            return SegSpan{owner_of(tile_cost(bq, kq, 0), CT, P),
                           owner_of(tile_cost(bq, kq, nt - 1), CT, P)};
        };
        // Merge the partials of CTAs c0..c1 of piece `seg`, in CTA order, for
        // output idx; CTA `own` (if any) contributes (own_m, own_num, own_den)
        // from registers instead of its stored partial.  The order, and so the
        // rounding, is the same whichever CTA merges.
        auto fold_partials = [&](int seg, int c0, int c1, int own, float own_m, float own_num,
                                 float own_den, int idx, float &m, float &num, float &den) {
            const int g = idx / D;
            const float *base = p.partials + (int64_t)seg * stride;
            m = -INFINITY;
            num = 0.0f;
            den = 0.0f;
#pragma unroll 4
            for (int pc = c0; pc <= c1; ++pc) {
                const float *part = base + (int64_t)pc * stride;
                const bool mine = pc == own;
                const float mp = mine ? own_m : __ldcg(part + G * D + g);
                const float np = mine ? own_num : __ldcg(part + idx);
                const float lp = mine ? own_den : __ldcg(part + G * D + G + g);
                const float mn = fmaxf(m, mp);
                const float fo = exp2_approx(m - mn), fp = exp2_approx(mp - mn);
                num = fmaf(num, fo, np * fp);
                den = fmaf(den, fo, lp * fp);
                m = mn;
            }
        };
        // Merge every partial of piece `seg` (this CTA was the last to
        // publish one) and write the output rows; reset the piece's counter.
        auto final_merge = [&](int seg) {
            const SegSpan sp = seg_span(seg);
            const int bq = seg / Hkv, kq = seg - (seg / Hkv) * Hkv;
            for (int idx = ctid; idx < G * D; idx += W * 32) {
                float m, num, den;
                fold_partials(seg, sp.c_first, sp.c_last, -1, 0.0f, 0.0f, 0.0f, idx, m, num, den);
                fold_prefix(bq, kq * G + idx / D, idx % D, m, num, den);
                p.out[((int64_t)bq * Hq + kq * G) * D + idx] = num / den;
            }
            if (ctid == 0)
                p.counters[seg] = 0;
        };
        int qn = 0;
        int64_t x = R0;
        while (x < R1) {
            const int b = find_seq(s_tstart, B, x);
            const int nt = (s_tstart[b + 1] - s_tstart[b]) / Hkv;
            const int off = (int)(x - s_tstart[b]);
            const int kvh = off / nt;
            const int ti0 = off - kvh * nt + s_lo[b] / C::TT;   // unit index in the sequence
            const int64_t seg_begin = (int64_t)s_tstart[b] + (int64_t)kvh * nt;
            const int64_t seg_end = seg_begin + nt;
            const int64_t xe = min(seg_end, R1);
            const int k0 = (int)(x - R0);
            const int k1 = (int)(xe - R0);
            const int L = s_len[b];
            const int lo = s_lo[b];

            // q of this (sequence, KV head) group.
            QRegs<D, G, KV> qr;             // CUDA-core tile math
            MmaState<D, G, KV, QS> mst;     // tensor-core tile math
            {
                const int slot = qn & 1;
                if (!mbar_wait_bounded(&qfull[slot], (qn >> 1) & 1, abort_flag) && !*abort_flag) {
                    *abort_flag = 1;
                    atomicOr(p.err, PKV_EBIT_TIMEOUT);
                }
                if constexpr (C::MMA)
                    load_q_mma<D, G, KV, QS>(mst, qring + slot * C::QSLOT, p.q_dtype, lane);
                else
                    load_q<D, G, KV>(qr, qring + slot * C::QSLOT, ds, p.q_dtype);
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&qempty[slot]);
                ++qn;
            }
            if (p.seq_prefix != nullptr && s_lo[b] > 0) {
                // the merged prefix rows of this piece's G heads, fetched now
                // for its end (a load there would wait behind the streaming)
                const float *src = p.prefix_part + ((int64_t)b * Hq + kvh * G) * (D + 4);
                for (int i = ctid; i < G * (D + 4) / 4; i += W * 32)
                    cp_async_16b(s_pre + 4 * i, src + 4 * i);
                asm volatile("cp.async.commit_group;" ::: "memory");
            }

            float m_run[C::NF], l_run[C::NF];
            float acc[G][C::VE];
#pragma unroll
            for (int r = 0; r < C::NF; ++r) {
                m_run[r] = -INFINITY;
                l_run[r] = 0.0f;
            }
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int e = 0; e < C::VE; ++e)
                    acc[g][e] = 0.0f;
            if constexpr (C::MMA) {
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    mst.m[r] = -INFINITY;
                    mst.l[r] = 0.0f;
                }
#pragma unroll
                for (int j = 0; j < D / 16; ++j)
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        mst.acc[j][u] = 0.0f;
            }

            const int kfirst = k0 + (w - k0 % W + W) % W;
            // tile k sits in ring stage st = k mod nst, round rnd = k / nst
            // (stepped along with k rather than divided out per tile)
            int rnd = kfirst / p.nst;
            int st = kfirst - rnd * p.nst;
            for (int k = kfirst; k < k1; k += W, st += W) {
                while (st >= p.nst) {
                    st -= p.nst;
                    ++rnd;
                }
                const int ti = ti0 + (k - k0);
                const int nvalid = min(C::TT, L - C::TT * ti);
                const int tlo = lo - C::TT * ti;         // > 0 only in the window's first unit
                // Warps take tiles round-robin and may drift apart, so this
                // warp can reach tile k while the stage's previous tile
                // (k - stages) is still landing; a parity wait alone would
                // mistake that phase for an older completed one.  So first
                // wait until the producer has armed this round of the stage
                // (it records the round after arming the barrier), then the
                // parity wait is unambiguous.
                const bool armed =
                    count_wait_bounded(misc + MISC_ISSUED + st, rnd + 1, abort_flag);
                if (!(armed && mbar_wait_bounded(&full[st], (uint32_t)rnd & 1u, abort_flag)) &&
                    !*abort_flag) {
                    *abort_flag = 1;
                    atomicOr(p.err, PKV_EBIT_TIMEOUT);
                }
                const unsigned char *sK = stages + st * C::STAGE_BYTES;
                const unsigned char *sV = sK + C::KV_BYTES;
                const __half *sKS =
                    reinterpret_cast<const __half *>(scale_ring + st * 2 * C::SC_BYTES);
                const __half *sVS = sKS + C::TT;
                if constexpr (C::MMA && C::SUB > 1) {
                    // the unit's 16-token tiles that hold attended tokens:
                    // 2-tile units scored together, 4-tile units tile by
                    // tile (the last one hands the stage back)
                    if constexpr (C::SUB == 2) {
                        mma_unit<D, G, KV, QS, C::SUB>(mst, sK, sV, sKS, sVS, nvalid, tlo,
                                                       p.scale_log2, lane, &empty[st]);
                    } else {
                        const int i0 = tlo > 0 ? tlo / TILE : 0;
                        const int i1 = (nvalid + TILE - 1) / TILE;
#pragma unroll 1
                        for (int i = i0; i < i1; ++i)
                            mma_tile<D, G, KV, QS>(mst, sK + i * C::KV_BYTES / C::SUB,
                                                   sV + i * C::KV_BYTES / C::SUB, sKS + i * TILE,
                                                   sVS + i * TILE, min(TILE, nvalid - i * TILE),
                                                   tlo - i * TILE, p.scale_log2, lane,
                                                   &empty[st], 0, i == i1 - 1);
                    }
                } else if constexpr (C::MMA) {
                    mma_tile<D, G, KV, QS>(mst, sK, sV, sKS, sVS, nvalid, tlo, p.scale_log2,
                                           lane, &empty[st], swz);
                } else {
                    // one 16-token tile on the CUDA cores; `release` hands the
                    // stage back after it
                    auto cc_tile = [&](const unsigned char *sK, const unsigned char *sV,
                                       const __half *sKS, const __half *sVS, int nvalid, int tlo,
                                       bool release) {
                        // After the reduction below the lane holds token t, heads g0 + r.
                        const int t = tq + C::TQ * (ds >> 1);
                        const int g0 = G >= 2 ? (G / 2) * (ds & 1) : 0;

                        // ---- take this lane's part of the tile into registers and hand
                        // the stage back at once, so that the next copy into it starts
                        // while this warp computes
                        uint4 kr[C::TPL][C::CPL];
                        load_k<D, G, KV>(kr, sK, tq, ds);
                        float ks_t = 1.0f, vs_t = 1.0f;
                        if constexpr (quantized(KV)) {
                            ks_t = __half2float(sKS[t]);
                            vs_t = __half2float(sVS[t]);
                        }
                        // (with G = 8 the heads' accumulators need the registers; V is
                        // then read from the stage, which is released after P.V)
                        constexpr bool VREG = VRaw<D, KV>::IN_REGS && G <= 4;
                        typename VRaw<D, KV>::type vr[TILE];
                        if constexpr (VREG) {
        #pragma unroll
                            for (int tt = 0; tt < TILE; ++tt)
                                vr[tt] = load_v_raw<D, KV>(sV, tt, lane);
                            if (release) {
                                __syncwarp();
                                if (lane == 0)
                                    mbar_arrive(&empty[st]);
                            }
                        }

                        // ---- scores: partial dots, then reduce-scatter over the DS lanes
                        float part[C::NP];
        #pragma unroll
                        for (int j = 0; j < C::NP; ++j)
                            part[j] = 0.0f;
                        qk_tile<D, G, KV>(part, qr, kr);
                        reduce_scatter<C::NP, C::DS / 2>(part, ds);
                        float s[C::NF];
                        float kscale = p.scale_log2;
                        if constexpr (quantized(KV))
                            kscale *= ks_t;
                        bool above = false;
        #pragma unroll
                        for (int r = 0; r < C::NF; ++r) {
                            s[r] = (t < nvalid && t >= tlo) ? part[r] * kscale : -INFINITY;
                            above |= s[r] > m_run[r];
                        }
                        // The running maximum only needs to move when some score
                        // exceeds it (softmax is shift invariant, so any running value
                        // that is one of the scores seen is exact); most tiles skip
                        // the per-head maximum and the rescale.
                        const bool moved = __any_sync(FULL_MASK, above);
                        float corr[C::NF];
                        if (moved) {
        #pragma unroll
                            for (int r = 0; r < C::NF; ++r) {
                                float mx = s[r];
        #pragma unroll
                                for (int mask = 2; mask < 32; mask <<= 1)
                                    mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, mask));
                                const float mnew = fmaxf(m_run[r], mx);   // finite: a valid token
                                corr[r] = exp2_approx(m_run[r] - mnew);
                                l_run[r] *= corr[r];
                                m_run[r] = mnew;
                            }
                        }
                        float pr[C::NF];
        #pragma unroll
                        for (int r = 0; r < C::NF; ++r) {
                            pr[r] = exp2_approx(s[r] - m_run[r]);
                            l_run[r] += pr[r];
                        }
                        // Publish {p, p} pairs (p times the V scale for int8) and, when
                        // the maximum moved, the rescale factors.
                        if (G >= 2 || (ds & 1) == 0) {
                            const float vsc = vs_t;
                            float2 *pp = reinterpret_cast<float2 *>(ps + t * 2 * G) + g0;
        #pragma unroll
                            for (int r = 0; r < C::NF; ++r) {
                                const float v = pr[r] * vsc;
                                pp[r] = make_float2(v, v);
                            }
                            if (moved && tq == 0 && (ds >> 1) == 0) {
        #pragma unroll
                                for (int r = 0; r < C::NF; ++r)
                                    ps[TILE * 2 * G + g0 + r] = corr[r];
                            }
                        }
                        __syncwarp();

                        // ---- weighted V
                        if (moved) {
        #pragma unroll
                            for (int g = 0; g < G; ++g) {
                                const float cg = ps[TILE * 2 * G + g];
        #pragma unroll
                                for (int e = 0; e < C::VE; ++e)
                                    acc[g][e] *= cg;
                            }
                        }
                        auto pv_token = [&](int tt) {
                            float v[C::VE];
                            if constexpr (VREG)
                                unpack_v<D, KV>(v, vr[tt]);
                            else
                                load_v<D, KV>(v, sV, tt, lane);
                            const float *pt = ps + tt * 2 * G;
                            if constexpr (G == 1) {
                                const float2 w2 = *reinterpret_cast<const float2 *>(pt);
        #pragma unroll
                                for (int e = 0; e < C::VE; e += 2)
                                    fma2(acc[0][e], acc[0][e + 1], w2.x, w2.y, v[e], v[e + 1]);
                            } else {
        #pragma unroll
                                for (int g = 0; g < G; g += 2) {
                                    const float4 w4 = *reinterpret_cast<const float4 *>(pt + 2 * g);
        #pragma unroll
                                    for (int e = 0; e < C::VE; e += 2) {
                                        fma2(acc[g][e], acc[g][e + 1], w4.x, w4.y, v[e], v[e + 1]);
                                        fma2(acc[g + 1][e], acc[g + 1][e + 1], w4.z, w4.w, v[e], v[e + 1]);
                                    }
                                }
                            }
                        };
                        if (nvalid == TILE) {
        #pragma unroll
                            for (int tt = 0; tt < TILE; ++tt)
                                pv_token(tt);
                        } else {
        #pragma unroll
                            for (int tt = 0; tt < TILE; ++tt)
                                if (tt < nvalid)
                                    pv_token(tt);
                        }
                        if constexpr (!VREG) {
                            if (release) {
                                __syncwarp();
                                if (lane == 0)
                                    mbar_arrive(&empty[st]);
                            }
                        }
                    };
                    if constexpr (C::SUB > 1) {
                        // the unit's tiles that hold attended tokens, in order
                        const int i0 = tlo > 0 ? tlo / TILE : 0;
                        const int i1 = (nvalid + TILE - 1) / TILE;
#pragma unroll 1
                        for (int i = i0; i < i1; ++i)
                            cc_tile(sK + i * C::KV_BYTES / C::SUB, sV + i * C::KV_BYTES / C::SUB,
                                    sKS + i * TILE, sVS + i * TILE, min(TILE, nvalid - i * TILE),
                                    tlo - i * TILE, i == i1 - 1);
                    } else {
                        cc_tile(sK, sV, sKS, sVS, nvalid, tlo, true);
                    }
                }
            }

            // ---- merge the W warp states of this piece
            asm volatile("cp.async.wait_all;" ::: "memory");   // this piece's prefix rows
            if constexpr (C::MMA) {
                // lane (gid, tig) holds heads 2tig, 2tig+1 x elements
                // [gid D/8, (gid+1) D/8); l sums over the lane's tokens
                const int gid = lane >> 2, tig = lane & 3;
#pragma unroll
                for (int r = 0; r < 2; ++r)
#pragma unroll
                    for (int mask = 4; mask < 32; mask <<= 1)
                        mst.l[r] += __shfl_xor_sync(FULL_MASK, mst.l[r], mask);
                if constexpr (G < 8) {
                    // columns 2tig + G, +1 (lane + G/2) hold the low-part
                    // sums of the lane's heads
#pragma unroll
                    for (int j = 0; j < D / 16; ++j)
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            mst.acc[j][u] += __shfl_down_sync(FULL_MASK, mst.acc[j][u], G / 2);
                }
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int h = 2 * tig + r;
                    if (h < G) {
#pragma unroll
                        for (int j = 0; j < D / 16; ++j)
                            *reinterpret_cast<float2 *>(mw + h * D + gid * (D / 8) + 2 * j) =
                                make_float2(mst.acc[j][r], mst.acc[j][r + 2]);
                        if (gid == 0) {
                            mw[G * D + h] = mst.m[r];
                            mw[G * D + G + h] = mst.l[r];
                        }
                    }
                }
            } else {
    #pragma unroll
                for (int r = 0; r < C::NF; ++r)
    #pragma unroll
                    for (int mask = 2; mask < 32; mask <<= 1)
                        l_run[r] += __shfl_xor_sync(FULL_MASK, l_run[r], mask);
    #pragma unroll
                for (int g = 0; g < G; ++g)
    #pragma unroll
                    for (int e = 0; e < C::VE; ++e)
                        mw[g * D + lane * C::VE + e] = acc[g][e];
                if (tq == 0 && (ds >> 1) == 0 && (G >= 2 || ds == 0)) {
                    const int g0 = G >= 2 ? (G / 2) * (ds & 1) : 0;
    #pragma unroll
                    for (int r = 0; r < C::NF; ++r) {
                        mw[G * D + g0 + r] = m_run[r];
                        mw[G * D + G + g0 + r] = l_run[r];
                    }
                }
            }
            named_bar_sync(1, W * 32);

            const int c_first = owner_of(tile_cost(b, kvh, 0), CT, P);
            const int c_last = owner_of(tile_cost(b, kvh, nt - 1), CT, P);
            const bool whole = c_first == c_last;
            const bool last_piece = xe == R1;
            const int seg = b * Hkv + kvh;
            // The CTA's last piece, if split: look (without waiting) whether
            // every other CTA holding a part of it has already published;
            // then this CTA merges at once instead of publishing its own.
            int published = -1;
            if (!whole && last_piece && ctid == 0)
                published = ld_relaxed_gpu(p.counters + seg);
            // Merge the W warp states of each output this thread owns.
            constexpr int MO = (G * D + W * 32 - 1) / (W * 32);
            float o_m[MO], o_num[MO], o_den[MO];
#pragma unroll
            for (int j = 0; j < MO; ++j) {
                const int idx = ctid + j * W * 32;
                o_m[j] = -INFINITY;
                o_num[j] = 0.0f;
                o_den[j] = 0.0f;
                if (idx < G * D) {
                    const int g = idx / D;
                    float M = -INFINITY;
#pragma unroll
                    for (int ww = 0; ww < W; ++ww)
                        M = fmaxf(M, merge[ww * stride + G * D + g]);
                    float num = 0.0f, den = 0.0f;
#pragma unroll
                    for (int ww = 0; ww < W; ++ww) {
                        const float f = exp2_approx(merge[ww * stride + G * D + g] - M);
                        num = fmaf(f, merge[ww * stride + idx], num);
                        den = fmaf(f, merge[ww * stride + G * D + G + g], den);
                    }
                    o_m[j] = M;
                    o_num[j] = num;
                    o_den[j] = den;
                }
            }
            float *orow = p.out + ((int64_t)b * Hq + kvh * G) * D;
            if (whole) {
#pragma unroll
                for (int j = 0; j < MO; ++j) {
                    const int idx = ctid + j * W * 32;
                    if (idx < G * D) {
                        float m = o_m[j], num = o_num[j], den = o_den[j];
                        fold_prefix_staged(b, idx / D, idx % D, m, num, den);
                        orow[idx] = num / den;
                    }
                }
                named_bar_sync(1, W * 32);   // the merge buffer is free again
            } else {
                int merge_now = 0;
                if (last_piece) {
                    if (ctid == 0) {
                        merge_now = published == c_last - c_first;
                        if (merge_now)
                            __threadfence();   // acquire: their partials are visible
                        misc[4] = merge_now;
                    }
                    named_bar_sync(1, W * 32);
                    merge_now = misc[4];
                }
                if (merge_now) {
#pragma unroll
                    for (int j = 0; j < MO; ++j) {
                        const int idx = ctid + j * W * 32;
                        if (idx < G * D) {
                            float m, num, den;
                            fold_partials(seg, c_first, c_last, cta, o_m[j], o_num[j], o_den[j],
                                          idx, m, num, den);
                            fold_prefix_staged(b, idx / D, idx % D, m, num, den);
                            orow[idx] = num / den;
                        }
                    }
                    if (ctid == 0)
                        p.counters[seg] = 0;
                } else {
                    float *part_out = p.partials + (int64_t)(cta + seg) * stride;
#pragma unroll
                    for (int j = 0; j < MO; ++j) {
                        const int idx = ctid + j * W * 32;
                        if (idx < G * D) {
                            part_out[idx] = o_num[j];
                            if ((idx % D) == 0) {
                                part_out[G * D + idx / D] = o_m[j];
                                part_out[G * D + G + idx / D] = o_den[j];
                            }
                        }
                    }
                    // Publish: one thread fences for the CTA after the barrier
                    // (which orders every thread's partial stores before it),
                    // then counts this CTA in.  Mid-stream only that thread's
                    // warp waits for the round trip; a CTA that turns out to
                    // be the last one merges at its end.
                    named_bar_sync(1, W * 32);
                    if (ctid == 0) {
                        __threadfence();
                        const int old = atomicAdd(p.counters + seg, 1);
                        if (old == c_last - c_first) {
                            __threadfence();
                            misc[last_piece ? 5 : 6] = seg + 1;
                        }
                    }
                }
            }
            x = xe;
        }

        // Pieces whose partials this CTA was the last to publish.
        named_bar_sync(1, W * 32);
        if (misc[6])
            final_merge(misc[6] - 1);
        if (misc[5])
            final_merge(misc[5] - 1);
    }

    // Let every copy this CTA issued land before the CTA exits (only matters
    // after a timeout; otherwise the consumers already waited for all of them).
    __syncthreads();
    if (*abort_flag && tid == W * 32) {
        for (int s = 0; s < p.nst; ++s)
            if (misc[MISC_ISSUED + s] > 0)
                mbar_wait_bounded(&full[s], (uint32_t)((misc[MISC_ISSUED + s] - 1) & 1), misc + 2);
        for (int s = 0; s < 2; ++s)
            if (misc[MISC_QISSUED + s] > 0)
                mbar_wait_bounded(&qfull[s], (uint32_t)((misc[MISC_QISSUED + s] - 1) & 1), misc + 2);
    }
}

// ---- host side ---------------------------------------------------------------

template <int D, int G, int KV, bool QS>
int launch_t(const pkv_pool *pool, const Params &base, int batch, int max_seq_len,
             cudaStream_t stream)
{
    using C = Cfg<D, G, KV>;
    Params prm = base;
    // Tiles of the tensor-core tile math come by swizzled tensor copies when
    // a tile is 16 rows of one block (block size >= 16).
    prm.swz = 0;
    if constexpr (C::SUB > 1) {
        // units gather rows of min(bs, 16) tokens from 2-D views of the caches
        const int rt = gather_row_tokens(pool->block_size, C::TT);
        if (!encode_gather_row_map(&prm.tm_k, prm.k_cache, C::ROWB, rt, pool) ||
            !encode_gather_row_map(&prm.tm_v, prm.v_cache, C::ROWB, rt, pool))
            return PKV_ERR_CUDA;
    }
    if constexpr (C::SWIZZLE_OK) {
        if (pool->block_size >= TILE) {
            if (!encode_swizzled_tile_map(&prm.tm_k, prm.k_cache, C::ROWB, pool) ||
                !encode_swizzled_tile_map(&prm.tm_v, prm.v_cache, C::ROWB, pool))
                return PKV_ERR_CUDA;
            prm.swz = 1;
        }
    }
    const Layout fixed = make_layout<D, G, KV>(0, batch, prm.seq_prefix != nullptr);
    const int budget = pool->max_smem_optin - fixed.total - 256;
    // a stage: its K and V tiles, their scales and two barriers
    int nst = budget / (C::STAGE_BYTES + 2 * C::SC_BYTES + 16);
    if (nst > MAX_STAGES)
        nst = MAX_STAGES;
    if (nst < 2)
        return PKV_ERR_UNSUPPORTED;
    prm.nst = nst;
    const Layout lay = make_layout<D, G, KV>(nst, batch, prm.seq_prefix != nullptr);

    // The dynamic shared-memory limit is an attribute of the kernel in the
    // current device's context (a context that a device reset replaces), so
    // it is set on every call rather than remembered by the process.
    if (cudaFuncSetAttribute(paged_decode_kernel<D, G, KV, QS>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, lay.total) != cudaSuccess)
        return PKV_ERR_CUDA;
    const int64_t max_tiles =
        (int64_t)batch * pool->num_kv_heads * ((max_seq_len + C::TT - 1) / C::TT);
    int64_t P = pool->num_sms;
    if (P > max_tiles)
        P = max_tiles;
    if (P < 1)
        P = 1;
    if (launch_pdl(paged_decode_kernel<D, G, KV, QS>, dim3((unsigned)P), dim3(C::NTHREADS),
                   (size_t)lay.total, stream, prm) != cudaSuccess)
        return PKV_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

// The tensor-core tile math multiplies q in the cache's MMA type (bf16 for
// bf16 caches, else fp16); a q of another type goes in as two parts.
template <int D, int G, int KV>
int launch_q(const pkv_pool *pool, const Params &prm, int batch, int max_seq_len,
             cudaStream_t s)
{
    if constexpr (mma_path(KV, G)) {
        const int mma_type = MmaBf16<KV>::v ? PKV_BF16 : PKV_F16;
        if (prm.q_dtype != mma_type)
            return launch_t<D, G, KV, true>(pool, prm, batch, max_seq_len, s);
    }
    return launch_t<D, G, KV, false>(pool, prm, batch, max_seq_len, s);
}

template <int D, int KV>
int launch_g(const pkv_pool *pool, int G, const Params &prm, int batch, int max_seq_len,
             cudaStream_t s)
{
    switch (G) {
    case 1: return launch_q<D, 1, KV>(pool, prm, batch, max_seq_len, s);
    case 2: return launch_q<D, 2, KV>(pool, prm, batch, max_seq_len, s);
    case 4: return launch_q<D, 4, KV>(pool, prm, batch, max_seq_len, s);
    case 8: return launch_q<D, 8, KV>(pool, prm, batch, max_seq_len, s);
    }
    return PKV_ERR_UNSUPPORTED;
}

template <int KV>
int launch_d(const pkv_pool *pool, int G, const Params &prm, int batch, int max_seq_len,
             cudaStream_t s)
{
    if constexpr (KV == PKV_I4) {
        // a 64-wide 4-bit row is 32 bytes, below the four 16-byte chunks a
        // row is split into; the pool refuses that shape
        return launch_g<128, KV>(pool, G, prm, batch, max_seq_len, s);
    } else {
        if (pool->head_dim == 64)
            return launch_g<64, KV>(pool, G, prm, batch, max_seq_len, s);
        return launch_g<128, KV>(pool, G, prm, batch, max_seq_len, s);
    }
}

}  // namespace kern
}  // namespace pkv
