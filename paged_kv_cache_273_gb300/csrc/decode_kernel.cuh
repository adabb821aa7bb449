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
//    so the kernel is built to stream K/V at HBM bandwidth.  CUDA cores, no
//    tensor cores: G query heads per K/V byte is far below the tensor ridge.
//  * The batch's work is a list of 16-token tiles, ordered by (sequence,
//    KV head, tile).  A persistent grid of one CTA per SM takes an equal,
//    contiguous share of that list (split-K across the sequence axis,
//    balanced to +-1 tile whatever the length mix).
//  * In each CTA one producer warp issues bulk async copies (cp.async.bulk)
//    of whole K and V tiles, located through the block table, into a ring of
//    shared-memory stages guarded by mbarriers; eight consumer warps take
//    tiles round-robin, each keeping its own online-softmax state (the
//    FlashAttention idea of never materialising the score row, from the
//    guide's "Flash attention: don't build the giant matrix").
//  * At the end of each (sequence, KV head) piece the consumer warps merge
//    their states.  A piece that is the whole sequence is written to `out`;
//    otherwise the CTA stores a partial (max, sum, weighted V) and the last
//    CTA to finish that sequence/head (a counter in the workspace) merges
//    all partials in a fixed order and resets the counter.
//  * Every mbarrier wait is bounded; on timeout the kernel records
//    PKV_EBIT_TIMEOUT, winds down without further waits and lets its own
//    copies drain before exiting.

#pragma once

#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "device_common.cuh"

namespace pkv {
namespace kern {

using namespace dev;

constexpr int TILE = 16;        // tokens per pipeline stage
constexpr int NWARP_C = 8;      // consumer warps per CTA
constexpr int NTHREADS = (NWARP_C + 1) * 32;
constexpr int MAX_STAGES = 32;
// misc ints in shared memory: [0] abort flag, [1] "merge partials" flag,
// [2] a constant zero, [8..8+NWARPS) scan scratch, [32..32+MAX_STAGES) last
// issued round per stage (+1; 0 = never), [64..66) q copies issued per slot.
constexpr int MISC_INTS = 72;
constexpr int MISC_ISSUED = 32;
constexpr int MISC_QISSUED = 64;

__host__ __device__ constexpr int round_up(int x, int a) { return (x + a - 1) / a * a; }

template <int KV>
struct KvBytes;
template <> struct KvBytes<PKV_F32> { static constexpr int v = 4; };
template <> struct KvBytes<PKV_F16> { static constexpr int v = 2; };
template <> struct KvBytes<PKV_BF16> { static constexpr int v = 2; };
template <> struct KvBytes<PKV_I8> { static constexpr int v = 1; };

template <int D, int G, int KV>
struct Cfg {
    static constexpr int W = NWARP_C;
    static constexpr int EB = KvBytes<KV>::v;
    static constexpr int ROWB = D * EB;            // bytes of one cached row
    static constexpr int NCH = ROWB / 16;          // 16-byte chunks per row
    static constexpr int DS = NCH >= 8 ? 8 : NCH;  // lanes sharing one token's dot product
    static constexpr int TQ = 32 / DS;             // token groups per warp
    static constexpr int TPL = TILE / TQ;          // tokens per lane per tile
    static constexpr int CPL = NCH / DS;           // chunks per lane per token
    static constexpr int NP = TPL * G;             // partial dots per lane
    static constexpr int NF = G >= 2 ? G / 2 : 1;  // scores per lane after reduction
    static constexpr int VE = D / 32;              // V elements per lane
    static constexpr int KV_BYTES = TILE * ROWB;
    static constexpr int SC_BYTES = KV == PKV_I8 ? TILE * 2 : 0;
    static constexpr int STAGE_BYTES = round_up(2 * KV_BYTES + 2 * SC_BYTES, 128);
    static constexpr int QSLOT = round_up(G * D * 4, 128);   // fits any q dtype
    static constexpr int MERGE_FLOATS = W * G * (D + 2);
    static constexpr int PS_FLOATS = W * (TILE * G + G);
    static_assert(NCH >= 4 && (NCH % DS) == 0, "row must split into 16-byte chunks");
    static_assert(TPL * TQ == TILE, "tile split");
};

struct Params {
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
    int num_blocks;
    int q_dtype;
    int q_bytes;
    int nst;
    float scale_log2;   // scale * log2(e): scores live in the log2 domain
};

// Shared-memory carve-up (dynamic), identical on host and device.
struct Layout {
    int stages, qring, merge, ps, lens, tstart, bars, misc, total;
};

template <int D, int G, int KV>
__host__ __device__ inline Layout make_layout(int nst, int batch)
{
    using C = Cfg<D, G, KV>;
    Layout L;
    int o = 0;
    L.stages = o; o += nst * C::STAGE_BYTES;
    L.qring = o; o += 2 * C::QSLOT;
    L.merge = o; o += C::MERGE_FLOATS * 4;
    L.ps = o; o += C::PS_FLOATS * 4;
    L.lens = o; o += batch * 4;
    L.tstart = o; o += (batch + 1) * 4;
    o = round_up(o, 8);
    L.bars = o; o += (2 * nst + 4) * 8;
    L.misc = o; o += MISC_INTS * 4;
    L.total = round_up(o, 128);
    return L;
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
            } else {
#pragma unroll
                for (int u = 0; u < 16; ++u)
                    qr.w[g][c][u] = q_elem(qs, g * D + chunk * 16 + u, q_dtype);
            }
        }
}

// part[ii*G + g] += q[g] . K[token t_ii] over this lane's chunks.
template <int D, int G, int KV>
__device__ __forceinline__ void qk_tile(float (&part)[Cfg<D, G, KV>::NP],
                                        const QRegs<D, G, KV> &qr, const unsigned char *sK,
                                        int tq, int ds)
{
    using C = Cfg<D, G, KV>;
#pragma unroll
    for (int ii = 0; ii < C::TPL; ++ii) {
        const int t = tq + C::TQ * ii;
#pragma unroll
        for (int c = 0; c < C::CPL; ++c) {
            const int chunk = ds + C::DS * c;
            const uint4 kw = *reinterpret_cast<const uint4 *>(sK + t * C::ROWB + chunk * 16);
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
            } else {
                float kf[16];
                const uint32_t wds[4] = {kw.x ^ 0x80808080u, kw.y ^ 0x80808080u,
                                         kw.z ^ 0x80808080u, kw.w ^ 0x80808080u};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    kf[4 * u + 0] = i8_to_float<0>(wds[u]);
                    kf[4 * u + 1] = i8_to_float<1>(wds[u]);
                    kf[4 * u + 2] = i8_to_float<2>(wds[u]);
                    kf[4 * u + 3] = i8_to_float<3>(wds[u]);
                }
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float a = part[ii * G + g];
#pragma unroll
                    for (int u = 0; u < 16; ++u)
                        a = fmaf(qr.w[g][c][u], kf[u], a);
                    part[ii * G + g] = a;
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
    constexpr int ROWB = D * KvBytes<KV>::v;
    const unsigned char *p = sV + t * ROWB + lane * VE * KvBytes<KV>::v;
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
    } else {
        if constexpr (VE == 4) {
            const uint32_t b = *reinterpret_cast<const uint32_t *>(p) ^ 0x80808080u;
            v[0] = i8_to_float<0>(b); v[1] = i8_to_float<1>(b);
            v[2] = i8_to_float<2>(b); v[3] = i8_to_float<3>(b);
        } else {
            const uint32_t b = (uint32_t)(*reinterpret_cast<const uint16_t *>(p)) ^ 0x8080u;
            v[0] = i8_to_float<0>(b); v[1] = i8_to_float<1>(b);
        }
    }
}

// ---- the kernel ---------------------------------------------------------------

template <int D, int G, int KV>
__global__ void __launch_bounds__(NTHREADS, 1) paged_decode_kernel(const Params p)
{
    using C = Cfg<D, G, KV>;
    constexpr int W = C::W;
    extern __shared__ __align__(128) unsigned char smem[];
    const Layout lay = make_layout<D, G, KV>(p.nst, p.batch);
    unsigned char *stages = smem + lay.stages;
    unsigned char *qring = smem + lay.qring;
    float *merge = reinterpret_cast<float *>(smem + lay.merge);
    float *psbuf = reinterpret_cast<float *>(smem + lay.ps);
    int *s_len = reinterpret_cast<int *>(smem + lay.lens);
    int *s_tstart = reinterpret_cast<int *>(smem + lay.tstart);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + lay.bars);
    uint64_t *empty = full + p.nst;
    uint64_t *qfull = empty + p.nst;
    uint64_t *qempty = qfull + 2;
    int *misc = reinterpret_cast<int *>(smem + lay.misc);
    volatile int *abort_flag = misc + 0;  // set on any timeout
    // misc[1]: "this CTA merges the partials"; misc[2]: zero word; misc[8..]: scan scratch

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int Hkv = p.num_kv_heads;
    const int B = p.batch;

    if (tid == 0) {
        for (int s = 0; s < p.nst; ++s) {
            mbar_init(&full[s], 1);
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

    // Sequence lengths (validated) and the exclusive prefix of tiles.
    for (int b = tid; b < B; b += NTHREADS) {
        int L = __ldg(p.seq_lens + b);
        if (L < 0 || L > p.len_cap) {
            if (blockIdx.x == 0)
                atomicOr(p.err, PKV_EBIT_SEQLEN);
            L = 0;
        }
        s_len[b] = L;
    }
    __syncthreads();
    {
        const int per = (B + NTHREADS - 1) / NTHREADS;
        const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
        int sum = 0;
        for (int b = b0; b < b1; ++b)
            sum += ((s_len[b] + TILE - 1) / TILE) * Hkv;
        int incl = sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(FULL_MASK, incl, off);
            if (lane >= off)
                incl += y;
        }
        int *wsum = misc + 8;
        if (lane == 31)
            wsum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int v = lane < (NTHREADS / 32) ? wsum[lane] : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(FULL_MASK, v, off);
                if (lane >= off)
                    v += y;
            }
            if (lane < (NTHREADS / 32))
                wsum[lane] = v;
        }
        __syncthreads();
        int base = (warp > 0 ? wsum[warp - 1] : 0) + incl - sum;
        for (int b = b0; b < b1; ++b) {
            s_tstart[b] = base;
            base += ((s_len[b] + TILE - 1) / TILE) * Hkv;
        }
        if (tid == 0)
            s_tstart[B] = wsum[NTHREADS / 32 - 1];
    }
    __syncthreads();

    // The T tiles are split over P = min(grid, T) CTAs, so that every CTA
    // that takes part owns at least one tile and the CTAs holding pieces of
    // one sequence/head are consecutive (the merge counts on both).
    const int64_t T = s_tstart[B];
    const int P = (int)min((int64_t)gridDim.x, T);
    const int cta = blockIdx.x;
    const int64_t R0 = cta < P ? (int64_t)cta * T / P : 0;
    const int64_t R1 = cta < P ? (int64_t)(cta + 1) * T / P : 0;
    const int Hq = p.num_q_heads;

    if (warp == W) {
        // ================= producer warp =================
        int64_t seg_prev = -1;
        int qn = 0;
        const int n_local = (int)(R1 - R0);
        const int bs = p.block_size;
        const uint64_t policy = policy_evict_first();
        for (int k0 = 0; k0 < n_local; k0 += 32) {
            // Lane j describes tile R0 + k0 + j.
            int b = 0, kvh = 0, ti = 0, nvalid = 0, nblk = 0;
            int32_t id0 = -1, id1 = -1, id2 = -1, id3 = -1;
            if (k0 + lane < n_local) {
                const int64_t x = R0 + k0 + lane;
                b = find_seq(s_tstart, B, x);
                const int nt = (s_tstart[b + 1] - s_tstart[b]) / Hkv;
                const int off = (int)(x - s_tstart[b]);
                kvh = off / nt;
                ti = off - kvh * nt;
                nvalid = min(TILE, s_len[b] - TILE * ti);
                const int32_t *row = p.block_tables + (int64_t)b * p.max_blocks_per_seq;
                const int first = (TILE * ti) >> p.bs_log2;
                if (bs >= TILE) {
                    nblk = 1;
                    id0 = __ldg(row + first);
                } else {
                    nblk = (nvalid + bs - 1) >> p.bs_log2;   // 1..4 (bs >= 4)
                    id0 = __ldg(row + first);
                    if (nblk > 1) id1 = __ldg(row + first + 1);
                    if (nblk > 2) id2 = __ldg(row + first + 2);
                    if (nblk > 3) id3 = __ldg(row + first + 3);
                }
            }
            const int cnt = min(32, n_local - k0);
            for (int j = 0; j < cnt; ++j) {
                const int bj = __shfl_sync(FULL_MASK, b, j);
                const int kvhj = __shfl_sync(FULL_MASK, kvh, j);
                const int tij = __shfl_sync(FULL_MASK, ti, j);
                const int nbj = __shfl_sync(FULL_MASK, nblk, j);
                int32_t ids[4];
                ids[0] = __shfl_sync(FULL_MASK, id0, j);
                ids[1] = __shfl_sync(FULL_MASK, id1, j);
                ids[2] = __shfl_sync(FULL_MASK, id2, j);
                ids[3] = __shfl_sync(FULL_MASK, id3, j);
                if (lane == 0) {
                    const int k = k0 + j;
                    const int64_t seg = (int64_t)bj * Hkv + kvhj;
                    if (seg != seg_prev) {
                        const int slot = qn & 1;
                        if (mbar_wait_bounded(&qempty[slot], ((qn >> 1) & 1) ^ 1, abort_flag)) {
                            const uint32_t qbytes = (uint32_t)(G * D * p.q_bytes);
                            mbar_arrive_expect_tx(&qfull[slot], qbytes);
                            const unsigned char *qsrc = static_cast<const unsigned char *>(p.q) +
                                                        ((int64_t)bj * Hq + kvhj * G) * D * p.q_bytes;
                            bulk_g2s(qring + slot * C::QSLOT, qsrc, qbytes, &qfull[slot]);
                            misc[MISC_QISSUED + slot] = (qn >> 1) + 1;
                        } else if (!*abort_flag) {
                            *abort_flag = 1;
                            atomicOr(p.err, PKV_EBIT_TIMEOUT);
                        }
                        ++qn;
                        seg_prev = seg;
                    }
                    const int st = k % p.nst;
                    const uint32_t par = (uint32_t)((k / p.nst) & 1) ^ 1u;
                    if (mbar_wait_bounded(&empty[st], par, abort_flag)) {
                        unsigned char *sK = stages + st * C::STAGE_BYTES;
                        unsigned char *sV = sK + C::KV_BYTES;
                        unsigned char *sKS = sV + C::KV_BYTES;
                        unsigned char *sVS = sKS + C::SC_BYTES;
                        // Count bytes of the copies that will be issued.
                        const int rows_per_copy = bs >= TILE ? TILE : bs;
                        const uint32_t kv_copy = (uint32_t)(rows_per_copy * C::ROWB);
                        const uint32_t sc_copy = (uint32_t)(rows_per_copy * 2);
                        uint32_t total = 0;
                        bool bad = false;
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            if (u < nbj) {
                                if (ids[u] >= 0 && ids[u] < p.num_blocks)
                                    total += 2 * kv_copy + (KV == PKV_I8 ? 2 * sc_copy : 0);
                                else
                                    bad = true;
                            }
                        }
                        if (bad)
                            atomicOr(p.err, PKV_EBIT_BLOCK);
                        mbar_arrive_expect_tx(&full[st], total);
                        misc[MISC_ISSUED + st] = k / p.nst + 1;
                        const int in_block = (TILE * tij) & (bs - 1);
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            if (u < nbj && ids[u] >= 0 && ids[u] < p.num_blocks) {
                                const int64_t row0 =
                                    ((int64_t)ids[u] * Hkv + kvhj) * bs + (bs >= TILE ? in_block : 0);
                                const int dst_row = u * rows_per_copy;
                                bulk_g2s_hint(sK + dst_row * C::ROWB, p.k_cache + row0 * C::ROWB,
                                              kv_copy, &full[st], policy);
                                bulk_g2s_hint(sV + dst_row * C::ROWB, p.v_cache + row0 * C::ROWB,
                                              kv_copy, &full[st], policy);
                                if constexpr (KV == PKV_I8) {
                                    bulk_g2s(sKS + dst_row * 2, p.k_scales + row0, sc_copy, &full[st]);
                                    bulk_g2s(sVS + dst_row * 2, p.v_scales + row0, sc_copy, &full[st]);
                                }
                            }
                        }
                    } else if (!*abort_flag) {
                        *abort_flag = 1;
                        atomicOr(p.err, PKV_EBIT_TIMEOUT);
                    }
                }
                __syncwarp();
            }
        }
    } else {
        // ================= consumer warps =================
        const int w = warp;
        const int ds = lane % C::DS;
        const int tq = lane / C::DS;
        const int ctid = tid;                  // 0 .. W*32-1
        float *ps = psbuf + w * (TILE * G + G);
        float *mw = merge + w * G * (D + 2);

        // Zero rows of empty sequences; sequence b is CTA (b % grid)'s job.
        for (int b = cta; b < B; b += gridDim.x) {
            if (s_len[b] == 0)
                for (int idx = ctid; idx < Hq * D; idx += W * 32)
                    p.out[(int64_t)b * Hq * D + idx] = 0.0f;
        }

        int qn = 0;
        int64_t x = R0;
        while (x < R1) {
            const int b = find_seq(s_tstart, B, x);
            const int nt = (s_tstart[b + 1] - s_tstart[b]) / Hkv;
            const int off = (int)(x - s_tstart[b]);
            const int kvh = off / nt;
            const int ti0 = off - kvh * nt;
            const int64_t seg_begin = (int64_t)s_tstart[b] + (int64_t)kvh * nt;
            const int64_t seg_end = seg_begin + nt;
            const int64_t xe = min(seg_end, R1);
            const int k0 = (int)(x - R0);
            const int k1 = (int)(xe - R0);
            const int L = s_len[b];

            // q of this (sequence, KV head) group.
            QRegs<D, G, KV> qr;
            {
                const int slot = qn & 1;
                if (!mbar_wait_bounded(&qfull[slot], (qn >> 1) & 1, abort_flag) && !*abort_flag) {
                    *abort_flag = 1;
                    atomicOr(p.err, PKV_EBIT_TIMEOUT);
                }
                load_q<D, G, KV>(qr, qring + slot * C::QSLOT, ds, p.q_dtype);
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&qempty[slot]);
                ++qn;
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

            const int kfirst = k0 + (w - k0 % W + W) % W;
            for (int k = kfirst; k < k1; k += W) {
                const int ti = ti0 + (k - k0);
                const int nvalid = min(TILE, L - TILE * ti);
                const int st = k % p.nst;
                if (!mbar_wait_bounded(&full[st], (uint32_t)((k / p.nst) & 1), abort_flag) &&
                    !*abort_flag) {
                    *abort_flag = 1;
                    atomicOr(p.err, PKV_EBIT_TIMEOUT);
                }
                const unsigned char *sK = stages + st * C::STAGE_BYTES;
                const unsigned char *sV = sK + C::KV_BYTES;
                const __half *sKS = reinterpret_cast<const __half *>(sV + C::KV_BYTES);
                const __half *sVS = sKS + TILE;

                // ---- scores: partial dots, then reduce-scatter over the DS lanes
                float part[C::NP];
#pragma unroll
                for (int j = 0; j < C::NP; ++j)
                    part[j] = 0.0f;
                qk_tile<D, G, KV>(part, qr, sK, tq, ds);
                reduce_scatter<C::NP, C::DS / 2>(part, ds);
                // Lane holds token t, heads g0 + r (r < NF).
                const int t = tq + C::TQ * (ds >> 1);
                const int g0 = G >= 2 ? (G / 2) * (ds & 1) : 0;
                float s[C::NF];
                float kscale = p.scale_log2;
                if constexpr (KV == PKV_I8)
                    kscale *= __half2float(sKS[t]);
#pragma unroll
                for (int r = 0; r < C::NF; ++r)
                    s[r] = t < nvalid ? part[r] * kscale : -INFINITY;
                // Tile maximum per head over the lanes holding that head.
                float mx[C::NF];
#pragma unroll
                for (int r = 0; r < C::NF; ++r) {
                    mx[r] = s[r];
#pragma unroll
                    for (int mask = 2; mask < 32; mask <<= 1)
                        mx[r] = fmaxf(mx[r], __shfl_xor_sync(FULL_MASK, mx[r], mask));
                }
                float corr[C::NF], pr[C::NF];
#pragma unroll
                for (int r = 0; r < C::NF; ++r) {
                    const float mnew = fmaxf(m_run[r], mx[r]);   // finite: tile has a valid token
                    corr[r] = exp2f(m_run[r] - mnew);
                    pr[r] = exp2f(s[r] - mnew);
                    l_run[r] = l_run[r] * corr[r] + pr[r];
                    m_run[r] = mnew;
                }
                // Publish p (times the V scale for int8) and the rescale factors.
                if (G >= 2 || (ds & 1) == 0) {
                    float vsc = 1.0f;
                    if constexpr (KV == PKV_I8)
                        vsc = __half2float(sVS[t]);
#pragma unroll
                    for (int r = 0; r < C::NF; ++r)
                        ps[t * G + g0 + r] = pr[r] * vsc;
                    if (tq == 0 && (ds >> 1) == 0) {
#pragma unroll
                        for (int r = 0; r < C::NF; ++r)
                            ps[TILE * G + g0 + r] = corr[r];
                    }
                }
                __syncwarp();

                // ---- weighted V
                float cg[G];
#pragma unroll
                for (int g = 0; g < G; ++g)
                    cg[g] = ps[TILE * G + g];
#pragma unroll
                for (int g = 0; g < G; ++g)
#pragma unroll
                    for (int e = 0; e < C::VE; ++e)
                        acc[g][e] *= cg[g];
                if (nvalid == TILE) {
#pragma unroll
                    for (int tt = 0; tt < TILE; ++tt) {
                        float v[C::VE];
                        load_v<D, KV>(v, sV, tt, lane);
#pragma unroll
                        for (int g = 0; g < G; ++g) {
                            const float pg = ps[tt * G + g];
#pragma unroll
                            for (int e = 0; e < C::VE; ++e)
                                acc[g][e] = fmaf(pg, v[e], acc[g][e]);
                        }
                    }
                } else {
                    for (int tt = 0; tt < nvalid; ++tt) {
                        float v[C::VE];
                        load_v<D, KV>(v, sV, tt, lane);
#pragma unroll
                        for (int g = 0; g < G; ++g) {
                            const float pg = ps[tt * G + g];
#pragma unroll
                            for (int e = 0; e < C::VE; ++e)
                                acc[g][e] = fmaf(pg, v[e], acc[g][e]);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&empty[st]);
            }

            // ---- merge the W warp states of this piece
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
            named_bar_sync(1, W * 32);

            const int c_first = owner_of(seg_begin, T, P);
            const int c_last = owner_of(seg_end - 1, T, P);
            const bool whole = c_first == c_last;
            const int seg = b * Hkv + kvh;
            const int stride = G * (D + 2);
            float *part_out = p.partials + (int64_t)(cta + seg) * stride;
            for (int idx = ctid; idx < G * D; idx += W * 32) {
                const int g = idx / D;
                float M = -INFINITY;
#pragma unroll
                for (int ww = 0; ww < W; ++ww)
                    M = fmaxf(M, merge[ww * stride + G * D + g]);
                float num = 0.0f, den = 0.0f;
#pragma unroll
                for (int ww = 0; ww < W; ++ww) {
                    const float f = exp2f(merge[ww * stride + G * D + g] - M);
                    num = fmaf(f, merge[ww * stride + idx], num);
                    den = fmaf(f, merge[ww * stride + G * D + G + g], den);
                }
                if (whole) {
                    p.out[((int64_t)b * Hq + kvh * G) * D + idx] = num / den;
                } else {
                    part_out[idx] = num;
                    if ((idx % D) == 0) {
                        part_out[G * D + g] = M;
                        part_out[G * D + G + g] = den;
                    }
                }
            }
            if (!whole) {
                __threadfence();
                named_bar_sync(1, W * 32);
                if (ctid == 0) {
                    const int old = atomicAdd(p.counters + seg, 1);
                    misc[1] = (old == c_last - c_first) ? 1 : 0;
                }
                named_bar_sync(1, W * 32);
                if (misc[1]) {
                    __threadfence();
                    const float *base = p.partials + (int64_t)(c_first + seg) * stride;
                    const int npieces = c_last - c_first + 1;
                    for (int idx = ctid; idx < G * D; idx += W * 32) {
                        const int g = idx / D;
                        float M = -INFINITY;
                        for (int pc = 0; pc < npieces; ++pc)
                            M = fmaxf(M, __ldcg(base + pc * stride + G * D + g));
                        float num = 0.0f, den = 0.0f;
                        for (int pc = 0; pc < npieces; ++pc) {
                            const float f = exp2f(__ldcg(base + pc * stride + G * D + g) - M);
                            num = fmaf(f, __ldcg(base + pc * stride + idx), num);
                            den = fmaf(f, __ldcg(base + pc * stride + G * D + G + g), den);
                        }
                        p.out[((int64_t)b * Hq + kvh * G) * D + idx] = num / den;
                    }
                    if (ctid == 0)
                        p.counters[seg] = 0;
                }
            }
            named_bar_sync(1, W * 32);
            x = xe;
        }
    }

    // Let every copy this CTA issued land before the CTA exits (only matters
    // after a timeout; otherwise the consumers already waited for all of them).
    __syncthreads();
    if (*abort_flag && tid == NWARP_C * 32) {
        for (int s = 0; s < p.nst; ++s)
            if (misc[MISC_ISSUED + s] > 0)
                mbar_wait_bounded(&full[s], (uint32_t)((misc[MISC_ISSUED + s] - 1) & 1), misc + 2);
        for (int s = 0; s < 2; ++s)
            if (misc[MISC_QISSUED + s] > 0)
                mbar_wait_bounded(&qfull[s], (uint32_t)((misc[MISC_QISSUED + s] - 1) & 1), misc + 2);
    }
}

// ---- host side ---------------------------------------------------------------

template <int D, int G, int KV>
int launch_t(const pkv_pool *pool, const Params &base, int batch, int max_seq_len,
             cudaStream_t stream)
{
    using C = Cfg<D, G, KV>;
    Params prm = base;
    const Layout fixed = make_layout<D, G, KV>(0, batch);
    const int budget = pool->max_smem_optin - fixed.total - 256;
    int nst = budget / (C::STAGE_BYTES + 16);
    if (nst > MAX_STAGES)
        nst = MAX_STAGES;
    if (nst < 2)
        return PKV_ERR_UNSUPPORTED;
    prm.nst = nst;
    const Layout lay = make_layout<D, G, KV>(nst, batch);

    static int configured_smem = 0;   // per instantiation
    static std::mutex mu;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (lay.total > configured_smem) {
            if (cudaFuncSetAttribute(paged_decode_kernel<D, G, KV>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     lay.total) != cudaSuccess)
                return PKV_ERR_CUDA;
            configured_smem = lay.total;
        }
    }
    const int64_t max_tiles =
        (int64_t)batch * pool->num_kv_heads * ((max_seq_len + TILE - 1) / TILE);
    int64_t P = pool->num_sms;
    if (P > max_tiles)
        P = max_tiles;
    if (P < 1)
        P = 1;
    paged_decode_kernel<D, G, KV><<<(int)P, NTHREADS, lay.total, stream>>>(prm);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

template <int D, int KV>
int launch_g(const pkv_pool *pool, int G, const Params &prm, int batch, int max_seq_len,
             cudaStream_t s)
{
    switch (G) {
    case 1: return launch_t<D, 1, KV>(pool, prm, batch, max_seq_len, s);
    case 2: return launch_t<D, 2, KV>(pool, prm, batch, max_seq_len, s);
    case 4: return launch_t<D, 4, KV>(pool, prm, batch, max_seq_len, s);
    case 8: return launch_t<D, 8, KV>(pool, prm, batch, max_seq_len, s);
    }
    return PKV_ERR_UNSUPPORTED;
}

template <int KV>
int launch_d(const pkv_pool *pool, int G, const Params &prm, int batch, int max_seq_len,
             cudaStream_t s)
{
    if (pool->head_dim == 64)
        return launch_g<64, KV>(pool, G, prm, batch, max_seq_len, s);
    return launch_g<128, KV>(pool, G, prm, batch, max_seq_len, s);
}

}  // namespace kern
}  // namespace pkv
