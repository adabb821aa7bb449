/*
 * CPU oracle for single-token decode attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or constant with the
 * CUDA library: every format conversion, index formula and reduction below is
 * written out again here from its definition.
 *
 * Sources (the three web pages on the KV cache):
 *   [NOTES] "KV cache: the engine behind fast LLM inference"
 *           (curiosity-9m6.pages.dev/notes/0043)
 *   [VIS]   KV cache visualization (cuuduongthancong.com/~galles/visualization/KVCache.html)
 *   [GUIDE] jovanaeducation.com/guides/l-is-2
 *
 * Everything is plain and slow on purpose: attention is evaluated in fp64
 * straight from its definition, after the cached rows have been gathered
 * through the block table into contiguous arrays.  The int8 quantizer runs in
 * fp32 (each step one IEEE operation) so that its integer codes are a fixed,
 * exact function of the input bits.
 *
 * Layouts (fixed by this library, the pages are silent on them):
 *   k_cache, v_cache : [num_blocks][num_kv_heads][block_size][head_dim]
 *   k_scales, v_scales (int8 cache only) : [num_blocks][num_kv_heads][block_size] fp16
 *   q                : [batch][num_q_heads][head_dim]
 *   block_tables     : [batch][max_blocks_per_seq] int32
 *   out              : [batch][num_q_heads][head_dim] fp64
 *
 * Parity status: every function here is pinned by the CPU tests (closed
 * forms, worked figures from the pages, brute force, library routines);
 * none is unpinned.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2, ORC_I8 = 3, ORC_I4 = 4 };

/* ------------------------------------------------------------------ */
/* Number formats, from the IEEE 754 binary16 / bfloat16 definitions.  */
/* ------------------------------------------------------------------ */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double orc_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);            /* subnormal: f * 2^-14 * 2^-10 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16 is the upper half of a binary32 word. */
double orc_bf16_to_double(uint16_t b)
{
    uint32_t w = (uint32_t)b << 16;
    float x;
    memcpy(&x, &w, 4);
    return (double)x;
}

/* binary32 -> binary16, round to nearest, ties to even; overflow gives inf. */
uint16_t orc_float_to_half_rne(float x)
{
    uint32_t w;
    memcpy(&w, &x, 4);
    uint16_t sign = (uint16_t)((w >> 16) & 0x8000);
    double a = fabs((double)x);
    if (x != x)
        return (uint16_t)(sign | 0x7e00);
    if (a >= 65520.0)                  /* at or above max + half ulp: rounds to inf */
        return (uint16_t)(sign | 0x7c00);
    /* The exact value is a; pick the binary16 quantum for its binade and
     * round a / quantum to an integer, ties to even.  Everything is exact
     * in fp64 because binary32 has 24 significant bits. */
    int e;
    if (a < ldexp(1.0, -14)) {
        e = -14;                              /* subnormal range, quantum 2^-24 */
    } else {
        frexp(a, &e);                         /* a = m * 2^e, m in [0.5, 1) */
        e -= 1;                               /* a in [2^e, 2^(e+1)) */
    }
    double quantum = ldexp(1.0, e - 10);
    double n = a / quantum;                   /* exact */
    double fl = floor(n);
    double rem = n - fl;
    double r;
    if (rem > 0.5)
        r = fl + 1.0;
    else if (rem < 0.5)
        r = fl;
    else
        r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
    double v = r * quantum;                   /* exact, may step up a binade */
    if (v >= 65520.0)
        return (uint16_t)(sign | 0x7c00);
    /* encode v */
    if (v < ldexp(1.0, -14)) {
        uint16_t frac = (uint16_t)(v / ldexp(1.0, -24));
        return (uint16_t)(sign | frac);
    }
    int ev;
    double m = frexp(v, &ev);                 /* v = m * 2^ev, m in [0.5,1) */
    int biased = ev - 1 + 15;
    uint16_t frac = (uint16_t)((m * 2.0 - 1.0) * 1024.0);
    return (uint16_t)(sign | (biased << 10) | frac);
}

static double load_elem(const void *base, int dtype, int64_t idx)
{
    switch (dtype) {
    case ORC_F32: return (double)((const float *)base)[idx];
    case ORC_F16: return orc_half_to_double(((const uint16_t *)base)[idx]);
    case ORC_BF16: return orc_bf16_to_double(((const uint16_t *)base)[idx]);
    case ORC_I8: return (double)((const int8_t *)base)[idx];
    case ORC_I4: {
        /* element idx is nibble idx % 2 of byte idx / 2 (low nibble first),
         * a two's-complement 4-bit code */
        unsigned byte = ((const uint8_t *)base)[idx / 2];
        int nib = (int)((idx % 2) ? (byte >> 4) : (byte & 15u));
        return (double)(nib >= 8 ? nib - 16 : nib);
    }
    default: return NAN;
    }
}

static int elem_bytes(int dtype)
{
    switch (dtype) {
    case ORC_F32: return 4;
    case ORC_F16: case ORC_BF16: return 2;
    case ORC_I8: return 1;
    default: return 0;
    }
}

/* ------------------------------------------------------------------ */
/* Slot mapping.                                                        */
/* [VIS] "PagedAttention: the cache in blocks": each request keeps a    */
/* block table, the ordered list of its block numbers, and blocks are   */
/* a fixed number of tokens.  So logical position pos of a request lies */
/* in its (pos / bs)-th block, at offset pos % bs inside that block.    */
/* The cache slot is that physical block times bs plus the offset.      */
/* ------------------------------------------------------------------ */
int64_t orc_slot_of(const int32_t *block_table_row, int block_size, int64_t pos)
{
    int64_t logical_block = pos / block_size;
    int64_t offset = pos % block_size;
    return (int64_t)block_table_row[logical_block] * block_size + offset;
}

/* Slot mapping for a step: sequence b gets n_new[b] new tokens at
 * positions start[b] .. start[b]+n_new[b]-1; slots are written in
 * sequence order. */
void orc_slot_mapping(const int32_t *block_tables, int max_blocks_per_seq, int block_size,
                      int batch, const int32_t *start, const int32_t *n_new, int32_t *slots)
{
    int64_t k = 0;
    for (int b = 0; b < batch; ++b)
        for (int j = 0; j < n_new[b]; ++j)
            slots[k++] = (int32_t)orc_slot_of(block_tables + (int64_t)b * max_blocks_per_seq,
                                              block_size, (int64_t)start[b] + j);
}

/* Byte offset of element (slot, head, i) in a [NB][Hkv][bs][D] cache. */
static int64_t cache_index(int64_t slot, int head, int i, int block_size, int num_kv_heads,
                           int head_dim)
{
    int64_t blk = slot / block_size;
    int64_t off = slot % block_size;
    return ((blk * num_kv_heads + head) * block_size + off) * head_dim + i;
}

/* ------------------------------------------------------------------ */
/* Append: [NOTES] "What happens at each decoding step", step 4 (the    */
/* new token's key and value join the cache); [VIS] "The idea".  The new */
/* rows are copied bit for bit to their slots.  slot < 0 marks a padding */
/* token and is skipped.                                                */
/* ------------------------------------------------------------------ */
void orc_append(const void *k_new, const void *v_new, int dtype, const int32_t *slots,
                int num_tokens, int num_kv_heads, int head_dim, int block_size,
                void *k_cache, void *v_cache)
{
    int eb = elem_bytes(dtype);
    for (int t = 0; t < num_tokens; ++t) {
        if (slots[t] < 0)
            continue;
        for (int h = 0; h < num_kv_heads; ++h) {
            int64_t src = ((int64_t)t * num_kv_heads + h) * head_dim;
            int64_t dst = cache_index(slots[t], h, 0, block_size, num_kv_heads, head_dim);
            memcpy((char *)k_cache + dst * eb, (const char *)k_new + src * eb, (size_t)head_dim * eb);
            memcpy((char *)v_cache + dst * eb, (const char *)v_new + src * eb, (size_t)head_dim * eb);
        }
    }
}

/* ------------------------------------------------------------------ */
/* Copy-on-write: [VIS] "PagedAttention: the cache in blocks".  Sequences */
/* that begin alike may reference one physical copy of their first blocks; */
/* a sharer that must modify such a block first gets a private block with */
/* the same rows.  So every element (head, offset, i) of      */
/* block src[j] is copied to the same place in block dst[j].  One call   */
/* handles one array: a K or V cache (row = head_dim elements), or the   */
/* int8 scales (row = 1 element of 2 bytes).                             */
/* ------------------------------------------------------------------ */
void orc_block_copy(void *cache, int elem_size, int num_kv_heads, int block_size, int row_len,
                    const int32_t *src, const int32_t *dst, int n)
{
    for (int j = 0; j < n; ++j)
        for (int h = 0; h < num_kv_heads; ++h)
            for (int off = 0; off < block_size; ++off)
                for (int i = 0; i < row_len; ++i) {
                    int64_t from = cache_index((int64_t)src[j] * block_size + off, h, i,
                                               block_size, num_kv_heads, row_len);
                    int64_t to = cache_index((int64_t)dst[j] * block_size + off, h, i,
                                             block_size, num_kv_heads, row_len);
                    memcpy((char *)cache + to * elem_size, (const char *)cache + from * elem_size,
                           (size_t)elem_size);
                }
}

/* ------------------------------------------------------------------ */
/* int8 quantization of one (token, head) row.                          */
/* [NOTES] "How serving systems tame the cost", "Quantized KV cache":   */
/* the cached K and V may be kept in fewer bits (int8 codes in place of  */
/* fp16 values).  The pages fix no scheme; this library's reading is     */
/* symmetric per-token-per-head quantization with an fp16 scale:         */
/*   amax = max |x_i|            (fp32)                                  */
/*   s    = fp16_rne(amax / 127) (fp32 division, then round to fp16)     */
/*   code = clamp(round_half_even(x_i / s), -127, 127)   (fp32 division) */
/* A zero scale (amax == 0, or amax/127 below the fp16 range) gives all  */
/* codes 0.                                                              */
/* ------------------------------------------------------------------ */
static float rint_half_even_f(float x)
{
    /* x is finite here.  Integers at or above 2^23 are already exact. */
    float a = fabsf(x);
    if (a >= 8388608.0f)
        return x;
    float fl = floorf(a);
    float rem = a - fl;                       /* exact for a < 2^23 */
    float r;
    if (rem > 0.5f)
        r = fl + 1.0f;
    else if (rem < 0.5f)
        r = fl;
    else
        r = (fmodf(fl, 2.0f) == 0.0f) ? fl : fl + 1.0f;
    return x < 0 ? -r : r;
}

void orc_quantize_row_q8(const float *x, int n, int8_t *codes, uint16_t *scale_bits)
{
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) {
        float a = fabsf(x[i]);
        if (a > amax)
            amax = a;
    }
    volatile float s32 = amax / 127.0f;
    uint16_t s16 = orc_float_to_half_rne(s32);
    *scale_bits = s16;
    float s = (float)orc_half_to_double(s16);
    for (int i = 0; i < n; ++i) {
        if (s == 0.0f) {
            codes[i] = 0;
            continue;
        }
        volatile float r = x[i] / s;
        float c = rint_half_even_f(r);
        if (c > 127.0f)
            c = 127.0f;
        if (c < -127.0f)
            c = -127.0f;
        codes[i] = (int8_t)c;
    }
}

/* Quantize-on-append: the new rows (in_dtype f32/f16/bf16, widened to
 * fp32 exactly) are quantized per (token, head) and written with their
 * scales to the int8 cache. */
void orc_append_q8(const void *k_new, const void *v_new, int in_dtype, const int32_t *slots,
                   int num_tokens, int num_kv_heads, int head_dim, int block_size,
                   int8_t *k_cache, int8_t *v_cache, uint16_t *k_scales, uint16_t *v_scales)
{
    float *row = (float *)malloc(sizeof(float) * head_dim);
    for (int t = 0; t < num_tokens; ++t) {
        if (slots[t] < 0)
            continue;
        for (int h = 0; h < num_kv_heads; ++h) {
            int64_t src = ((int64_t)t * num_kv_heads + h) * head_dim;
            int64_t dst = cache_index(slots[t], h, 0, block_size, num_kv_heads, head_dim);
            int64_t sidx = dst / head_dim;    /* [NB][Hkv][bs] */
            for (int pass = 0; pass < 2; ++pass) {
                const void *srcp = pass == 0 ? k_new : v_new;
                for (int i = 0; i < head_dim; ++i)
                    row[i] = (float)load_elem(srcp, in_dtype, src + i);
                if (pass == 0)
                    orc_quantize_row_q8(row, head_dim, k_cache + dst, &k_scales[sidx]);
                else
                    orc_quantize_row_q8(row, head_dim, v_cache + dst, &v_scales[sidx]);
            }
        }
    }
    free(row);
}

/* ------------------------------------------------------------------ */
/* 4-bit quantization ([NOTES] "Quantized KV cache" stores the cache in  */
/* fewer bits; [VIS] "What the page leaves out" names 8-bit and 4-bit   */
/* caches).  The same symmetric per-token-per-head scheme as int8 with   */
/* the 4-bit range:                                                      */
/*   amax = max |x_i|            (fp32)                                  */
/*   s    = fp16_rne(amax / 7)   (fp32 division, then round to fp16)     */
/*   code = clamp(round_half_even(x_i / s), -7, 7)                       */
/* Codes are stored two per byte, element 2j in the low nibble of byte j */
/* and element 2j+1 in the high nibble, as 4-bit two's complement.  A    */
/* zero scale gives all codes 0.                                         */
/* ------------------------------------------------------------------ */
void orc_quantize_row_q4(const float *x, int n, int8_t *codes, uint16_t *scale_bits)
{
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) {
        float a = fabsf(x[i]);
        if (a > amax)
            amax = a;
    }
    volatile float s32 = amax / 7.0f;
    uint16_t s16 = orc_float_to_half_rne(s32);
    *scale_bits = s16;
    float s = (float)orc_half_to_double(s16);
    for (int i = 0; i < n; ++i) {
        if (s == 0.0f) {
            codes[i] = 0;
            continue;
        }
        volatile float r = x[i] / s;
        float c = rint_half_even_f(r);
        if (c > 7.0f)
            c = 7.0f;
        if (c < -7.0f)
            c = -7.0f;
        codes[i] = (int8_t)c;
    }
}

/* Two codes per byte: element 2j in the low nibble of byte j. */
void orc_pack_q4(const int8_t *codes, int n, uint8_t *bytes)
{
    for (int j = 0; j < n / 2; ++j)
        bytes[j] = (uint8_t)(((unsigned)codes[2 * j] & 15u) |
                             (((unsigned)codes[2 * j + 1] & 15u) << 4));
}

void orc_append_q4(const void *k_new, const void *v_new, int in_dtype, const int32_t *slots,
                   int num_tokens, int num_kv_heads, int head_dim, int block_size,
                   uint8_t *k_cache, uint8_t *v_cache, uint16_t *k_scales, uint16_t *v_scales)
{
    float *row = (float *)malloc(sizeof(float) * head_dim);
    int8_t *codes = (int8_t *)malloc((size_t)head_dim);
    for (int t = 0; t < num_tokens; ++t) {
        if (slots[t] < 0)
            continue;
        for (int h = 0; h < num_kv_heads; ++h) {
            int64_t src = ((int64_t)t * num_kv_heads + h) * head_dim;
            int64_t dst = cache_index(slots[t], h, 0, block_size, num_kv_heads, head_dim);
            int64_t sidx = dst / head_dim;
            for (int kv = 0; kv < 2; ++kv) {
                const void *in = kv == 0 ? k_new : v_new;
                for (int i = 0; i < head_dim; ++i)
                    row[i] = (float)load_elem(in, in_dtype, src + i);
                if (kv == 0) {
                    orc_quantize_row_q4(row, head_dim, codes, &k_scales[sidx]);
                    orc_pack_q4(codes, head_dim, k_cache + dst / 2);
                } else {
                    orc_quantize_row_q4(row, head_dim, codes, &v_scales[sidx]);
                    orc_pack_q4(codes, head_dim, v_cache + dst / 2);
                }
            }
        }
    }
    free(codes);
    free(row);
}

/* ------------------------------------------------------------------ */
/* Gather: read sequence b's first L cached rows of KV head h through   */
/* its block table into a contiguous fp64 array [L][D]; int8 rows are    */
/* dequantized as code * scale.  [VIS] "PagedAttention: the cache in     */
/* blocks" (block table maps logical to physical blocks).                */
/* ------------------------------------------------------------------ */
/* Rows of positions first .. last-1 (rows[0] is position first). */
void orc_gather_range(const void *cache, const uint16_t *scales, int dtype,
                      const int32_t *block_table_row, int first, int last, int head,
                      int num_kv_heads, int head_dim, int block_size, double *rows)
{
    for (int t = first; t < last; ++t) {
        int64_t slot = orc_slot_of(block_table_row, block_size, t);
        int64_t base = cache_index(slot, head, 0, block_size, num_kv_heads, head_dim);
        double sc = 1.0;
        if (dtype == ORC_I8 || dtype == ORC_I4)
            sc = orc_half_to_double(scales[base / head_dim]);
        for (int i = 0; i < head_dim; ++i)
            rows[(int64_t)(t - first) * head_dim + i] = load_elem(cache, dtype, base + i) * sc;
    }
}

void orc_gather(const void *cache, const uint16_t *scales, int dtype, const int32_t *block_table_row,
                int seq_len, int head, int num_kv_heads, int head_dim, int block_size, double *rows)
{
    orc_gather_range(cache, scales, dtype, block_table_row, 0, seq_len, head, num_kv_heads,
                     head_dim, block_size, rows);
}

/* ------------------------------------------------------------------ */
/* Attention of one query against L contiguous rows, fp64:              */
/* softmax(q . K^T * scale) . V   ([NOTES] "Concept" and step 3 of      */
/* "What happens at each decoding step"; scale is 1/sqrt(d) there).     */
/* Two passes: scores and their maximum, then normalised weights.       */
/* L == 0 gives a zero row.                                             */
/* ------------------------------------------------------------------ */
void orc_attend_rows(const double *q, const double *krows, const double *vrows, int seq_len,
                     int head_dim, double scale, double *out, double *scores)
{
    for (int i = 0; i < head_dim; ++i)
        out[i] = 0.0;
    if (seq_len <= 0)
        return;
    double m = -INFINITY;
    for (int t = 0; t < seq_len; ++t) {
        double s = 0.0;
        for (int i = 0; i < head_dim; ++i)
            s += q[i] * krows[(int64_t)t * head_dim + i];
        s *= scale;
        scores[t] = s;
        if (s > m)
            m = s;
    }
    double denom = 0.0;
    for (int t = 0; t < seq_len; ++t) {
        double w = exp(scores[t] - m);
        scores[t] = w;
        denom += w;
    }
    for (int t = 0; t < seq_len; ++t) {
        double w = scores[t] / denom;
        for (int i = 0; i < head_dim; ++i)
            out[i] += w * vrows[(int64_t)t * head_dim + i];
    }
}

/* ------------------------------------------------------------------ */
/* Paged decode attention for a batch.  For every sequence b and query  */
/* head h: gather K and V of KV head h / G (G = Hq / Hkv consecutive     */
/* query heads share one KV head, [VIS] "How much memory", GQA) through  */
/* the block table, then attend.  seq_lens count the new token, which   */
/* has already been appended.                                           */
/* Returns 0, or -1 when a table entry or length is out of range.       */
/* nthreads <= 0 uses the OpenMP default.                               */
/* ------------------------------------------------------------------ */
/* Sliding window (a variant [VIS] "What the page leaves out" names): with
 * window > 0 a sequence attends over its last min(window, L) rows only,
 * positions L - window .. L-1; the same softmax over fewer rows.  Rows
 * before the window are neither gathered nor looked up.  window == 0 is
 * full attention. */
static int window_start(int L, int window)
{
    return (window > 0 && L > window) ? L - window : 0;
}

int orc_paged_decode_attention_window(const void *q, int q_dtype, int num_q_heads,
                                      const void *k_cache, const void *v_cache,
                                      const uint16_t *k_scales, const uint16_t *v_scales,
                                      int kv_dtype, int num_blocks, int num_kv_heads,
                                      int head_dim, int block_size, const int32_t *block_tables,
                                      int max_blocks_per_seq, const int32_t *seq_lens, int batch,
                                      int window, double scale, double *out, int nthreads)
{
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || window < 0)
        return -1;
    int group = num_q_heads / num_kv_heads;
    for (int b = 0; b < batch; ++b) {
        if (seq_lens[b] < 0 || seq_lens[b] > (int64_t)max_blocks_per_seq * block_size)
            return -1;
        int nb = (seq_lens[b] + block_size - 1) / block_size;
        for (int j = window_start(seq_lens[b], window) / block_size; j < nb; ++j) {
            int32_t id = block_tables[(int64_t)b * max_blocks_per_seq + j];
            if (id < 0 || id >= num_blocks)
                return -1;
        }
    }
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    /* One work item per (sequence, KV head): gather once, attend for the G
     * query heads of the group. */
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t item = 0; item < (int64_t)batch * num_kv_heads; ++item) {
        int b = (int)(item / num_kv_heads);
        int kvh = (int)(item % num_kv_heads);
        int L = seq_lens[b];
        int lo = window_start(L, window);
        int n = L - lo;
        const int32_t *row = block_tables + (int64_t)b * max_blocks_per_seq;
        double *kr = (double *)malloc(sizeof(double) * ((size_t)n * head_dim + 1));
        double *vr = (double *)malloc(sizeof(double) * ((size_t)n * head_dim + 1));
        double *sc = (double *)malloc(sizeof(double) * ((size_t)n + 1));
        double *qd = (double *)malloc(sizeof(double) * head_dim);
        orc_gather_range(k_cache, k_scales, kv_dtype, row, lo, L, kvh, num_kv_heads, head_dim,
                         block_size, kr);
        orc_gather_range(v_cache, v_scales, kv_dtype, row, lo, L, kvh, num_kv_heads, head_dim,
                         block_size, vr);
        for (int g = 0; g < group; ++g) {
            int h = kvh * group + g;
            int64_t qb = ((int64_t)b * num_q_heads + h) * head_dim;
            for (int i = 0; i < head_dim; ++i)
                qd[i] = load_elem(q, q_dtype, qb + i);
            orc_attend_rows(qd, kr, vr, n, head_dim, scale, out + qb, sc);
        }
        free(kr);
        free(vr);
        free(sc);
        free(qd);
    }
    return 0;
}

int orc_paged_decode_attention(const void *q, int q_dtype, int num_q_heads, const void *k_cache,
                               const void *v_cache, const uint16_t *k_scales,
                               const uint16_t *v_scales, int kv_dtype, int num_blocks,
                               int num_kv_heads, int head_dim, int block_size,
                               const int32_t *block_tables, int max_blocks_per_seq,
                               const int32_t *seq_lens, int batch, double scale, double *out,
                               int nthreads)
{
    return orc_paged_decode_attention_window(q, q_dtype, num_q_heads, k_cache, v_cache, k_scales,
                                             v_scales, kv_dtype, num_blocks, num_kv_heads,
                                             head_dim, block_size, block_tables,
                                             max_blocks_per_seq, seq_lens, batch, 0, scale, out,
                                             nthreads);
}

/* ------------------------------------------------------------------ */
/* Prefill attention ([VIS] "Prefill and decode feel different": the    */
/* prompt is processed as one batch of tokens; [GUIDE] "How the cache turns the */
/* loop cheap": the prompt's keys and values are all made, and cached,  */
/* in that one pass).  Sequence b has n_b new tokens, the last n_b of    */
/* its seq_lens[b] cached rows (already appended); new token i sits at   */
/* position p = seq_lens[b] - n_b + i and attends over positions 0..p    */
/* (causal),                                                             */
/* with the softmax of [NOTES] "Concept".  q rows are sequence-major:    */
/* q[q_start[b] + i][h][:], and so is out.                                */
/* ------------------------------------------------------------------ */
int orc_paged_prefill_attention(const void *q, int q_dtype, int num_q_heads, const void *k_cache,
                                const void *v_cache, int kv_dtype, int num_blocks,
                                int num_kv_heads, int head_dim, int block_size,
                                const int32_t *block_tables, int max_blocks_per_seq,
                                const int32_t *q_start, const int32_t *seq_lens, int batch,
                                double scale, double *out, int nthreads)
{
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0)
        return -1;
    int group = num_q_heads / num_kv_heads;
    for (int b = 0; b < batch; ++b) {
        int n = q_start[b + 1] - q_start[b];
        if (n < 0 || seq_lens[b] < n || seq_lens[b] > (int64_t)max_blocks_per_seq * block_size)
            return -1;
        int nb = (seq_lens[b] + block_size - 1) / block_size;
        for (int j = 0; j < nb; ++j) {
            int32_t id = block_tables[(int64_t)b * max_blocks_per_seq + j];
            if (id < 0 || id >= num_blocks)
                return -1;
        }
    }
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t item = 0; item < (int64_t)batch * num_kv_heads; ++item) {
        int b = (int)(item / num_kv_heads);
        int kvh = (int)(item % num_kv_heads);
        int L = seq_lens[b];
        int n = q_start[b + 1] - q_start[b];
        const int32_t *row = block_tables + (int64_t)b * max_blocks_per_seq;
        double *kr = (double *)malloc(sizeof(double) * ((size_t)L * head_dim + 1));
        double *vr = (double *)malloc(sizeof(double) * ((size_t)L * head_dim + 1));
        double *sc = (double *)malloc(sizeof(double) * ((size_t)L + 1));
        double *qd = (double *)malloc(sizeof(double) * head_dim);
        orc_gather(k_cache, NULL, kv_dtype, row, L, kvh, num_kv_heads, head_dim, block_size, kr);
        orc_gather(v_cache, NULL, kv_dtype, row, L, kvh, num_kv_heads, head_dim, block_size, vr);
        for (int i = 0; i < n; ++i) {
            int p = L - n + i;
            for (int g = 0; g < group; ++g) {
                int h = kvh * group + g;
                int64_t qb = ((int64_t)(q_start[b] + i) * num_q_heads + h) * head_dim;
                for (int d = 0; d < head_dim; ++d)
                    qd[d] = load_elem(q, q_dtype, qb + d);
                orc_attend_rows(qd, kr, vr, p + 1, head_dim, scale, out + qb, sc);
            }
        }
        free(kr);
        free(vr);
        free(sc);
        free(qd);
    }
    return 0;
}

int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------ */
/* Memory figures.  [VIS] "How much memory": bytes per token =          */
/* 2 (K and V) x layers x KV heads x head dim x bytes per number;       */
/* [GUIDE] "The catch: the cache eats your GPU" gives the same product. */
/* ------------------------------------------------------------------ */
int64_t orc_kv_bytes_per_token(int64_t n_layers, int64_t n_kv_heads, int64_t head_dim,
                               int64_t bytes_per_number)
{
    return 2 * n_layers * n_kv_heads * head_dim * bytes_per_number;
}

/* ------------------------------------------------------------------ */
/* Toy generation loop, [VIS] "Without vs with the cache".  A prompt of  */
/* p tokens is followed by s decode steps.  Token embeddings x[t] (one   */
/* per position, given) are projected to q, k, v by fixed matrices      */
/* Wq, Wk, Wv ([D][E] row-major).  The uncached lane recomputes k and v  */
/* for every token of the prefix at every step; the cached lane computes */
/* them once and keeps them in a paged cache of block size bs (blocks    */
/* taken in order 0, 1, 2, ...).  Both lanes attend the newest token's   */
/* query against every row.  Rows computed are counted per step.        */
/* Outputs: out_nocache, out_cache [s+1][D] (step 0 = end of prefill),   */
/* rows_nocache, rows_cache [s+1].                                      */
/* ------------------------------------------------------------------ */
static void project(const double *W, const double *x, int D, int E, double *y)
{
    for (int r = 0; r < D; ++r) {
        double acc = 0.0;
        for (int c = 0; c < E; ++c)
            acc += W[(int64_t)r * E + c] * x[c];
        y[r] = acc;
    }
}

void orc_toy_generation(const double *x, int prompt_len, int decode_steps, int E, int D,
                        const double *Wq, const double *Wk, const double *Wv, int block_size,
                        double *out_nocache, double *out_cache, int64_t *rows_nocache,
                        int64_t *rows_cache)
{
    int n = prompt_len + decode_steps;
    double scale = 1.0 / sqrt((double)D);
    double *q = (double *)malloc(sizeof(double) * D);
    double *kr = (double *)malloc(sizeof(double) * (size_t)n * D);
    double *vr = (double *)malloc(sizeof(double) * (size_t)n * D);
    double *sc = (double *)malloc(sizeof(double) * n);
    int nblocks = (n + block_size - 1) / block_size;
    /* paged cache for the cached lane: one KV head */
    double *kc = (double *)malloc(sizeof(double) * (size_t)nblocks * block_size * D);
    double *vc = (double *)malloc(sizeof(double) * (size_t)nblocks * block_size * D);
    /* a non-identity table: logical block j lives in physical block nblocks-1-j */
    int32_t *table = (int32_t *)malloc(sizeof(int32_t) * nblocks);
    for (int j = 0; j < nblocks; ++j)
        table[j] = nblocks - 1 - j;
    double *kg = (double *)malloc(sizeof(double) * (size_t)n * D);
    double *vg = (double *)malloc(sizeof(double) * (size_t)n * D);

    for (int step = 0; step <= decode_steps; ++step) {
        int len = prompt_len + step;          /* tokens seen after this step */
        int newest = len - 1;
        /* uncached lane: recompute every row */
        int64_t cnt = 0;
        for (int t = 0; t < len; ++t) {
            project(Wk, x + (int64_t)t * E, D, E, kr + (int64_t)t * D);
            project(Wv, x + (int64_t)t * E, D, E, vr + (int64_t)t * D);
            ++cnt;
        }
        rows_nocache[step] = cnt;
        project(Wq, x + (int64_t)newest * E, D, E, q);
        orc_attend_rows(q, kr, vr, len, D, scale, out_nocache + (int64_t)step * D, sc);
        /* cached lane: compute only the rows not yet cached, append them */
        int first_new = step == 0 ? 0 : len - 1;
        cnt = 0;
        for (int t = first_new; t < len; ++t) {
            int64_t slot = orc_slot_of(table, block_size, t);
            project(Wk, x + (int64_t)t * E, D, E, kc + slot * D);
            project(Wv, x + (int64_t)t * E, D, E, vc + slot * D);
            ++cnt;
        }
        rows_cache[step] = cnt;
        for (int t = 0; t < len; ++t) {
            int64_t slot = orc_slot_of(table, block_size, t);
            memcpy(kg + (int64_t)t * D, kc + slot * D, sizeof(double) * D);
            memcpy(vg + (int64_t)t * D, vc + slot * D, sizeof(double) * D);
        }
        orc_attend_rows(q, kg, vg, len, D, scale, out_cache + (int64_t)step * D, sc);
    }
    free(q); free(kr); free(vr); free(sc); free(kc); free(vc); free(table); free(kg); free(vg);
}
