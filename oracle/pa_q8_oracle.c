/*
 * pa_q8 oracle -- a plain, slow CPU statement of the int8 paged-KV decode
 * path, used ONLY as test infrastructure: by the tests, by the package's
 * smoke check and by the benchmark's CPU-baseline leg.  The product path
 * never links, loads or calls this file, and it shares no code, header,
 * table or constant with the CUDA kernels.
 *
 * What it restates (from the pages' own descriptions, in its own code):
 *
 *  - reshape_and_cache_q8.comp (hanzo-ml 0.11.93), header comment and main():
 *    per (token, kv_head) vector, amax = max |x| starting from 0;
 *    inv = 127/amax (0 when amax is 0); code = clamp(round(x * inv), -127, 127);
 *    4 codes per u32 word in little-endian byte lanes (two's complement);
 *    then one word holding the f32 bit pattern of amax/127 (1.0 when amax
 *    is 0); the token vector lands at
 *    [block, kv_head, offset, word] of a [num_blocks, num_kv_heads,
 *    block_size, head_size/4 + 1] u32 cache; slot 0xFFFFFFFF is skipped.
 *
 *  - paged_attn_q8.comp (hanzo-ml 0.11.92), header comment ("output =
 *    softmax(scale*Q.K^T).V", dequantise as code * token_scale) and main()
 *    (GQA head map kv_head = head / (num_heads / num_kv_heads); logical
 *    token t sits in block_tables[seq][t / block_size] at offset
 *    t % block_size; context_len clamped).
 *
 *  - attention.rs (cherenkov qwen4_exp gpu), attention_b: a context split
 *    into parts whose partial results are merged by a combine step.  The
 *    merge of (max, sum, weighted sum) partials by their log-sum-exp is
 *    written out in oracle_combine below.
 *
 *  - the contiguous q8 cache with a side scale region of attention.rs
 *    (kv_append_q8; one scale per 32-element group), its append and decode.
 *
 *  - the f32 cache variant (paged_attn.comp, named by paged_attn_q8.comp's
 *    header comment as the same math over an f32 cache): a copy writer and
 *    the same fp64 decode over f32 values (end of this file).
 *
 * Arithmetic.  The writer is bit-exact by construction: every f32 operation
 * of the shader (one division, one product, one division for the scale) is
 * done in double and rounded once to float.  For +, -, *, / of two floats
 * that equals the correctly rounded f32 result, because a double carries
 * 53 >= 2*24 + 2 bits.  Rounding is half away from zero (C round()), the
 * reading taken for the shader's round().  The decode is computed in double
 * from the dequantised cache; no blocking, no online rescaling, no
 * reassociation beyond summing in logical token / dimension order.
 *
 * Readings where the pages leave a step open:
 *  - no epsilon in the softmax denominator (the decode shader adds 1e-6);
 *  - context_len is clamped to max_blocks_per_seq * block_size;
 *  - context_len == 0 gives an all-zero output row;
 *  - a NaN product x * inv (only 0 * inf, when 127/amax overflowed for a
 *    tiny amax) gives code 0; +-inf clamps to +-127 in the float domain.
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -fopenmp -ffp-contract=off
 *        -fno-fast-math pa_q8_oracle.c -lm
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define PAD_SLOT 0xFFFFFFFFu

static float float_from_bits(uint32_t u) { float f; memcpy(&f, &u, sizeof f); return f; }
static uint32_t bits_from_float(float f) { uint32_t u; memcpy(&u, &f, sizeof u); return u; }

/* Byte lane `lane` of a packed word as a signed code (two's complement). */
static int code_at(uint32_t word, int lane)
{
    int v = (int)((word >> (8 * lane)) & 0xFFu);
    return v >= 128 ? v - 256 : v;
}

/* round-half-away-from-zero, then clamp to [-127, 127] in the float domain */
static int quantise_one(float t)
{
    if (t != t) return 0;
    double r = round((double)t);
    if (r > 127.0) r = 127.0;
    if (r < -127.0) r = -127.0;
    return (int)r;
}

/* Threads the parallel loops use from now on (rows are independent, so the
 * count changes no result); n <= 0 leaves it unchanged. */
void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Quantise one head_size-long f32 vector into head_size/4 code words plus
 * one scale word (reshape_and_cache_q8.comp, main(): amax reduce -> scale ->
 * pack).  words must hold head_size/4 + 1 entries. */
void oracle_quantize_vector(const float *x, int head_size, uint32_t *words)
{
    float amax = 0.0f;
    for (int d = 0; d < head_size; ++d) {
        float a = fabsf(x[d]);
        if (a > amax) amax = a;
    }
    float inv = amax > 0.0f ? (float)(127.0 / (double)amax) : 0.0f;
    for (int w = 0; w < head_size / 4; ++w) {
        uint32_t word = 0;
        for (int l = 0; l < 4; ++l) {
            float t = (float)((double)x[4 * w + l] * (double)inv);
            int q = quantise_one(t);
            word |= ((uint32_t)q & 0xFFu) << (8 * l);
        }
        words[w] = word;
    }
    float scale = amax > 0.0f ? (float)((double)amax / 127.0) : 1.0f;
    words[head_size / 4] = bits_from_float(scale);
}

/* reshape_and_cache_q8.comp, main(): one writer call.  key/value rows are
 * [num_tokens, num_kv_heads, head_size] f32 with row strides key_stride /
 * value_stride (f32 elements). */
void oracle_reshape_and_cache(const float *key, const float *value,
                              uint32_t *key_cache, uint32_t *value_cache,
                              const uint32_t *slot_mapping, int64_t num_tokens,
                              int64_t key_stride, int64_t value_stride,
                              int num_kv_heads, int head_size, int block_size)
{
    const int64_t wpt = head_size / 4 + 1;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < num_tokens; ++i) {
        uint32_t slot = slot_mapping[i];
        if (slot == PAD_SLOT) continue;
        int64_t block = (int64_t)(slot / (uint32_t)block_size);
        int64_t off = (int64_t)(slot % (uint32_t)block_size);
        for (int h = 0; h < num_kv_heads; ++h) {
            int64_t dst = ((block * num_kv_heads + h) * block_size + off) * wpt;
            oracle_quantize_vector(key + i * key_stride + (int64_t)h * head_size, head_size,
                                   key_cache + dst);
            oracle_quantize_vector(value + i * value_stride + (int64_t)h * head_size, head_size,
                                   value_cache + dst);
        }
    }
}

/* The dequantised vector (code * token scale, exact in double) of logical
 * token t of sequence s, kv head g. */
static void dequant_token(const uint32_t *cache, const uint32_t *block_tables,
                          int max_blocks_per_seq, int num_kv_heads, int head_size,
                          int block_size, int s, int g, int64_t t, double *out)
{
    const int64_t wpt = head_size / 4 + 1;
    uint32_t block = block_tables[(int64_t)s * max_blocks_per_seq + t / block_size];
    int64_t off = t % block_size;
    const uint32_t *vec = cache + (((int64_t)block * num_kv_heads + g) * block_size + off) * wpt;
    double scale = (double)float_from_bits(vec[head_size / 4]);
    for (int d = 0; d < head_size; ++d)
        out[d] = (double)code_at(vec[d / 4], d % 4) * scale;
}

static int64_t clamped_len(const uint32_t *context_lens, int s, int max_blocks_per_seq, int block_size)
{
    int64_t c = context_lens[s];
    int64_t cap = (int64_t)max_blocks_per_seq * block_size;
    return c < cap ? c : cap;
}

/* Partial attention of the query vector qv (head_size floats) against kv head
 * g of sequence s over logical tokens [t0, t1): m = max_t z_t,
 * l = sum_t e^(z_t - m), acc[d] = sum_t e^(z_t - m) v_t[d], z_t = scale * q . k_t.
 * An empty range gives m = -inf, l = 0, acc = 0. */
static void attend(const float *qv, const uint32_t *key_cache, const uint32_t *value_cache,
                   const uint32_t *block_tables, int num_kv_heads, int head_size, int block_size,
                   int max_blocks_per_seq, double scale, int s, int g, int64_t t0, int64_t t1,
                   double *m_out, double *l_out, double *acc)
{
    for (int d = 0; d < head_size; ++d) acc[d] = 0.0;
    *l_out = 0.0;
    *m_out = -INFINITY;
    if (t1 <= t0) return;

    double *z = (double *)malloc(sizeof(double) * (size_t)(t1 - t0));
    double *vec = (double *)malloc(sizeof(double) * (size_t)head_size);
    double m = -INFINITY;
    for (int64_t t = t0; t < t1; ++t) {
        dequant_token(key_cache, block_tables, max_blocks_per_seq, num_kv_heads, head_size,
                      block_size, s, g, t, vec);
        double dot = 0.0;
        for (int d = 0; d < head_size; ++d) dot += (double)qv[d] * vec[d];
        z[t - t0] = scale * dot;
        if (z[t - t0] > m) m = z[t - t0];
    }
    double l = 0.0;
    for (int64_t t = t0; t < t1; ++t) {
        double p = exp(z[t - t0] - m);
        l += p;
        dequant_token(value_cache, block_tables, max_blocks_per_seq, num_kv_heads, head_size,
                      block_size, s, g, t, vec);
        for (int d = 0; d < head_size; ++d) acc[d] += p * vec[d];
    }
    *m_out = m;
    *l_out = l;
    free(vec);
    free(z);
}

/* Partial attention of query row (s, h) over logical tokens [t0, t1), with
 * kv head g = h / (num_heads / num_kv_heads); q is [num_seqs][num_heads][head_size]. */
void oracle_decode_partial(const float *q, const uint32_t *key_cache, const uint32_t *value_cache,
                           const uint32_t *block_tables, int num_heads, int num_kv_heads,
                           int head_size, int block_size, int max_blocks_per_seq, double scale,
                           int s, int h, int64_t t0, int64_t t1,
                           double *m_out, double *l_out, double *acc)
{
    const int g = h / (num_heads / num_kv_heads);
    const float *qv = q + ((int64_t)s * num_heads + h) * head_size;
    attend(qv, key_cache, value_cache, block_tables, num_kv_heads, head_size, block_size,
           max_blocks_per_seq, scale, s, g, t0, t1, m_out, l_out, acc);
}

/* Merge n partials (m_i, l_i, acc_i[D]) of one query row by their
 * log-sum-exp: M = max m_i; L = sum l_i e^(m_i - M);
 * out = sum acc_i e^(m_i - M) / L.  L == 0 (no tokens) gives zeros. */
void oracle_combine(const double *m, const double *l, const double *acc, int n, int head_size,
                    double *out)
{
    double M = -INFINITY;
    for (int i = 0; i < n; ++i) if (m[i] > M) M = m[i];
    for (int d = 0; d < head_size; ++d) out[d] = 0.0;
    if (M == -INFINITY) return;
    double L = 0.0;
    for (int i = 0; i < n; ++i) {
        if (l[i] == 0.0) continue;
        double w = exp(m[i] - M);
        L += l[i] * w;
        for (int d = 0; d < head_size; ++d) out[d] += acc[(int64_t)i * head_size + d] * w;
    }
    for (int d = 0; d < head_size; ++d) out[d] /= L;
}

/* Decode: out[s, h, :] = softmax(scale * q[s,h] . K^T) V over the clamped
 * context of sequence s.  rows == NULL computes every (s, h); otherwise
 * rows holds n_rows (s, h) pairs and out is [n_rows, head_size]. */
void oracle_decode(double *out, const float *q, const uint32_t *key_cache,
                   const uint32_t *value_cache, const uint32_t *block_tables,
                   const uint32_t *context_lens, int num_seqs, int num_heads, int num_kv_heads,
                   int head_size, int block_size, int max_blocks_per_seq, double scale,
                   const int32_t *rows, int64_t n_rows)
{
    int64_t n = rows ? n_rows : (int64_t)num_seqs * num_heads;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < n; ++i) {
        int s = rows ? rows[2 * i] : (int)(i / num_heads);
        int h = rows ? rows[2 * i + 1] : (int)(i % num_heads);
        double *o = out + i * head_size;
        double m, l;
        int64_t c = clamped_len(context_lens, s, max_blocks_per_seq, block_size);
        oracle_decode_partial(q, key_cache, value_cache, block_tables, num_heads, num_kv_heads,
                              head_size, block_size, max_blocks_per_seq, scale, s, h, 0, c,
                              &m, &l, o);
        if (c == 0) continue;           /* all zeros */
        for (int d = 0; d < head_size; ++d) o[d] /= l;
    }
}

/* Multi-row causal decode ("attention.rs", attention_b: the per-row loop
 * over b with t_len = base_pos + b + 1).  Sequence s holds
 * c = min(context_len, max_blocks_per_seq * block_size) tokens, the last
 * num_rows of which are the rows being decoded; query row b attends to the
 * first c - (num_rows - 1 - b) tokens (none -> a zero row).
 * q and out are [num_seqs][num_rows][num_heads][head_size]. */
void oracle_decode_rows(double *out, const float *q, const uint32_t *key_cache,
                        const uint32_t *value_cache, const uint32_t *block_tables,
                        const uint32_t *context_lens, int num_seqs, int num_rows, int num_heads,
                        int num_kv_heads, int head_size, int block_size, int max_blocks_per_seq,
                        double scale)
{
    const int64_t n = (int64_t)num_seqs * num_rows * num_heads;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < n; ++i) {
        const int s = (int)(i / ((int64_t)num_rows * num_heads));
        const int b = (int)((i / num_heads) % num_rows);
        const int h = (int)(i % num_heads);
        double *o = out + i * head_size;
        const int64_t c = clamped_len(context_lens, s, max_blocks_per_seq, block_size);
        const int64_t t1 = c - (num_rows - 1 - b);
        double m, l;
        const int g = h / (num_heads / num_kv_heads);
        const float *qv = q + (((int64_t)s * num_rows + b) * num_heads + h) * head_size;
        attend(qv, key_cache, value_cache, block_tables, num_kv_heads, head_size, block_size,
               max_blocks_per_seq, scale, s, g, 0, t1 > 0 ? t1 : 0, &m, &l, o);
        if (t1 <= 0) continue;          /* zeros */
        for (int d = 0; d < head_size; ++d) o[d] /= l;
    }
}

/* ------------------------------------------------------------------------
 * The f32 cache variant.  paged_attn_q8.comp's header comment describes the
 * q8 shader as the same math and workgroup structure as paged_attn.comp,
 * which reads an f32 cache ("1 byte/elem vs the f32 cache's 4"), and
 * reshape_and_cache_q8.comp says its slot rule mirrors the f32 writer.
 * Neither f32 shader is on the pages; the reading taken here is the q8
 * layout with f32 elements and no scale word:
 * [num_blocks, num_kv_heads, block_size, head_size] f32.  The writer copies
 * each (token, kv head) vector to its slot (PAD slots skipped); the decode
 * is the same fp64 softmax as oracle_decode over those values.
 * ------------------------------------------------------------------------ */

void oracle_reshape_and_cache_f32(const float *key, const float *value,
                                  float *key_cache, float *value_cache,
                                  const uint32_t *slot_mapping, int64_t num_tokens,
                                  int64_t key_stride, int64_t value_stride,
                                  int num_kv_heads, int head_size, int block_size)
{
    for (int64_t i = 0; i < num_tokens; ++i) {
        uint32_t slot = slot_mapping[i];
        if (slot == PAD_SLOT) continue;
        int64_t block = (int64_t)(slot / (uint32_t)block_size);
        int64_t off = (int64_t)(slot % (uint32_t)block_size);
        for (int h = 0; h < num_kv_heads; ++h) {
            int64_t dst = ((block * num_kv_heads + h) * block_size + off) * head_size;
            memcpy(key_cache + dst, key + i * key_stride + (int64_t)h * head_size,
                   sizeof(float) * (size_t)head_size);
            memcpy(value_cache + dst, value + i * value_stride + (int64_t)h * head_size,
                   sizeof(float) * (size_t)head_size);
        }
    }
}

/* The f32 vector of logical token t of sequence s, kv head g. */
static const float *f32_token(const float *cache, const uint32_t *block_tables,
                              int max_blocks_per_seq, int num_kv_heads, int head_size,
                              int block_size, int s, int g, int64_t t)
{
    uint32_t block = block_tables[(int64_t)s * max_blocks_per_seq + t / block_size];
    int64_t off = t % block_size;
    return cache + (((int64_t)block * num_kv_heads + g) * block_size + off) * head_size;
}

/* out[s, h, :] = softmax(scale * q[s,h] . K^T) V over the clamped context of
 * sequence s, K and V read from the f32 caches; rows as in oracle_decode. */
void oracle_decode_f32(double *out, const float *q, const float *key_cache,
                       const float *value_cache, const uint32_t *block_tables,
                       const uint32_t *context_lens, int num_seqs, int num_heads, int num_kv_heads,
                       int head_size, int block_size, int max_blocks_per_seq, double scale,
                       const int32_t *rows, int64_t n_rows)
{
    int64_t n = rows ? n_rows : (int64_t)num_seqs * num_heads;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < n; ++i) {
        int s = rows ? rows[2 * i] : (int)(i / num_heads);
        int h = rows ? rows[2 * i + 1] : (int)(i % num_heads);
        int g = h / (num_heads / num_kv_heads);
        const float *qv = q + ((int64_t)s * num_heads + h) * head_size;
        double *o = out + i * head_size;
        for (int d = 0; d < head_size; ++d) o[d] = 0.0;
        int64_t c = clamped_len(context_lens, s, max_blocks_per_seq, block_size);
        if (c == 0) continue;           /* all zeros */
        double *z = (double *)malloc(sizeof(double) * (size_t)c);
        double m = -INFINITY;
        for (int64_t t = 0; t < c; ++t) {
            const float *k = f32_token(key_cache, block_tables, max_blocks_per_seq, num_kv_heads,
                                       head_size, block_size, s, g, t);
            double dot = 0.0;
            for (int d = 0; d < head_size; ++d) dot += (double)qv[d] * (double)k[d];
            z[t] = scale * dot;
            if (z[t] > m) m = z[t];
        }
        double l = 0.0;
        for (int64_t t = 0; t < c; ++t) {
            double p = exp(z[t] - m);
            l += p;
            const float *v = f32_token(value_cache, block_tables, max_blocks_per_seq, num_kv_heads,
                                       head_size, block_size, s, g, t);
            for (int d = 0; d < head_size; ++d) o[d] += p * (double)v[d];
        }
        for (int d = 0; d < head_size; ++d) o[d] /= l;
        free(z);
    }
}

/* ------------------------------------------------------------------------
 * The contiguous q8 cache with a side scale region ("attention.rs",
 * cherenkov qwen4_exp gpu: the kv_append_q8 dispatch with its parameters
 * row = kv_row, t0, nb and scale_off = kv_q8_side(max_t, kv_row), launched as
 * nb * (kv_row / 32) * 2 subgroups).  The shader is not on the page; the
 * reading taken here:
 *  - one sequence's cache: for each position t < max_t a row of
 *    kv_row = num_kv_heads * head_size int8 codes, 4 per u32 word in
 *    little-endian lanes (kv head major, as the rows arrive), then a side
 *    region of f32 scales, one per 32-element group of a row (one subgroup
 *    per group of K and of V), group j of position t at word
 *    scale_off + t * kv_row / 32 + j, scale_off = max_t * kv_row / 4;
 *  - a group is quantised like a token vector of the paged cache (amax over
 *    its 32 values, codes clamp(round(x * 127/amax)), scale amax/127, 1.0
 *    for an all-zero group);
 *  - S sequences sit back to back, max_t * kv_row / 4 + max_t * kv_row / 32
 *    words apart; a row's slot is s * max_t + t (0xFFFFFFFF skips it).
 * ------------------------------------------------------------------------ */

static int64_t cq_seq_words(int64_t max_t, int64_t kv_row) { return max_t * kv_row / 4 + max_t * kv_row / 32; }

void oracle_cq_append(const float *key, const float *value, uint32_t *key_cache, uint32_t *value_cache,
                      const uint32_t *slot_mapping, int64_t num_tokens, int64_t key_stride,
                      int64_t value_stride, int num_kv_heads, int head_size, int64_t max_t)
{
    const int64_t kv_row = (int64_t)num_kv_heads * head_size;
    const int64_t groups = kv_row / 32;
    const int64_t sw = cq_seq_words(max_t, kv_row);
    uint32_t g[9];
    for (int64_t i = 0; i < num_tokens; ++i) {
        uint32_t slot = slot_mapping[i];
        if (slot == PAD_SLOT) continue;
        const int64_t s = slot / max_t, t = slot % max_t;
        const int64_t codes = s * sw + t * (kv_row / 4);
        const int64_t scales = s * sw + max_t * (kv_row / 4) + t * groups;
        for (int64_t j = 0; j < groups; ++j) {
            oracle_quantize_vector(key + i * key_stride + 32 * j, 32, g);
            memcpy(key_cache + codes + 8 * j, g, 8 * sizeof(uint32_t));
            key_cache[scales + j] = g[8];
            oracle_quantize_vector(value + i * value_stride + 32 * j, 32, g);
            memcpy(value_cache + codes + 8 * j, g, 8 * sizeof(uint32_t));
            value_cache[scales + j] = g[8];
        }
    }
}

/* Dequantised element e (0 <= e < kv_row) of position t of sequence s. */
static double cq_value(const uint32_t *cache, int64_t max_t, int64_t kv_row, int s, int64_t t, int64_t e)
{
    const int64_t base = (int64_t)s * cq_seq_words(max_t, kv_row);
    const uint32_t word = cache[base + t * (kv_row / 4) + e / 4];
    const double scale = (double)float_from_bits(cache[base + max_t * (kv_row / 4) + t * (kv_row / 32) + e / 32]);
    return (double)code_at(word, (int)(e % 4)) * scale;
}

/* out[s, h, :] = softmax(scale * q[s,h] . K^T) V over positions
 * [0, min(context_len, max_t)) of sequence s's contiguous cache, kv head
 * g = h / (num_heads / num_kv_heads) (elements g*head_size ..); rows as in
 * oracle_decode. */
void oracle_cq_decode(double *out, const float *q, const uint32_t *key_cache, const uint32_t *value_cache,
                      const uint32_t *context_lens, int num_seqs, int num_heads, int num_kv_heads,
                      int head_size, int64_t max_t, double scale, const int32_t *rows, int64_t n_rows)
{
    const int64_t kv_row = (int64_t)num_kv_heads * head_size;
    int64_t n = rows ? n_rows : (int64_t)num_seqs * num_heads;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < n; ++i) {
        int s = rows ? rows[2 * i] : (int)(i / num_heads);
        int h = rows ? rows[2 * i + 1] : (int)(i % num_heads);
        int g = h / (num_heads / num_kv_heads);
        const float *qv = q + ((int64_t)s * num_heads + h) * head_size;
        double *o = out + i * head_size;
        for (int d = 0; d < head_size; ++d) o[d] = 0.0;
        int64_t c = context_lens[s];
        if (c > max_t) c = max_t;
        if (c == 0) continue;
        double *z = (double *)malloc(sizeof(double) * (size_t)c);
        double m = -INFINITY;
        for (int64_t t = 0; t < c; ++t) {
            double dot = 0.0;
            for (int d = 0; d < head_size; ++d)
                dot += (double)qv[d] * cq_value(key_cache, max_t, kv_row, s, t, (int64_t)g * head_size + d);
            z[t] = scale * dot;
            if (z[t] > m) m = z[t];
        }
        double l = 0.0;
        for (int64_t t = 0; t < c; ++t) {
            double p = exp(z[t] - m);
            l += p;
            for (int d = 0; d < head_size; ++d)
                o[d] += p * cq_value(value_cache, max_t, kv_row, s, t, (int64_t)g * head_size + d);
        }
        for (int d = 0; d < head_size; ++d) o[d] /= l;
        free(z);
    }
}
