/*
 * pagedkv_oracle.c -- plain, slow, fp64 CPU oracle for paged KV-cache attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
 * the benchmark's CPU-baseline / reference arm may load this library.  It
 * shares no code, header or constant with the CUDA path.
 *
 * Every function below is the plain definition of the operation, written out
 * loop by loop with no blocking, fusion or reordering:
 *
 *  - Scaled dot-product attention  A = softmax(Q K^T / sqrt(d_h) + M) V, with
 *    M_ij = 0 for j <= i and -inf otherwise ("注意力演进与推理流程" (attention
 *    evolution and inference), section 1.1 MHA formula derivation; vLLM concepts
 *    deep dive, section 1, Self-Attention steps 2-4).
 *  - GQA head sharing: query head h reads KV group g = floor(h / G),
 *    G = n_q / n_kv ("注意力演进与推理流程", section 3.1 GQA formula derivation).
 *  - Decode: Attention(q_t, K_<=t, V_<=t) needs no causal mask; the new token's
 *    K/V is written at position cache_len before the read ("LLM 推理全过程的维度
 *    变化与核心公式", section "Decode 阶段维度流转").
 *  - Paging: K/V live in fixed-size physical blocks found through a block table;
 *    the attention formula is unchanged, only the layout differs (same page,
 *    section "KV Cache 的形状与增长"; vLLM concepts deep dive, section 1, last
 *    paragraph: kernels take a block table and a slot mapping).
 *  - Flash-Decoding: split cache_len into parts, then a log-sum-exp reduction;
 *    the softmax is the same, computed in two stages (same walkthrough page,
 *    section "工程优化怎么嵌进公式", Flash Decoding paragraph).
 *  - Chunked prefill: the chunk's queries at absolute positions c + i see keys
 *    j <= c + i; the formula is unchanged ("注意力演进与推理流程", 变革 3;
 *    walkthrough page, Chunked Prefill paragraph).
 *  - Per-token KV size 2 * L * n_kv * d * dtype_size (vLLM concepts deep dive,
 *    section 1, KV cache size formula).
 *  - Sliding window: only the most recent W tokens' K and V are kept, so a
 *    query at position p sees keys p - W < j <= p (walkthrough page, section
 *    "KV Cache 的形状与增长", Sliding Window Attention item).
 *  - FP8 KV cache: K and V quantised per token (and per KV head) to 8-bit
 *    floats with a scale each, halving the cache (same section, INT8 / FP8 KV
 *    Cache item; xinc.fun archive 233, section 7: the error depends on the
 *    group size and the scaling).  Format: E4M3 (1 sign, 4 exponent bits with
 *    bias 7, 3 mantissa bits, largest finite 448, no infinities).
 *  - Block copy at a branch: sequences sharing a prefix (or parallel
 *    candidates) reference the same physical blocks until they branch, where a
 *    new block is allocated (xinc.fun archive 233, section 6).
 *
 * Data layout (readings; the pages fix none):
 *   bf16 values are passed as their 16-bit patterns (uint16_t) and widened
 *   exactly to double.  FP8 caches hold E4M3 codes (uint8_t) in the same
 *   [num_blocks][n_kv][block_size][head_dim] layout, with fp32 scales
 *   [num_blocks][n_kv][block_size] (one per token and KV head).
 *   k_cache, v_cache : [num_blocks][n_kv][block_size][head_dim]
 *   block_tables     : [num_seqs][max_blocks]
 *   q                : [total_q_rows][n_q][head_dim]; cu_q_lens[num_seqs+1]
 *   out              : [total_q_rows][n_q][head_dim] (double)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ---- sizes and index rules ------------------------------------------------ */

/* Bytes of K plus V that one token occupies over `layers` layers. */
int64_t oracle_kv_bytes_per_token(int64_t layers, int64_t n_kv, int64_t head_dim, int64_t dtype_size)
{
    return 2 * layers * n_kv * head_dim * dtype_size;
}

/* KV group read by query head h: floor(h / G) with G = n_q / n_kv. */
int32_t oracle_kv_group(int32_t h, int32_t n_q, int32_t n_kv)
{
    int32_t G = n_q / n_kv;
    return h / G;
}

/* Physical slot of logical token `pos` of a sequence: table[pos / bs] * bs + pos % bs. */
int64_t oracle_slot_of(const int32_t *table_row, int32_t pos, int32_t block_size)
{
    return (int64_t)table_row[pos / block_size] * block_size + pos % block_size;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ---- cache write ------------------------------------------------------------
 * For each new token t and KV head h: the row key[t][h][:] is stored at
 * physical slot s = slot_mapping[t], i.e. block s / block_size, offset
 * s % block_size.  Negative slots mark padding and are skipped.  Slots at or
 * past num_blocks * block_size are skipped as well (undefined input).
 */
void oracle_kv_reshape_and_cache(const uint16_t *key, const uint16_t *value,
                                 uint16_t *k_cache, uint16_t *v_cache,
                                 const int32_t *slot_mapping, int32_t num_tokens,
                                 int32_t num_blocks, int32_t block_size,
                                 int32_t n_kv, int32_t head_dim)
{
    for (int32_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0 || slot >= (int64_t)num_blocks * block_size)
            continue;
        int64_t blk = slot / block_size;
        int64_t off = slot % block_size;
        for (int32_t h = 0; h < n_kv; ++h) {
            for (int32_t k = 0; k < head_dim; ++k) {
                int64_t src = ((int64_t)t * n_kv + h) * head_dim + k;
                int64_t dst = ((blk * n_kv + h) * block_size + off) * head_dim + k;
                k_cache[dst] = key[src];
                v_cache[dst] = value[src];
            }
        }
    }
}

/* ---- attention --------------------------------------------------------------
 * For each sequence b with q_len = cu_q_lens[b+1] - cu_q_lens[b] query rows and
 * context length ctx = context_lens[b] (which already counts the q_len new
 * tokens), query row r sits at absolute position p = ctx - q_len + r and sees
 * the keys j = 0 .. p (causal rule; for decode q_len = 1 and p = ctx - 1, so
 * every cached key is visible and no mask applies).
 *
 *   s_j   = scale * sum_k q[r][h][k] * K_b[j][g(h)][k]
 *   w_j   = exp(s_j - max_i s_i) / sum_i exp(s_i - max_i s_i)
 *   out   = sum_j w_j * V_b[j][g(h)]
 *   lse   = max_i s_i + log(sum_i exp(s_i - max_i s_i))      (optional)
 *
 * K_b[j] is read through the block table: block block_tables[b][j / bs],
 * offset j % bs.  Returns 0, or -1 on a bad argument.
 */
/* A cache holds bf16 values, or E4M3 codes with one fp32 scale per (slot, head). */
typedef struct {
    const void *data;
    const float *scale; /* NULL: bf16 cache */
} cache_ref;

double oracle_e4m3_decode(uint8_t c);

/* Element k of the row at (block blk, head g, offset off), as a real number. */
static double cache_elem(cache_ref c, int64_t blk, int32_t off, int32_t g, int32_t n_kv, int32_t bs,
                         int32_t d, int32_t k)
{
    const int64_t row = (blk * n_kv + g) * bs + off;
    if (!c.scale)
        return bf16_to_double(((const uint16_t *)c.data)[row * d + k]);
    return oracle_e4m3_decode(((const uint8_t *)c.data)[row * d + k]) * (double)c.scale[row];
}

static double key_dot(const uint16_t *qrow, cache_ref kc, int64_t blk, int32_t off, int32_t g, int32_t n_kv,
                      int32_t bs, int32_t d)
{
    double acc = 0.0;
    for (int32_t k = 0; k < d; ++k)
        acc += bf16_to_double(qrow[k]) * cache_elem(kc, blk, off, g, n_kv, bs, d, k);
    return acc;
}

static int paged_attention(double *out, double *lse, const uint16_t *q, const int32_t *cu_q_lens,
                           int32_t num_seqs, int32_t n_q, cache_ref kc, cache_ref vc,
                           const int32_t *block_tables, int32_t max_blocks, const int32_t *context_lens,
                           int32_t num_blocks, int32_t n_kv, int32_t block_size, int32_t head_dim,
                           double scale, int32_t window)
{
    if (n_kv <= 0 || n_q % n_kv != 0 || num_seqs < 0)
        return -1;
    const int32_t G = n_q / n_kv;
    const int32_t total_rows = cu_q_lens[num_seqs];
    /* row -> sequence */
    int32_t *row_seq = (int32_t *)malloc(sizeof(int32_t) * (size_t)(total_rows > 0 ? total_rows : 1));
    for (int32_t b = 0; b < num_seqs; ++b) {
        int32_t q_len = cu_q_lens[b + 1] - cu_q_lens[b];
        int32_t ctx = context_lens[b];
        if (q_len < 0 || ctx < q_len || ctx > max_blocks * block_size) {
            free(row_seq);
            return -1;
        }
        for (int32_t r = cu_q_lens[b]; r < cu_q_lens[b + 1]; ++r)
            row_seq[r] = b;
    }
    for (int32_t b = 0; b < num_seqs; ++b)
        for (int32_t j = 0; j < (context_lens[b] + block_size - 1) / block_size; ++j) {
            int32_t blk = block_tables[(int64_t)b * max_blocks + j];
            if (blk < 0 || blk >= num_blocks) {
                free(row_seq);
                return -1;
            }
        }

    const int64_t work = (int64_t)total_rows * n_q;
    int status = 0;
#pragma omp parallel
    {
        int32_t cap = 0;
        double *s = NULL;
#pragma omp for schedule(dynamic, 1)
        for (int64_t item = 0; item < work; ++item) {
            const int32_t row = (int32_t)(item / n_q);
            const int32_t h = (int32_t)(item % n_q);
            const int32_t b = row_seq[row];
            const int32_t q_len = cu_q_lens[b + 1] - cu_q_lens[b];
            const int32_t ctx = context_lens[b];
            const int32_t pos = ctx - q_len + (row - cu_q_lens[b]);
            const int32_t nvis = pos + 1; /* keys 0..pos */
            /* sliding window: keys j0..pos only */
            const int32_t j0 = (window > 0 && pos + 1 > window) ? pos + 1 - window : 0;
            const int32_t g = h / G;
            const int32_t *trow = block_tables + (int64_t)b * max_blocks;
            const uint16_t *qrow = q + ((int64_t)row * n_q + h) * head_dim;
            double *orow = out + ((int64_t)row * n_q + h) * head_dim;
            if (nvis > cap) {
                free(s);
                cap = nvis;
                s = (double *)malloc(sizeof(double) * (size_t)cap);
            }
            double m = -INFINITY;
            for (int32_t j = j0; j < nvis; ++j) {
                s[j] = scale * key_dot(qrow, kc, trow[j / block_size], j % block_size, g, n_kv, block_size,
                                       head_dim);
                if (s[j] > m)
                    m = s[j];
            }
            double l = 0.0;
            for (int32_t j = j0; j < nvis; ++j) {
                s[j] = exp(s[j] - m);
                l += s[j];
            }
            for (int32_t k = 0; k < head_dim; ++k)
                orow[k] = 0.0;
            for (int32_t j = j0; j < nvis; ++j) {
                const double w = s[j] / l;
                for (int32_t k = 0; k < head_dim; ++k)
                    orow[k] += w * cache_elem(vc, trow[j / block_size], j % block_size, g, n_kv, block_size,
                                              head_dim, k);
            }
            if (lse)
                lse[(int64_t)row * n_q + h] = m + log(l);
        }
        free(s);
    }
    free(row_seq);
    return status;
}

int oracle_paged_attention(double *out, double *lse, const uint16_t *q, const int32_t *cu_q_lens,
                           int32_t num_seqs, int32_t n_q, const uint16_t *k_cache,
                           const uint16_t *v_cache, const int32_t *block_tables, int32_t max_blocks,
                           const int32_t *context_lens, int32_t num_blocks, int32_t n_kv,
                           int32_t block_size, int32_t head_dim, double scale, int32_t window)
{
    const cache_ref kc = {k_cache, NULL}, vc = {v_cache, NULL};
    return paged_attention(out, lse, q, cu_q_lens, num_seqs, n_q, kc, vc, block_tables, max_blocks,
                           context_lens, num_blocks, n_kv, block_size, head_dim, scale, window);
}

/* The same attention over an FP8 cache: K_j = decode(code) * k_scale[slot][head]. */
int oracle_paged_attention_fp8(double *out, double *lse, const uint16_t *q, const int32_t *cu_q_lens,
                               int32_t num_seqs, int32_t n_q, const uint8_t *k_cache, const uint8_t *v_cache,
                               const float *k_scale, const float *v_scale, const int32_t *block_tables,
                               int32_t max_blocks, const int32_t *context_lens, int32_t num_blocks,
                               int32_t n_kv, int32_t block_size, int32_t head_dim, double scale,
                               int32_t window)
{
    const cache_ref kc = {k_cache, k_scale}, vc = {v_cache, v_scale};
    return paged_attention(out, lse, q, cu_q_lens, num_seqs, n_q, kc, vc, block_tables, max_blocks,
                           context_lens, num_blocks, n_kv, block_size, head_dim, scale, window);
}

/* ---- Flash-Decoding partials and their log-sum-exp merge --------------------
 * Decode only (one query row per sequence).  Part p of sequence b covers the
 * keys [p * part_tokens, min((p + 1) * part_tokens, ctx)).  For each (b, h, p):
 *   m_p = max_j s_j,  l_p = sum_j exp(s_j - m_p),  o_p = sum_j exp(s_j - m_p) V[j]
 * Parts that hold no key get m_p = -inf, l_p = 0, o_p = 0.
 * Layouts: m, l [num_seqs][n_q][max_parts]; o [num_seqs][n_q][max_parts][head_dim].
 */
int oracle_decode_partials(double *m_out, double *l_out, double *o_out, const uint16_t *q,
                           int32_t num_seqs, int32_t n_q, const uint16_t *k_cache,
                           const uint16_t *v_cache, const int32_t *block_tables, int32_t max_blocks,
                           const int32_t *context_lens, int32_t n_kv, int32_t block_size,
                           int32_t head_dim, double scale, int32_t part_tokens, int32_t max_parts)
{
    if (n_kv <= 0 || n_q % n_kv != 0 || part_tokens <= 0)
        return -1;
    const int32_t G = n_q / n_kv;
    const cache_ref kc = {k_cache, NULL};
    for (int32_t b = 0; b < num_seqs; ++b)
        if ((context_lens[b] + part_tokens - 1) / part_tokens > max_parts)
            return -1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t item = 0; item < (int64_t)num_seqs * n_q; ++item) {
        const int32_t b = (int32_t)(item / n_q), h = (int32_t)(item % n_q), g = h / G;
        const int32_t ctx = context_lens[b];
        const int32_t *trow = block_tables + (int64_t)b * max_blocks;
        const uint16_t *qrow = q + ((int64_t)b * n_q + h) * head_dim;
        for (int32_t p = 0; p < max_parts; ++p) {
            const int64_t pi = ((int64_t)b * n_q + h) * max_parts + p;
            double *o = o_out + pi * head_dim;
            for (int32_t k = 0; k < head_dim; ++k)
                o[k] = 0.0;
            const int32_t j0 = p * part_tokens;
            const int32_t j1 = (j0 + part_tokens < ctx) ? j0 + part_tokens : ctx;
            double m = -INFINITY, l = 0.0;
            for (int32_t j = j0; j < j1; ++j) {
                double sj = scale * key_dot(qrow, kc, trow[j / block_size], j % block_size, g, n_kv,
                                            block_size, head_dim);
                if (sj > m)
                    m = sj;
            }
            for (int32_t j = j0; j < j1; ++j) {
                double e = exp(scale * key_dot(qrow, kc, trow[j / block_size], j % block_size, g, n_kv,
                                               block_size, head_dim) -
                               m);
                const uint16_t *vrow =
                    v_cache + (((int64_t)trow[j / block_size] * n_kv + g) * block_size + j % block_size) *
                                  (int64_t)head_dim;
                l += e;
                for (int32_t k = 0; k < head_dim; ++k)
                    o[k] += e * bf16_to_double(vrow[k]);
            }
            m_out[pi] = m;
            l_out[pi] = l;
        }
    }
    return 0;
}

/* Log-sum-exp merge of partials:
 *   M = max_p m_p;  out = sum_p exp(m_p - M) o_p / sum_p exp(m_p - M) l_p
 * Parts with m_p = -inf contribute nothing.
 */
void oracle_lse_merge(double *out, const double *m_in, const double *l_in, const double *o_in,
                      int32_t rows, int32_t max_parts, int32_t head_dim)
{
    for (int32_t r = 0; r < rows; ++r) {
        double M = -INFINITY;
        for (int32_t p = 0; p < max_parts; ++p)
            if (m_in[(int64_t)r * max_parts + p] > M)
                M = m_in[(int64_t)r * max_parts + p];
        double den = 0.0;
        double *o = out + (int64_t)r * head_dim;
        for (int32_t k = 0; k < head_dim; ++k)
            o[k] = 0.0;
        for (int32_t p = 0; p < max_parts; ++p) {
            const double mp = m_in[(int64_t)r * max_parts + p];
            if (mp == -INFINITY)
                continue;
            const double w = exp(mp - M);
            den += w * l_in[(int64_t)r * max_parts + p];
            for (int32_t k = 0; k < head_dim; ++k)
                o[k] += w * o_in[((int64_t)r * max_parts + p) * head_dim + k];
        }
        for (int32_t k = 0; k < head_dim; ++k)
            o[k] /= den;
    }
}

/* ---- FP8 (E4M3) codes -------------------------------------------------------
 * Code layout s.eeee.mmm, exponent bias 7.  e > 0: (-1)^s 2^(e-7) (1 + m/8);
 * e = 0: (-1)^s 2^-6 (m/8).  The two codes s.1111.111 are NaN; there are no
 * infinities, so the largest finite magnitude is 2^8 * 1.75 = 448.
 */
double oracle_e4m3_decode(uint8_t c)
{
    const int sgn = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7)
        return NAN;
    const double mag = e ? ldexp(1.0 + m / 8.0, e - 7) : ldexp(m / 8.0, -6);
    return sgn ? -mag : mag;
}

/* Nearest E4M3 value to x, ties to the even code; magnitudes past 448 saturate
 * to 448 and NaN stays NaN.  Works from the definition above: the spacing of
 * representable values is 2^(e-10) in binade [2^(e-7), 2^(e-6)) and 2^-9 below
 * 2^-6. */
uint8_t oracle_e4m3_encode(float x)
{
    if (isnan(x))
        return 0x7F;
    const uint8_t sgn = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0)
        return sgn | 0x7E;
    int e2;
    frexp(a, &e2); /* a = f * 2^e2, f in [0.5, 1): binade exponent e2 - 1 */
    int be = e2 - 1;
    if (a == 0.0 || be < -6)
        be = -6; /* subnormal spacing 2^-9 below 2^-6 */
    const double step = ldexp(1.0, be - 3);
    double n = floor(a / step);
    const double rem = a / step - n;
    if (rem > 0.5 || (rem == 0.5 && fmod(n, 2.0) == 1.0))
        n += 1.0; /* n * step is now the rounded magnitude (exact in double) */
    const double r = n * step;
    if (r >= 448.0)
        return sgn | 0x7E;
    if (r < ldexp(1.0, -6)) /* subnormal: m = r / 2^-9 */
        return sgn | (uint8_t)(r / ldexp(1.0, -9));
    int e3;
    frexp(r, &e3);
    const int e = e3 - 1 + 7; /* biased exponent */
    const int m = (int)((r / ldexp(1.0, e3 - 1) - 1.0) * 8.0);
    return sgn | (uint8_t)(e << 3) | (uint8_t)m;
}

/* ---- FP8 cache write ----------------------------------------------------------
 * One scale per token and KV head (per-token quantisation): with a = max_k |x_k|
 * over the head's 128 values (fp32, exact), a' = max(a, 2^-100) so the scale
 * stays a normal number,
 *     inv   = 448 / a'          (fp32, round to nearest)
 *     code  = E4M3(x_k * inv)   (fp32 product, then nearest-even code)
 *     scale = a' / 448          (fp32, round to nearest)
 * and x_k is recovered as decode(code) * scale.  Every step is a single
 * correctly rounded fp32 operation, so the codes are exactly reproducible.
 * Slots as in oracle_kv_reshape_and_cache.
 */
static void quantize_row(const uint16_t *src, uint8_t *codes, float *scale, int32_t d)
{
    float a = 0.0f;
    for (int32_t k = 0; k < d; ++k) {
        const float v = (float)fabs(bf16_to_double(src[k]));
        if (v > a)
            a = v;
    }
    const float floor_a = 0x1p-100f;
    if (a < floor_a)
        a = floor_a;
    volatile float inv = 448.0f / a;
    for (int32_t k = 0; k < d; ++k) {
        volatile float y = (float)bf16_to_double(src[k]) * inv;
        codes[k] = oracle_e4m3_encode(y);
    }
    volatile float sc = a / 448.0f;
    *scale = sc;
}

void oracle_kv_reshape_and_cache_fp8(const uint16_t *key, const uint16_t *value, uint8_t *k_cache,
                                     uint8_t *v_cache, float *k_scale, float *v_scale,
                                     const int32_t *slot_mapping, int32_t num_tokens, int32_t num_blocks,
                                     int32_t block_size, int32_t n_kv, int32_t head_dim)
{
    /* Tokens are independent (slots are distinct), so they may run in parallel. */
#pragma omp parallel for schedule(static)
    for (int32_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0 || slot >= (int64_t)num_blocks * block_size)
            continue;
        int64_t blk = slot / block_size;
        int64_t off = slot % block_size;
        for (int32_t h = 0; h < n_kv; ++h) {
            const int64_t src = ((int64_t)t * n_kv + h) * head_dim;
            const int64_t row = (blk * n_kv + h) * block_size + off;
            quantize_row(key + src, k_cache + row * head_dim, &k_scale[row], head_dim);
            quantize_row(value + src, v_cache + row * head_dim, &v_scale[row], head_dim);
        }
    }
}

/* ---- block copy at a branch ------------------------------------------------------
 * pairs[2i] -> pairs[2i+1], in order, every byte of the block (all heads and
 * slots; call once per K cache, V cache and scale array).  block_bytes is the
 * size of one block of that array. */
void oracle_copy_blocks(uint8_t *cache, const int32_t *pairs, int32_t n_pairs, int64_t block_bytes)
{
    for (int32_t i = 0; i < n_pairs; ++i) {
        const int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        for (int64_t b = 0; b < block_bytes; ++b)
            cache[dst * block_bytes + b] = cache[src * block_bytes + b];
    }
}
