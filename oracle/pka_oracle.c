/*
 * pka_oracle.c -- TEST INFRASTRUCTURE, not part of the product.
 *
 * A plain, slow, obviously-correct fp64 CPU statement of what the paged-KV
 * attention forward computes.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library; the CUDA path never links,
 * calls or includes anything from here, and nothing here comes from the CUDA
 * path.  Every bf16 input is widened exactly to double; every sum is a plain
 * left-to-right loop in double precision.
 *
 * Sources (the three web pages on vLLM's attention backends):
 *  [FA/FI]   "FlashAttention y FlashInfer: los dos grandes backends de atencion
 *            en GPU" (vllm-arch-zh.pages.dev/es/attention/flash)
 *  [blog]    "El especialista del plato estrella: el backend de atencion de
 *            vLLM" (blog.lo0.es, cascade-attention tag)
 *  [backend] "AttentionBackend: capa de abstraccion de backends de atencion"
 *            (vllm-arch-zh.pages.dev/es/attention/backend)
 *
 * Readings taken where the pages are silent (each is listed with its reason
 * in the design notes of the repository):
 *  - causal alignment is bottom-right: query i of a sequence with prior
 *    context c sees keys 0..c+i;
 *  - seq_lens counts the whole KV length including this step's tokens;
 *  - query head h reads kv head h / (num_heads / num_kv_heads);
 *  - the log-sum-exp is in natural-log units;
 *  - a key range with no admitted key has lse = -inf and output 0, and is the
 *    identity of the merge.
 *
 * Build flag ORACLE_MUTANT=n plants one deliberate mistake (used only by the
 * test that proves the pins catch such mistakes); 0 (default) is the oracle.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

/* Exact value of a bf16 bit pattern: bf16 is the upper half of an IEEE
 * binary32, so shifting the 16 bits up gives the float exactly. */
static double bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Row (block, kv, offset, head) of the pool shaped
 * (num_blocks, 2, block_size, num_kv_heads, head_size), K at kv=0, V at kv=1
 * -- [FA/FI] "Flujo de datos", get_kv_cache_shape. */
static const uint16_t *pool_row(const uint16_t *cache, int64_t block, int64_t kv,
                                int64_t offset, int64_t head, int64_t block_size,
                                int64_t num_kv_heads, int64_t head_size)
{
    int64_t row = ((block * 2 + kv) * block_size + offset) * num_kv_heads + head;
    return cache + row * head_size;
}

/*
 * FP8 E4M3 (the OCP 8-bit floating-point format: 1 sign bit, 4 exponent bits
 * with bias 7, 3 mantissa bits; no infinities; S.1111.111 is NaN; largest
 * finite 448 = 1.75 * 2^8; subnormals m/8 * 2^-6).  The pages name an fp8
 * e4m3 KV cache ([FA/FI] "Resumen en una frase" and "Limites y fallos":
 * fp8 / fp8_e4m3 KV cache) without a quantisation rule; the reading taken:
 * one fp32 scale per tensor (k_scale for K, v_scale for V), code =
 * e4m3(x / scale) with x / scale computed in fp32, rounded to nearest
 * (ties to the even code) and saturated to +-448; value = code * scale.
 */
static double e4m3_value(uint8_t c)
{
    int sign = c >> 7, ex = (c >> 3) & 15, man = c & 7;
    double v;
    if (ex == 15 && man == 7)
        return NAN;
#if ORACLE_MUTANT == 13
    if (ex == 0)
        v = ldexp((double)man, -10);
#else
    if (ex == 0)
        v = ldexp((double)man, -9); /* subnormal: man/8 * 2^-6 */
#endif
#if ORACLE_MUTANT == 15
    else
        v = ldexp(8.0 + man, ex - 11);
#else
    else
        v = ldexp(8.0 + man, ex - 10); /* (1 + man/8) * 2^(ex-7) */
#endif
    return sign ? -v : v;
}

/* Nearest e4m3 code to the float y: the 127 non-negative finite codes in
 * increasing order are scanned for the closest value; a tie goes to the code
 * whose last mantissa bit is 0; |y| above 448 saturates to 448; the sign is
 * kept (also for zero); NaN gives 0x7f.  mag[c] = e4m3_value(c) for the
 * codes 0..0x7e, filled once by the caller. */
static uint8_t e4m3_encode(float y, const double *mag)
{
    if (y != y)
        return 0x7f;
    int neg = signbit(y) != 0;
    double a = fabs((double)y);
    uint8_t best = 0;
    if (a >= 448.0) {
#if ORACLE_MUTANT == 11
        best = 0x7f;
#else
        best = 0x7e;
#endif
    } else {
        double best_d = a; /* distance to code 0 */
        for (int c = 1; c <= 0x7e; ++c) {
            double d = fabs(mag[c] - a);
#if ORACLE_MUTANT == 10
            if (d <= best_d) {
#else
            if (d < best_d || (d == best_d && (c & 1) == 0)) {
#endif
                best = (uint8_t)c;
                best_d = d;
            }
        }
    }
    return (uint8_t)(best | (neg ? 0x80 : 0));
}

/* Codes of x[i] / scale (fp32 division) for n values (bf16 bit patterns). */
void oracle_quantize_e4m3(const uint16_t *x, int64_t n, float scale, uint8_t *out)
{
    double mag[0x7f];
    for (int c = 0; c < 0x7f; ++c)
        mag[c] = e4m3_value((uint8_t)c);
    for (int64_t i = 0; i < n; ++i) {
        float xf = (float)bf16_value(x[i]);
#if ORACLE_MUTANT == 12
        volatile float y = xf * scale;
#else
        volatile float y = xf / scale; /* fp32 division, as stored */
#endif
        out[i] = e4m3_encode(y, mag);
    }
}

double oracle_e4m3_value(uint8_t c) { return e4m3_value(c); }

/* Element e of row (block, kv, offset, head) of a pool in bf16 (codes8 ==
 * NULL) or e4m3 with per-tensor scales. */
typedef struct {
    const uint16_t *bf16;
    const uint8_t *codes8;
    double k_scale, v_scale;
    int64_t block_size, num_kv_heads, head_size;
} pool_view;

static double pool_elem(const pool_view *pv, int64_t block, int64_t kv, int64_t offset,
                        int64_t head, int64_t e)
{
    int64_t row = ((block * 2 + kv) * pv->block_size + offset) * pv->num_kv_heads + head;
#if ORACLE_MUTANT == 14
    if (pv->codes8)
        return e4m3_value(pv->codes8[row * pv->head_size + e]) * (kv ? pv->k_scale : pv->v_scale);
#else
    if (pv->codes8)
        return e4m3_value(pv->codes8[row * pv->head_size + e]) * (kv ? pv->v_scale : pv->k_scale);
#endif
    return bf16_value(pv->bf16[row * pv->head_size + e]);
}

/*
 * reshape_and_cache: for every new token t with slot = slot_mapping[t] >= 0,
 * copy key[t] into the K slot (slot / block_size, slot % block_size) of the
 * pool and value[t] into the V slot, byte for byte.  slot < 0 is padding and
 * is skipped.  The cache-update op is named in [FA/FI] "Responsabilidades"
 * (unified_kv_cache_update); slot = block * block_size + offset is the
 * addressing the pool shape implies.
 * Returns 0, or -1 when a slot lies outside the pool (nothing after it is
 * written).
 */
int oracle_reshape_and_cache(const uint16_t *key, const uint16_t *value, uint16_t *cache,
                             const int64_t *slot_mapping, int64_t num_tokens,
                             int64_t num_kv_heads, int64_t head_size, int64_t block_size,
                             int64_t num_blocks)
{
    int64_t row_elems = num_kv_heads * head_size;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= num_blocks * block_size)
            return -1;
        int64_t block = slot / block_size;
        int64_t offset = slot % block_size;
#if ORACLE_MUTANT == 9
        offset = (offset + 1) % block_size; /* planted: off-by-one slot */
#endif
        for (int64_t h = 0; h < num_kv_heads; ++h) {
            uint16_t *kd = (uint16_t *)pool_row(cache, block, 0, offset, h, block_size,
                                                num_kv_heads, head_size);
            uint16_t *vd = (uint16_t *)pool_row(cache, block, 1, offset, h, block_size,
                                                num_kv_heads, head_size);
            memcpy(kd, key + t * row_elems + h * head_size, (size_t)head_size * 2);
            memcpy(vd, value + t * row_elems + h * head_size, (size_t)head_size * 2);
        }
    }
    return 0;
}

/*
 * One query row q (head_size bf16) of sequence `bt_row` against the keys
 * j in [lo, hi) of that sequence, read through its block table
 * ([blog] "Como lee el backend el KV paginado": the kernel gathers the
 * physical blocks named by the block table):
 *     x_j = scale * <q, K_j>
 *     lse = m + ln sum_j exp(x_j - m),  m = max_j x_j
 *     out = sum_j exp(x_j - lse) * V_j
 * x is scratch of at least hi-lo doubles.
 * Returns 0, or -1 when a block-table entry it needs is outside the pool.
 */
static int attend_row(const uint16_t *q, const pool_view *pv, const int32_t *bt_row,
                      int64_t lo, int64_t hi, int64_t kv_head, int64_t head_size,
                      int64_t block_size, int64_t num_blocks, double scale, double *x,
                      double *out, double *lse)
{
    for (int64_t e = 0; e < head_size; ++e)
        out[e] = 0.0;
    if (hi <= lo) {
        *lse = -INFINITY;
        return 0;
    }
    double m = -INFINITY;
    for (int64_t j = lo; j < hi; ++j) {
        int64_t block = bt_row[j / block_size];
        if (block < 0 || block >= num_blocks)
            return -1;
#if ORACLE_MUTANT == 5
        int64_t k_kv = 1, k_off = j % block_size; /* planted: V used as K */
#elif ORACLE_MUTANT == 6
        int64_t k_kv = 0, k_off = (j + 1) % block_size; /* planted: wrong in-page offset */
#else
        int64_t k_kv = 0, k_off = j % block_size;
#endif
        double dot = 0.0;
        for (int64_t e = 0; e < head_size; ++e)
            dot += bf16_value(q[e]) * pool_elem(pv, block, k_kv, k_off, kv_head, e);
#if ORACLE_MUTANT == 1
        x[j - lo] = dot; /* planted: scale dropped */
#else
        x[j - lo] = scale * dot;
#endif
        if (x[j - lo] > m)
            m = x[j - lo];
    }
    double sum = 0.0;
    for (int64_t j = lo; j < hi; ++j)
#if ORACLE_MUTANT == 2
        sum += exp(m - x[j - lo]); /* planted: wrong sign */
#else
        sum += exp(x[j - lo] - m);
#endif
#if ORACLE_MUTANT == 7
    double l = m + log2(sum); /* planted: wrong log base */
#else
    double l = m + log(sum);
#endif
    for (int64_t j = lo; j < hi; ++j) {
        int64_t block = bt_row[j / block_size];
        double p = exp(x[j - lo] - l);
        for (int64_t e = 0; e < head_size; ++e)
            out[e] += p * pool_elem(pv, block, 1, j % block_size, kv_head, e);
    }
    *lse = l;
    return 0;
}

/* Sequence that owns token t: the s with qsl[s] <= t < qsl[s+1]
 * (query_start_loc as in [backend] "Archivos clave", CommonAttentionMetadata). */
static int64_t owner_seq(const int32_t *qsl, int64_t num_seqs, int64_t t)
{
    for (int64_t s = 0; s < num_seqs; ++s)
        if (t >= qsl[s] && t < qsl[s + 1])
            return s;
    return -1;
}

/*
 * Paged attention forward over the mixed batch ([FA/FI] "Flujo de datos":
 * query [num_tokens, num_heads, head_size]; [blog] "El truco del scheduler":
 * per sequence, how many queries it brings and how much KV it reads).
 *
 * For sequence s: q_s = qsl[s+1]-qsl[s] query tokens, L_s = seq_lens[s] keys,
 * prior context c_s = L_s - q_s.  Query i of s (token t = qsl[s]+i), head h,
 * reads kv head h / (num_heads/num_kv_heads) and admits key j iff
 *     key_lo <= j < min(key_hi, L_s)   and   (!causal || j <= c_s + i).
 * key_hi < 0 means "no upper restriction".  key_lo/key_hi let the tests state
 * split-KV and prefix/suffix passes as plain sub-ranges of the same sum.
 *
 * rows == NULL: every (token, head) row, out[(t*H+h)*D + e], lse[t*H+h].
 * rows != NULL: only the listed rows r = t*H + h, out[k*D + e], lse[k].
 * Returns 0, -1 for a block id outside the pool, -2 for bad metadata,
 * -3 for an allocation failure.
 */
static int paged_attention_view(const uint16_t *query, const pool_view *pv,
                                const int32_t *qsl, const int32_t *seq_lens,
                                const int32_t *block_table, int64_t block_table_stride,
                                int64_t num_seqs, int64_t num_heads, int64_t num_kv_heads,
                                int64_t head_size, int64_t block_size, int64_t num_blocks,
                                double scale, int causal, int64_t key_lo, int64_t key_hi,
                                const int64_t *rows, int64_t num_rows, double *out, double *lse)
{
    if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0)
        return -2;
    int64_t group = num_heads / num_kv_heads;
    int64_t num_tokens = qsl[num_seqs];
    int64_t total = rows ? num_rows : num_tokens * num_heads;
    int64_t max_len = 1;
    for (int64_t s = 0; s < num_seqs; ++s)
        if (seq_lens[s] > max_len)
            max_len = seq_lens[s];
    double *x = (double *)malloc((size_t)max_len * sizeof(double));
    if (!x)
        return -3;
    int rc = 0;
    for (int64_t k = 0; k < total && rc == 0; ++k) {
        int64_t r = rows ? rows[k] : k;
        int64_t t = r / num_heads;
        int64_t h = r % num_heads;
        int64_t s = owner_seq(qsl, num_seqs, t);
        if (s < 0) {
            rc = -2;
            break;
        }
        int64_t q_len = qsl[s + 1] - qsl[s];
        int64_t ctx = seq_lens[s] - q_len;
        if (ctx < 0) {
            rc = -2;
            break;
        }
        int64_t i = t - qsl[s];
        int64_t lo = key_lo > 0 ? key_lo : 0;
        int64_t hi = seq_lens[s];
        if (key_hi >= 0 && key_hi < hi)
            hi = key_hi;
#if ORACLE_MUTANT == 4
        if (causal && ctx + i < hi)
            hi = ctx + i; /* planted: diagonal key dropped */
#else
        if (causal && ctx + i + 1 < hi)
            hi = ctx + i + 1;
#endif
#if ORACLE_MUTANT == 3
        int64_t kv_head = h % num_kv_heads; /* planted: wrong GQA map */
#else
        int64_t kv_head = h / group;
#endif
        rc = attend_row(query + (t * num_heads + h) * head_size, pv,
                        block_table + s * block_table_stride, lo, hi, kv_head, head_size,
                        block_size, num_blocks, scale, x, out + k * head_size, lse + k);
    }
    free(x);
    return rc;
}

int oracle_paged_attention(const uint16_t *query, const uint16_t *cache, const int32_t *qsl,
                           const int32_t *seq_lens, const int32_t *block_table,
                           int64_t block_table_stride, int64_t num_seqs, int64_t num_heads,
                           int64_t num_kv_heads, int64_t head_size, int64_t block_size,
                           int64_t num_blocks, double scale, int causal, int64_t key_lo,
                           int64_t key_hi, const int64_t *rows, int64_t num_rows, double *out,
                           double *lse)
{
    pool_view pv = {cache, NULL, 1.0, 1.0, block_size, num_kv_heads, head_size};
    return paged_attention_view(query, &pv, qsl, seq_lens, block_table, block_table_stride,
                                num_seqs, num_heads, num_kv_heads, head_size, block_size,
                                num_blocks, scale, causal, key_lo, key_hi, rows, num_rows, out,
                                lse);
}

/*
 * oracle_paged_attention over an e4m3 pool (one byte per element, same
 * [num_blocks, 2, block_size, num_kv_heads, head_size] shape): K element
 * value = e4m3 code * k_scale, V element value = code * v_scale.
 */
int oracle_paged_attention_fp8(const uint16_t *query, const uint8_t *cache8, double k_scale,
                               double v_scale, const int32_t *qsl, const int32_t *seq_lens,
                               const int32_t *block_table, int64_t block_table_stride,
                               int64_t num_seqs, int64_t num_heads, int64_t num_kv_heads,
                               int64_t head_size, int64_t block_size, int64_t num_blocks,
                               double scale, int causal, const int64_t *rows, int64_t num_rows,
                               double *out, double *lse)
{
    pool_view pv = {NULL, cache8, k_scale, v_scale, block_size, num_kv_heads, head_size};
    return paged_attention_view(query, &pv, qsl, seq_lens, block_table, block_table_stride,
                                num_seqs, num_heads, num_kv_heads, head_size, block_size,
                                num_blocks, scale, causal, 0, -1, rows, num_rows, out, lse);
}

/*
 * reshape_and_cache into an e4m3 pool: K rows quantised with k_scale, V rows
 * with v_scale (oracle_quantize_e4m3), stored at the slot as in
 * oracle_reshape_and_cache.  Returns 0, or -1 for a slot outside the pool.
 */
int oracle_reshape_and_cache_fp8(const uint16_t *key, const uint16_t *value, uint8_t *cache8,
                                 const int64_t *slot_mapping, int64_t num_tokens,
                                 int64_t num_kv_heads, int64_t head_size, int64_t block_size,
                                 int64_t num_blocks, float k_scale, float v_scale)
{
    int64_t row_elems = num_kv_heads * head_size;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= num_blocks * block_size)
            return -1;
        int64_t block = slot / block_size, off = slot % block_size;
        oracle_quantize_e4m3(key + t * row_elems, row_elems, k_scale,
                             cache8 + ((block * 2 + 0) * block_size + off) * row_elems);
        oracle_quantize_e4m3(value + t * row_elems, row_elems, v_scale,
                             cache8 + ((block * 2 + 1) * block_size + off) * row_elems);
    }
    return 0;
}

/*
 * Log-sum-exp merge of two partial attentions over disjoint key sets
 * ([blog] "Que aporta FlashInfer: JIT y cascade attention": the prefix result
 * is combined with each request's own suffix; [backend] "Limites y fallos":
 * the cross-shard softmax denominator depends on the lse base, here ln):
 *     lse = ln(exp(lse_a) + exp(lse_b))
 *     out = exp(lse_a - lse) * o_a + exp(lse_b - lse) * o_b
 * A side with lse = -inf holds no keys and leaves the other side unchanged.
 */
void oracle_lse_merge(const double *o_a, const double *lse_a, const double *o_b,
                      const double *lse_b, int64_t num_rows, int64_t head_size, double *o_out,
                      double *lse_out)
{
    for (int64_t r = 0; r < num_rows; ++r) {
        double la = lse_a[r], lb = lse_b[r];
        double m = la > lb ? la : lb;
        if (m == -INFINITY) {
            for (int64_t e = 0; e < head_size; ++e)
                o_out[r * head_size + e] = 0.0;
            lse_out[r] = -INFINITY;
            continue;
        }
        double wa = exp(la - m), wb = exp(lb - m);
#if ORACLE_MUTANT == 8
        wb = 0.0 * wb; /* planted: second term dropped */
#endif
        double l = m + log(wa + wb);
        double ca = exp(la - l), cb = exp(lb - l);
#if ORACLE_MUTANT == 8
        cb = 0.0;
#endif
        for (int64_t e = 0; e < head_size; ++e)
            o_out[r * head_size + e] = ca * o_a[r * head_size + e] + cb * o_b[r * head_size + e];
        lse_out[r] = l;
    }
}

/*
 * Cascade attention as [blog] "Que aporta FlashInfer: JIT y cascade
 * attention" describes it: R requests share a prefix of P tokens; attention
 * over the shared prefix is computed once per query (all P prefix keys lie
 * before every query, so no mask applies to them), each request's own suffix
 * keys [P, L_s) are attended with the causal rule, and the two partial
 * results are merged by log-sum-exp.  ([FA/FI] "Motivacion de diseno":
 * the prefix is taken out of the batch and computed only once;
 * [backend] "Flujo de datos": build(common_prefix_len, ...).)
 * Same argument conventions as oracle_paged_attention.
 */
int oracle_cascade_attention(const uint16_t *query, const uint16_t *cache, const int32_t *qsl,
                             const int32_t *seq_lens, const int32_t *block_table,
                             int64_t block_table_stride, int64_t num_seqs, int64_t num_heads,
                             int64_t num_kv_heads, int64_t head_size, int64_t block_size,
                             int64_t num_blocks, double scale, int causal,
                             int64_t common_prefix_len, const int64_t *rows, int64_t num_rows,
                             double *out, double *lse)
{
    int64_t num_tokens = qsl[num_seqs];
    int64_t total = rows ? num_rows : num_tokens * num_heads;
    size_t n_o = (size_t)total * (size_t)head_size;
    double *o_p = (double *)malloc(n_o * sizeof(double));
    double *o_s = (double *)malloc(n_o * sizeof(double));
    double *l_p = (double *)malloc((size_t)total * sizeof(double));
    double *l_s = (double *)malloc((size_t)total * sizeof(double));
    int rc = -3;
    if (o_p && o_s && l_p && l_s) {
#if ORACLE_MUTANT == 17
        const int64_t prefix_hi = common_prefix_len - 1;
#else
        const int64_t prefix_hi = common_prefix_len;
#endif
#if ORACLE_MUTANT == 16
        const int64_t suffix_lo = common_prefix_len + 1;
#else
        const int64_t suffix_lo = common_prefix_len;
#endif
        rc = oracle_paged_attention(query, cache, qsl, seq_lens, block_table, block_table_stride,
                                    num_seqs, num_heads, num_kv_heads, head_size, block_size,
                                    num_blocks, scale, 0, 0, prefix_hi, rows, num_rows, o_p, l_p);
        if (rc == 0)
            rc = oracle_paged_attention(query, cache, qsl, seq_lens, block_table,
                                        block_table_stride, num_seqs, num_heads, num_kv_heads,
                                        head_size, block_size, num_blocks, scale, causal,
                                        suffix_lo, -1, rows, num_rows, o_s, l_s);
        if (rc == 0)
            oracle_lse_merge(o_p, l_p, o_s, l_s, total, head_size, out, lse);
    }
    free(o_p);
    free(o_s);
    free(l_p);
    free(l_s);
    return rc;
}
