/*
 * pa_oracle.c -- CPU oracle for the paged KV-cache decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain, obviously correct
 * statement of what the GPU library computes.  Only the test-suite, the smoke
 * check and the benchmark's CPU-baseline leg may build, load or call it.  The
 * product (the CUDA library) never calls it and shares no code with it.
 *
 * Sources (five web pages on paged KV caches):
 *  [gotburnout]  "PagedAttention & Gestion du KV-Cache" (gotburnout.io glossary),
 *                section 2 "Taxonomie architecturale et modele mental" (block-table
 *                figure: logical block 0 -> physical 7, 1 -> 2, 2 -> 11, 16 tokens
 *                per block) and section 3.01 "Partage de prefixes (Copy-on-Write)".
 *  [vernieres]   "Cache KV en production" (blog.fabienvernieres.com): opening
 *                section (attention compares the current query with the keys of all
 *                previous tokens and weights their values), "Un cache par requete"
 *                (cache grows by one token per decode step), "PagedAttention : la
 *                pagination appliquee au cache KV" (table from logical position to
 *                physical page), "Reduire le poids par token" (int8 / fp8 cache).
 *  [iavox]       ia-vox-magazine.com KV-cache article, sections "PagedAttention : la
 *                revolution de l'allocation memoire" (blocks of 16 or 32 tokens,
 *                mapping table) and "Quantization du KV cache" (int8; dynamic scale
 *                recomputed for every token).
 *  [deeplearn]   deeplearn.tn KV-cache article, "Le compromis fondamental de
 *                l'inference" (only the new token's query is needed; past K and V
 *                are reused) and "Le Paged Attention" (fixed 16-token blocks,
 *                block table from logical to physical addresses).
 *
 * Readings taken where the pages are silent (each one is also listed in the
 * design notes):
 *  - attention is textbook scaled dot-product softmax attention, scale given by
 *    the caller;
 *  - grouped query heads: query head h reads kv head h / (Hq / Hkv);
 *  - cache layout [N blocks][Hkv][bs][D] for K and for V; int8 scales [N][Hkv][bs];
 *  - a token at logical position p lives in physical block table[p / bs] at offset
 *    p % bs; a negative slot marks a padding token that is not written;
 *  - a sequence with zero context produces an all-zero output;
 *  - int8: symmetric absmax per (token, kv head), separately for K and V, computed
 *    in IEEE fp32: scale = absmax / 127 (1 when absmax is 0),
 *    q = clamp(rint(x / scale), -127, 127), round half to even; dequantised value
 *    is q * scale.
 *  - fp8 (e4m3: 1 sign, 4 exponent bits with bias 7, 3 mantissa bits, largest
 *    finite value 448, no infinities): the same dynamic per-(token, kv head) scheme
 *    with scale = absmax / 448 and code = e4m3(x / scale), rounded to nearest, ties
 *    to an even mantissa, magnitudes above 448 saturated to 448 ([iavox]: fp8 KV
 *    cache on recent GPUs; [vernieres]: int8 or fp8 entries).
 *
 * All attention arithmetic is fp64.  The quantiser is fp32 on purpose: its output
 * is an integer decided by floating point, so both sides take that decision in
 * the same (fp32) precision.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_OK = 0, ORACLE_BAD_ARG = 1, ORACLE_NO_MEMORY = 2 };
enum { ORACLE_KV_BF16 = 0, ORACLE_KV_INT8 = 1, ORACLE_KV_FP8 = 2 };

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static float bf16_to_float(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static double bf16_to_double(uint16_t bits) { return (double)bf16_to_float(bits); }

/* Offset (in elements) of row (block b, kv head h, in-block offset o) of a cache
 * laid out [N][Hkv][bs][D]. */
static int64_t cache_row(int64_t b, int h, int o, int Hkv, int bs, int D)
{
    return ((b * Hkv + h) * (int64_t)bs + o) * (int64_t)D;
}

/* Index of the (block b, kv head h, offset o) entry of a scale array [N][Hkv][bs]. */
static int64_t scale_index(int64_t b, int h, int o, int Hkv, int bs)
{
    return (b * Hkv + h) * (int64_t)bs + o;
}

int oracle_version(void) { return 1; }

/* Physical slot of logical position pos for a sequence with block table `table`.
 * [gotburnout] figure: tokens 0-15 form logical block 0, 16-31 block 1, ...; the
 * block table sends logical block j to a physical block; [vernieres] the table
 * maps each logical position of the sequence to a physical page. */
int64_t oracle_slot(const int32_t *table, int64_t pos, int bs)
{
    int64_t logical_block = pos / bs;
    int64_t offset = pos % bs;
    return (int64_t)table[logical_block] * bs + offset;
}

/* Append: write key/value rows [T][Hkv][D] of the new tokens into their slots of
 * the bf16 caches.  A negative slot is a padding token and is skipped; a slot at
 * or beyond N * bs is counted and skipped.  Returns the number of such
 * out-of-range slots.  ([vernieres] "Un cache par requete": each decode step adds
 * one token to the request's cache.) */
int64_t oracle_reshape_and_cache(const uint16_t *key, const uint16_t *value,
                                 uint16_t *k_cache, uint16_t *v_cache,
                                 const int64_t *slot_mapping, int T, int Hkv,
                                 int D, int bs, int64_t N)
{
    int64_t bad = 0;
    for (int t = 0; t < T; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= N * bs) {
            ++bad;
            continue;
        }
        int64_t b = slot / bs;
        int o = (int)(slot % bs);
        for (int h = 0; h < Hkv; ++h) {
            for (int d = 0; d < D; ++d) {
                int64_t src = ((int64_t)t * Hkv + h) * D + d;
                int64_t dst = cache_row(b, h, o, Hkv, bs, D) + d;
                k_cache[dst] = key[src];
                v_cache[dst] = value[src];
            }
        }
    }
    return bad;
}

/* Dynamic per-token int8 quantisation of one row of D bf16 values ([iavox]
 * "Quantization du KV cache": a scale recomputed for every token; 8 bits halve
 * the cache).  fp32, IEEE division, round half to even. */
static void quantize_row(const uint16_t *x, int D, int8_t *q, float *scale_out)
{
    float absmax = 0.0f;
    for (int d = 0; d < D; ++d) {
        float a = fabsf(bf16_to_float(x[d]));
        if (a > absmax)
            absmax = a;
    }
    float scale = (absmax > 0.0f) ? absmax / 127.0f : 1.0f;
    for (int d = 0; d < D; ++d) {
        float r = rintf(bf16_to_float(x[d]) / scale);
        if (r > 127.0f)
            r = 127.0f;
        if (r < -127.0f)
            r = -127.0f;
        q[d] = (int8_t)r;
    }
    *scale_out = scale;
}

/* Value of an e4m3 code: subnormal m * 2^-9 (exponent field 0), else
 * (1 + m/8) * 2^(e - 7).  The code 0x7f / 0xff (NaN) is never produced here. */
double oracle_fp8_decode(uint8_t code)
{
    int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double v = e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

/* Nearest e4m3 code of x (finite), ties to an even mantissa, |x| > 448 -> 448. */
uint8_t oracle_fp8_encode(float x)
{
    uint8_t sign = signbit(x) ? 0x80 : 0;
    double a = fabs((double)x);
    if (a == 0.0)
        return sign;
    int e2;
    frexp(a, &e2); /* a = f * 2^e2, f in [0.5, 1): floor(log2 a) = e2 - 1 */
    int E = e2 - 1;
    double quantum = E < -6 ? ldexp(1.0, -9) : ldexp(1.0, E - 3);
    double v = rint(a / quantum) * quantum; /* a / quantum is exact; rint: ties to even */
    if (v > 448.0)
        v = 448.0;
    if (v == 0.0)
        return sign;
    if (v < ldexp(1.0, -6))
        return sign | (uint8_t)(v / ldexp(1.0, -9)); /* subnormal */
    frexp(v, &e2);
    E = e2 - 1;
    int m = (int)(v / ldexp(1.0, E) * 8.0) - 8;
    return sign | (uint8_t)((E + 7) << 3) | (uint8_t)m;
}

/* Dynamic per-token fp8 quantisation of one row: scale = absmax / 448 (1 when the
 * row is zero), codes e4m3(x / scale) with the division in IEEE fp32. */
static void quantize_row_fp8(const uint16_t *x, int D, uint8_t *q, float *scale_out)
{
    float absmax = 0.0f;
    for (int d = 0; d < D; ++d) {
        float a = fabsf(bf16_to_float(x[d]));
        if (a > absmax)
            absmax = a;
    }
    float scale = (absmax > 0.0f) ? absmax / 448.0f : 1.0f;
    for (int d = 0; d < D; ++d)
        q[d] = oracle_fp8_encode(bf16_to_float(x[d]) / scale);
    *scale_out = scale;
}

/* fp8 quantise-and-append, as oracle_quantize_kv with e4m3 codes. */
int64_t oracle_quantize_kv_fp8(const uint16_t *key, const uint16_t *value,
                               uint8_t *k_cache, uint8_t *v_cache, float *k_scale,
                               float *v_scale, const int64_t *slot_mapping, int T,
                               int Hkv, int D, int bs, int64_t N)
{
    int64_t bad = 0;
    for (int t = 0; t < T; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= N * bs) {
            ++bad;
            continue;
        }
        int64_t b = slot / bs;
        int o = (int)(slot % bs);
        for (int h = 0; h < Hkv; ++h) {
            int64_t src = ((int64_t)t * Hkv + h) * D;
            int64_t dst = cache_row(b, h, o, Hkv, bs, D);
            int64_t si = scale_index(b, h, o, Hkv, bs);
            quantize_row_fp8(key + src, D, k_cache + dst, &k_scale[si]);
            quantize_row_fp8(value + src, D, v_cache + dst, &v_scale[si]);
        }
    }
    return bad;
}

/* fp8 counterpart of oracle_quantize_pool. */
void oracle_quantize_pool_fp8(const uint16_t *src, uint8_t *codes, float *scales,
                              int64_t rows, int D)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        quantize_row_fp8(src + r * D, D, codes + r * D, &scales[r]);
}

/* Quantise-and-append: for each new token t and kv head h, quantise the K row and
 * the V row separately and store codes in the int8 caches [N][Hkv][bs][D] and
 * scales in [N][Hkv][bs].  Slot rules as in oracle_reshape_and_cache. */
int64_t oracle_quantize_kv(const uint16_t *key, const uint16_t *value,
                           int8_t *k_cache, int8_t *v_cache, float *k_scale,
                           float *v_scale, const int64_t *slot_mapping, int T,
                           int Hkv, int D, int bs, int64_t N)
{
    int64_t bad = 0;
    for (int t = 0; t < T; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= N * bs) {
            ++bad;
            continue;
        }
        int64_t b = slot / bs;
        int o = (int)(slot % bs);
        for (int h = 0; h < Hkv; ++h) {
            int64_t src = ((int64_t)t * Hkv + h) * D;
            int64_t dst = cache_row(b, h, o, Hkv, bs, D);
            int64_t si = scale_index(b, h, o, Hkv, bs);
            quantize_row(key + src, D, k_cache + dst, &k_scale[si]);
            quantize_row(value + src, D, v_cache + dst, &v_scale[si]);
        }
    }
    return bad;
}

/* Quantise whole cache blocks in place of a bf16 source laid out like the cache
 * ([N][Hkv][bs][D]); used to build int8 test pools row by row with the same rule
 * as the append. */
void oracle_quantize_pool(const uint16_t *src, int8_t *codes, float *scales,
                          int64_t rows, int D)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        quantize_row(src + r * D, D, codes + r * D, &scales[r]);
}

/* Copy-on-write block copy ([gotburnout] 3.01: shared pages are copied only when
 * a request starts writing its own tokens).  mapping holds n (src, dst) pairs of
 * physical block ids; every byte of the K block and of the V block is copied, and
 * the per-token scales when scale arrays are given. */
int oracle_copy_blocks(uint8_t *k_cache, uint8_t *v_cache, float *k_scale,
                       float *v_scale, const int64_t *mapping, int n,
                       int64_t block_bytes, int scale_elems_per_block)
{
    for (int i = 0; i < n; ++i) {
        int64_t src = mapping[2 * i];
        int64_t dst = mapping[2 * i + 1];
        for (int64_t j = 0; j < block_bytes; ++j) {
            k_cache[dst * block_bytes + j] = k_cache[src * block_bytes + j];
            v_cache[dst * block_bytes + j] = v_cache[src * block_bytes + j];
        }
        if (k_scale != NULL && v_scale != NULL) {
            for (int j = 0; j < scale_elems_per_block; ++j) {
                k_scale[dst * scale_elems_per_block + j] =
                    k_scale[src * scale_elems_per_block + j];
                v_scale[dst * scale_elems_per_block + j] =
                    v_scale[src * scale_elems_per_block + j];
            }
        }
    }
    return ORACLE_OK;
}

/* Value of element d of the cache row (block b, kv head h, offset o), widened to
 * fp64; int8 entries are dequantised as code * scale. */
static double cache_value(const void *cache, const float *scales, int kv_dtype,
                          int64_t b, int h, int o, int d, int Hkv, int bs, int D)
{
    int64_t idx = cache_row(b, h, o, Hkv, bs, D) + d;
    if (kv_dtype == ORACLE_KV_BF16)
        return bf16_to_double(((const uint16_t *)cache)[idx]);
    if (kv_dtype == ORACLE_KV_FP8)
        return oracle_fp8_decode(((const uint8_t *)cache)[idx]) *
               (double)scales[scale_index(b, h, o, Hkv, bs)];
    return (double)((const int8_t *)cache)[idx] *
           (double)scales[scale_index(b, h, o, Hkv, bs)];
}

/* Step 1: expand the paged K and V of sequence s, kv head h into contiguous
 * [ctx][D] fp64 arrays, reading logical position t from physical block
 * table[t / bs] at offset t % bs. */
static void gather_sequence(double *K, double *V, const void *k_cache,
                            const void *v_cache, const float *k_scale,
                            const float *v_scale, int kv_dtype,
                            const int32_t *table, int ctx, int h, int Hkv,
                            int D, int bs)
{
    for (int t = 0; t < ctx; ++t) {
        int64_t b = table[t / bs];
        int o = t % bs;
        for (int d = 0; d < D; ++d) {
            K[(int64_t)t * D + d] =
                cache_value(k_cache, k_scale, kv_dtype, b, h, o, d, Hkv, bs, D);
            V[(int64_t)t * D + d] =
                cache_value(v_cache, v_scale, kv_dtype, b, h, o, d, Hkv, bs, D);
        }
    }
}

/* Step 2: textbook attention of one query vector over contiguous K, V:
 *   w_t = exp(score_t - max) / sum_u exp(score_u - max),
 *   score_t = scale * sum_d q_d K[t][d],
 *   out_d = sum_t w_t V[t][d].
 * w (length ctx) receives the softmax weights. */
static void attend(double *out, double *w, const double *q, const double *K,
                   const double *V, int ctx, int D, double scale)
{
    for (int d = 0; d < D; ++d)
        out[d] = 0.0;
    if (ctx == 0)
        return;
    double mx = -INFINITY;
    for (int t = 0; t < ctx; ++t) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += q[d] * K[(int64_t)t * D + d];
        w[t] = scale * dot;
        if (w[t] > mx)
            mx = w[t];
    }
    double denom = 0.0;
    for (int t = 0; t < ctx; ++t) {
        w[t] = exp(w[t] - mx);
        denom += w[t];
    }
    for (int t = 0; t < ctx; ++t)
        w[t] /= denom;
    for (int t = 0; t < ctx; ++t)
        for (int d = 0; d < D; ++d)
            out[d] += w[t] * V[(int64_t)t * D + d];
}

static int check_attention_args(int S, int Hq, int Hkv, int D, int bs, int M,
                                const int32_t *context_lens, int kv_dtype)
{
    if (S < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || bs <= 0 || M < 0)
        return ORACLE_BAD_ARG;
    if (Hq % Hkv != 0)
        return ORACLE_BAD_ARG;
    if (kv_dtype != ORACLE_KV_BF16 && kv_dtype != ORACLE_KV_INT8 && kv_dtype != ORACLE_KV_FP8)
        return ORACLE_BAD_ARG;
    for (int s = 0; s < S; ++s)
        if (context_lens[s] < 0 || (int64_t)context_lens[s] > (int64_t)M * bs)
            return ORACLE_BAD_ARG;
    return ORACLE_OK;
}

/* Paged decode attention: for every sequence s and query head h,
 *   out[s][h] = attention(q[s][h], K_s, V_s) over the context_lens[s] tokens of
 *   sequence s, K_s and V_s gathered through block_tables[s] ([M] entries) from
 *   kv head h / (Hq / Hkv).
 * q is [S][Hq][D] bf16, out is [S][Hq][D] fp64.  Caches are [N][Hkv][bs][D]
 * (bf16, or int8 / fp8 e4m3 with fp32 scales [N][Hkv][bs]). */
int oracle_paged_attention(double *out, const uint16_t *q, const void *k_cache,
                           const void *v_cache, const float *k_scale,
                           const float *v_scale, int kv_dtype,
                           const int32_t *block_tables, int M,
                           const int32_t *context_lens, int S, int Hq, int Hkv,
                           int D, int bs, double scale)
{
    int rc = check_attention_args(S, Hq, Hkv, D, bs, M, context_lens, kv_dtype);
    if (rc != ORACLE_OK)
        return rc;
    int G = Hq / Hkv;
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1) collapse(2) reduction(| : failed)
    for (int s = 0; s < S; ++s) {
        for (int hk = 0; hk < Hkv; ++hk) {
            int ctx = context_lens[s];
            size_t n = (size_t)(ctx > 0 ? ctx : 1);
            double *K = malloc(n * (size_t)D * sizeof(double));
            double *V = malloc(n * (size_t)D * sizeof(double));
            double *w = malloc(n * sizeof(double));
            double *qd = malloc((size_t)D * sizeof(double));
            if (!K || !V || !w || !qd) {
                failed = 1;
            } else {
                gather_sequence(K, V, k_cache, v_cache, k_scale, v_scale,
                                kv_dtype, block_tables + (int64_t)s * M, ctx,
                                hk, Hkv, D, bs);
                for (int g = 0; g < G; ++g) {
                    int h = hk * G + g; /* query head h reads kv head h / G */
                    const uint16_t *qs = q + ((int64_t)s * Hq + h) * D;
                    for (int d = 0; d < D; ++d)
                        qd[d] = bf16_to_double(qs[d]);
                    attend(out + ((int64_t)s * Hq + h) * D, w, qd, K, V, ctx, D,
                           scale);
                }
            }
            free(K);
            free(V);
            free(w);
            free(qd);
        }
    }
    return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/* Multi-token paged attention: the step that attends several new tokens of a
 * sequence at once -- a chunk of a long prompt (chunked prefill: deeplearn.tn, "Les
 * leviers d'optimisation en production"; gaiatechstar.com discussion, the reply on
 * chunked prefill) or the draft tokens a large model checks in one pass
 * (speculative decoding, same deeplearn.tn section).
 *
 * Sequence s brings L_s = query_start[s + 1] - query_start[s] new tokens whose K and
 * V are already in the cache at logical positions ctx_s - L_s .. ctx_s - 1
 * (ctx_s = context_lens[s] counts them).  New token i (query row
 * query_start[s] + i) sits at position p = ctx_s - L_s + i and attends every token
 * up to and including its own:
 *   out[row][h] = attention(q[row][h], K_s[0..p], V_s[0..p]),
 * which is exactly what one decode step per token, in order, would give (reading:
 * a token never sees the tokens after it; with L_s = 1 this is the decode step).
 * q and out are [T][Hq][D] (bf16 in, fp64 out); rows outside every
 * [query_start[s], query_start[s + 1]) are set to zero. */
int oracle_paged_prefill(double *out, const uint16_t *q, const void *k_cache,
                         const void *v_cache, const float *k_scale,
                         const float *v_scale, int kv_dtype,
                         const int32_t *block_tables, int M,
                         const int32_t *context_lens, const int32_t *query_start,
                         int S, int T, int Hq, int Hkv, int D, int bs, double scale)
{
    int rc = check_attention_args(S, Hq, Hkv, D, bs, M, context_lens, kv_dtype);
    if (rc != ORACLE_OK)
        return rc;
    if (T < 0 || query_start[0] < 0 || query_start[S] > T)
        return ORACLE_BAD_ARG;
    for (int s = 0; s < S; ++s) {
        int L = query_start[s + 1] - query_start[s];
        if (L < 0 || L > context_lens[s])
            return ORACLE_BAD_ARG;
    }
    memset(out, 0, (size_t)T * (size_t)Hq * (size_t)D * sizeof(double));
    int G = Hq / Hkv;
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1) collapse(2) reduction(| : failed)
    for (int s = 0; s < S; ++s) {
        for (int hk = 0; hk < Hkv; ++hk) {
            int ctx = context_lens[s];
            int L = query_start[s + 1] - query_start[s];
            size_t n = (size_t)(ctx > 0 ? ctx : 1);
            double *K = malloc(n * (size_t)D * sizeof(double));
            double *V = malloc(n * (size_t)D * sizeof(double));
            double *w = malloc(n * sizeof(double));
            double *qd = malloc((size_t)D * sizeof(double));
            if (!K || !V || !w || !qd) {
                failed = 1;
            } else {
                gather_sequence(K, V, k_cache, v_cache, k_scale, v_scale,
                                kv_dtype, block_tables + (int64_t)s * M, ctx,
                                hk, Hkv, D, bs);
                for (int i = 0; i < L; ++i) {
                    int64_t row = (int64_t)query_start[s] + i;
                    int visible = ctx - L + i + 1; /* positions 0 .. ctx - L + i */
                    for (int g = 0; g < G; ++g) {
                        int h = hk * G + g;
                        const uint16_t *qs = q + (row * Hq + h) * D;
                        for (int d = 0; d < D; ++d)
                            qd[d] = bf16_to_double(qs[d]);
                        attend(out + (row * Hq + h) * D, w, qd, K, V, visible, D,
                               scale);
                    }
                }
            }
            free(K);
            free(V);
            free(w);
            free(qd);
        }
    }
    return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/* Softmax weights of one (sequence s, query head h) pair, in logical token
 * order; w receives context_lens[s] values. */
int oracle_attention_weights(double *w, const uint16_t *q, const void *k_cache,
                             const void *v_cache, const float *k_scale,
                             const float *v_scale, int kv_dtype,
                             const int32_t *block_tables, int M,
                             const int32_t *context_lens, int S, int Hq,
                             int Hkv, int D, int bs, double scale, int s, int h)
{
    int rc = check_attention_args(S, Hq, Hkv, D, bs, M, context_lens, kv_dtype);
    if (rc != ORACLE_OK)
        return rc;
    if (s < 0 || s >= S || h < 0 || h >= Hq)
        return ORACLE_BAD_ARG;
    int ctx = context_lens[s];
    size_t n = (size_t)(ctx > 0 ? ctx : 1);
    double *K = malloc(n * (size_t)D * sizeof(double));
    double *V = malloc(n * (size_t)D * sizeof(double));
    double *qd = malloc((size_t)D * sizeof(double));
    double *o = malloc((size_t)D * sizeof(double));
    if (!K || !V || !qd || !o) {
        free(K);
        free(V);
        free(qd);
        free(o);
        return ORACLE_NO_MEMORY;
    }
    int G = Hq / Hkv;
    gather_sequence(K, V, k_cache, v_cache, k_scale, v_scale, kv_dtype,
                    block_tables + (int64_t)s * M, ctx, h / G, Hkv, D, bs);
    const uint16_t *qs = q + ((int64_t)s * Hq + h) * D;
    for (int d = 0; d < D; ++d)
        qd[d] = bf16_to_double(qs[d]);
    attend(o, w, qd, K, V, ctx, D, scale);
    free(K);
    free(V);
    free(qd);
    free(o);
    return ORACLE_OK;
}

/* Threads the OpenMP loops above use (1 when built without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Set the threads of later calls (n >= 1; no effect without OpenMP).  The results do
   not depend on it: each (sequence, kv head) pair is computed by one thread in a fixed
   order. */
void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
