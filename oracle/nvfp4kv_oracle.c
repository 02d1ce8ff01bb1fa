/*
 * CPU oracle for the NVFP4 paged KV-cache path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow reference that the
 * CUDA library is checked against.  Only the test suite, the smoke check and
 * the benchmark's CPU-baseline / reference arm may build, load or call it; the
 * product path never does.  It shares no code, header, table or constant with
 * the CUDA library.
 *
 * Sources (web pages; cited by title and section):
 *   [LMSYS-summary]  "SGLang stores KV cache in 4 bits: long-context decode
 *                    throughput rises 26-30%, and FP8 stalls first under agent
 *                    concurrency" (summary of the LMSYS post "Accelerating
 *                    Long-Context and Agentic Inference with NVFP4 KV Cache"),
 *                    sections Synopsis / Interpretation / Perspective.
 *   [RTX-PRO-6000]   "NVFP4-KV-Cache auf der NVIDIA RTX PRO 6000 Blackwell
 *                    Server Edition: Genauigkeit, Nutzer", sections
 *                    "Bytes pro Token: FP8 gegenueber NVFP4", "Geschwindigkeit",
 *                    "Unterstuetzung in den Engines".
 *
 * What the pages fix: E2M1 elements (1 sign, 2 exponent, 1 mantissa bit), one
 * FP8-E4M3 scale per 16 values, an FP32 per-tensor scale above them that the
 * experiments leave at 1.0 ([RTX-PRO-6000] "Bytes pro Token"; [LMSYS-summary]
 * Perspective); 8 bytes of packed data plus 1 byte of scale per 16 values
 * ([LMSYS-summary] Interpretation, last paragraph); a paged cache whose decode
 * kernel dequantises inside attention; an extend path that dequantises the
 * cached prefix into an FP8 workspace ([LMSYS-summary] Interpretation, second
 * paragraph).  Everything else (bit layout, rounding, nibble order, page
 * layout, softmax scale) is a reading; each reading is named where it is used.
 *
 * Precision: attention is accumulated in double.  Quantisation decisions
 * (the block scale and each element code) are taken on fp32 quotients, the
 * precision the kernels use, since the pages do not fix one.
 */
#include <math.h>
#include <stdlib.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Element format E2M1: 4 bits = sign | exponent(2) | mantissa(1).
 * Reading: exponent bias 1, exponent field 0 is subnormal (0 or 0.5), no
 * infinities or NaN; magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}.               */
double oracle_e2m1_value(uint8_t code)
{
    int sign = (code >> 3) & 1;
    int e = (code >> 1) & 3;
    int m = code & 1;
    double mag;
    if (e == 0)
        mag = 0.5 * m;                          /* subnormal: m * 2^(1-1) / 2 */
    else
        mag = ldexp(1.0 + 0.5 * m, e - 1);      /* (1 + m/2) * 2^(e-1)        */
    return sign ? -mag : mag;
}

/* Round-to-nearest-even onto the E2M1 grid with saturation, sign kept.
 * "Nearest" is measured exactly: for |y| <= 6 the difference between an fp32
 * value and a grid point is exact in double whenever the two candidates are
 * close to a tie (|y| >= 0.25 there), and far from a tie an inexact distance
 * cannot change which point is nearer.  |y| above the largest magnitude takes
 * the largest magnitude (saturation).  A tie goes to the code whose mantissa
 * bit is 0 (the even code).                                                  */
uint8_t oracle_e2m1_encode(float y)
{
    double a = fabs((double)y);
    uint8_t sign = signbit(y) ? 8 : 0;
    if (a > 6.0)
        return (uint8_t)(sign | 7);
    int best = 0;
    double bestd = INFINITY;
    for (int c = 0; c < 8; ++c) {
        double d = fabs(a - oracle_e2m1_value((uint8_t)c));
        if (d < bestd || (d == bestd && (c & 1) == 0 && (best & 1) != 0)) {
            best = c;
            bestd = d;
        }
    }
    return (uint8_t)(sign | best);
}

/* ------------------------------------------------------------------------ */
/* Scale format FP8 E4M3 (the "FN" variant: no infinities, 0x7F/0xFF = NaN).
 * Reading: bias 7, exponent field 0 subnormal (m/8 * 2^-6), largest finite
 * magnitude 448 = code 0x7E.                                                 */
double oracle_e4m3_value(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 15;
    int m = code & 7;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp(m / 8.0, -6);
    else
        mag = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* Round-to-nearest-even onto the finite E4M3 grid with saturation at 448,
 * sign kept (a negative value that rounds to zero gives 0x80).  The two grid
 * points around |y| are found by bisection over the 127 finite magnitudes
 * (codes 0x00..0x7E are increasing), then the nearer one is taken; exact for
 * the same reason as in oracle_e2m1_encode.                                  */
uint8_t oracle_e4m3_encode(float y)
{
    double a = fabs((double)y);
    uint8_t sign = signbit(y) ? 0x80 : 0;
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    int lo = 0, hi = 0x7E;                     /* value(lo) <= a < value(hi) */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (oracle_e4m3_value((uint8_t)mid) <= a)
            lo = mid;
        else
            hi = mid;
    }
    double dlo = a - oracle_e4m3_value((uint8_t)lo);
    double dhi = oracle_e4m3_value((uint8_t)hi) - a;
    int c;
    if (dlo < dhi)
        c = lo;
    else if (dhi < dlo)
        c = hi;
    else
        c = (lo & 1) ? hi : lo;                 /* tie: even mantissa bit     */
    return (uint8_t)(sign | c);
}

/* Element-wise helpers over arrays (so tests can sweep many values). */
void oracle_e2m1_encode_array(const float *y, uint8_t *out, int64_t n)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e2m1_encode(y[i]);
}

void oracle_e4m3_encode_array(const float *y, uint8_t *out, int64_t n)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_encode(y[i]);
}

/* ------------------------------------------------------------------------ */
/* NVFP4 block of 16 values ([RTX-PRO-6000] "Bytes pro Token": one E4M3 scale
 * per 16 E2M1 values, FP32 tensor scale above; [LMSYS-summary] Perspective:
 * the tensor scale is left at 1.0, calibrating it is the next step).
 * With tensor scale G (reading: a value is G * s * E2M1, so the block
 * procedure runs on y_i = fl32(x_i / G), which is x_i itself at G = 1):
 *   amax  = max |y_i|
 *   S     = E4M3_RNE_sat(fl32(amax / 6))         (6 = largest E2M1 magnitude)
 *   s     = value(S)
 *   q_i   = E2M1_RNE_sat(fl32(y_i / s)), or 0 for every i when s == 0
 * Packing (reading): byte j holds element 2j in its low nibble and element
 * 2j+1 in its high nibble.                                                   */
void oracle_quantize_block16(const float *x, uint8_t *packed8, uint8_t *scale_code, float global_scale)
{
    float y[16];
    for (int i = 0; i < 16; ++i)
        y[i] = (global_scale == 1.0f) ? x[i] : x[i] / global_scale;
    float amax = 0.0f;
    for (int i = 0; i < 16; ++i) {
        float a = fabsf(y[i]);
        if (a > amax)
            amax = a;
    }
    float s32 = amax / 6.0f;
    uint8_t S = oracle_e4m3_encode(s32);
    float s = (float)oracle_e4m3_value(S);
    uint8_t q[16];
    for (int i = 0; i < 16; ++i)
        q[i] = (s == 0.0f) ? 0 : oracle_e2m1_encode(y[i] / s);
    for (int j = 0; j < 8; ++j)
        packed8[j] = (uint8_t)(q[2 * j] | (q[2 * j + 1] << 4));
    *scale_code = S;
}

/* Cache layout (reading; the pages give only the 8 B + 1 B split):
 *   data [num_pages][num_kv_heads][page_size][head_dim/2]   packed E2M1
 *   scale[num_pages][num_kv_heads][page_size][head_dim/16]  E4M3
 * one pair of pools for K and one for V.  A token's slot is
 * page * page_size + offset.                                                 */
static size_t row_index(int64_t page, int h, int off, int Hkv, int P)
{
    return ((size_t)page * (size_t)Hkv + (size_t)h) * (size_t)P + (size_t)off;
}

/* Write side: quantise new K or V rows [T][Hkv][d] (fp32) into the slots
 * slot_mapping[t] (negative = skip).  [LMSYS-summary] Interpretation ¶2: the
 * prefill quantises the same data it attends on into the NVFP4 cache.
 * head_scale[h] is the tensor scale of kv head h (reading for per-head
 * scales: the tensor scale G times a per-head factor, rounded to fp32 once;
 * equal to G for every head without per-head factors).                        */
void oracle_quantize_append(const float *x, int T, int Hkv, int d,
                            const int32_t *slot_mapping, int P,
                            uint8_t *data, uint8_t *scale, const float *head_scale)
{
    int nb = d / 16;
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        int32_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        int64_t page = slot / P;
        int off = slot % P;
        for (int h = 0; h < Hkv; ++h) {
            size_t r = row_index(page, h, off, Hkv, P);
            const float *src = x + ((size_t)t * Hkv + h) * d;
            for (int blk = 0; blk < nb; ++blk)
                oracle_quantize_block16(src + 16 * blk,
                                        data + r * (size_t)(d / 2) + 8 * blk,
                                        scale + r * (size_t)nb + blk, head_scale[h]);
        }
    }
}

/* Dequantised value of channel c of one cached NVFP4 row: E2M1 x E4M3 x G.
 * The product is exact in double (at most 6 + 24 significant bits).          */
static double nvfp4_row_value(const uint8_t *data_row, const uint8_t *scale_row, int c, float global_scale)
{
    uint8_t byte = data_row[c / 2];
    uint8_t code = (c & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
    return oracle_e2m1_value(code) * oracle_e4m3_value(scale_row[c / 16]) * (double)global_scale;
}

/* Dequantise a whole row into fp32 (test helper; at G = 1 the products are
 * exact in fp32, otherwise rounded once). */
void oracle_dequant_rows(const uint8_t *data, const uint8_t *scale, int64_t rows,
                         int d, float *out, float global_scale)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int c = 0; c < d; ++c)
            out[r * d + c] = (float)nvfp4_row_value(data + r * (d / 2),
                                                    scale + r * (d / 16), c, global_scale);
}

/* ------------------------------------------------------------------------ */
/* Decode attention (one query token per sequence, GQA).
 * For sequence b and query head i (kv head h = i / g, g = Hq / Hkv):
 *   k_j, v_j = dequantised rows of token j < L_b, gathered through
 *              block_table[b][j / P], offset j % P
 *   s_j      = sm_scale * sum_c q_c k_jc
 *   o        = sum_j softmax(s)_j v_j
 * [LMSYS-summary] Interpretation ¶2 (decode dequantises inside attention);
 * [RTX-PRO-6000] "Geschwindigkeit" (bf16 queries against NVFP4 K/V).
 * q is the bf16 query widened to float.  All sums in double.  An empty
 * sequence (L_b = 0) yields zeros.  kind 0 = NVFP4 pools, kind 1 = FP8 pool
 * (data [pages][Hkv][P][d] E4M3, scale unused).                              */
static double cache_value(int kind, const uint8_t *data, const uint8_t *scale,
                          size_t r, int d, int c, float global_scale)
{
    if (kind == 0)
        return nvfp4_row_value(data + r * (size_t)(d / 2), scale + r * (size_t)(d / 16), c, global_scale);
    return oracle_e4m3_value(data[r * (size_t)d + c]);
}

static void paged_decode_generic(int kind,
                                 const uint8_t *k_data, const uint8_t *k_scale,
                                 const uint8_t *v_data, const uint8_t *v_scale,
                                 int Hkv, int P, int d,
                                 const float *q, int B, int Hq,
                                 const int32_t *block_table, int max_pages,
                                 const int32_t *seq_lens, double sm_scale,
                                 double *out, const float *k_head_scale, const float *v_head_scale)
{
    int g = Hq / Hkv;
#pragma omp parallel for schedule(dynamic, 1)
    for (int bi = 0; bi < B * Hq; ++bi) {
        int b = bi / Hq, i = bi % Hq, h = i / g;
        float gk = k_head_scale ? k_head_scale[h] : 1.0f, gv = v_head_scale ? v_head_scale[h] : 1.0f;
        int L = seq_lens[b];
        const float *qv = q + ((size_t)b * Hq + i) * d;
        double *o = out + ((size_t)b * Hq + i) * d;
        for (int c = 0; c < d; ++c)
            o[c] = 0.0;
        if (L <= 0)
            continue;
        double m;
        /* pass 1: scores and their maximum */
        double smax = -INFINITY;
        for (int j = 0; j < L; ++j) {
            int64_t page = block_table[(size_t)b * max_pages + j / P];
            size_t r = row_index(page, h, j % P, Hkv, P);
            double dot = 0.0;
            for (int c = 0; c < d; ++c)
                dot += (double)qv[c] * cache_value(kind, k_data, k_scale, r, d, c, gk);
            double sj = dot * sm_scale;
            if (sj > smax)
                smax = sj;
        }
        m = smax;
        /* pass 2: weights and the weighted sum of values */
        double denom = 0.0;
        for (int j = 0; j < L; ++j) {
            int64_t page = block_table[(size_t)b * max_pages + j / P];
            size_t r = row_index(page, h, j % P, Hkv, P);
            double dot = 0.0;
            for (int c = 0; c < d; ++c)
                dot += (double)qv[c] * cache_value(kind, k_data, k_scale, r, d, c, gk);
            double p = exp(dot * sm_scale - m);
            denom += p;
            for (int c = 0; c < d; ++c)
                o[c] += p * cache_value(kind, v_data, v_scale, r, d, c, gv);
        }
        for (int c = 0; c < d; ++c)
            o[c] /= denom;
    }
}

void oracle_paged_decode(const uint8_t *k_data, const uint8_t *k_scale,
                         const uint8_t *v_data, const uint8_t *v_scale,
                         int Hkv, int P, int d, const float *q, int B, int Hq,
                         const int32_t *block_table, int max_pages,
                         const int32_t *seq_lens, double sm_scale, double *out,
                         const float *k_head_scale, const float *v_head_scale)
{
    paged_decode_generic(0, k_data, k_scale, v_data, v_scale, Hkv, P, d, q, B, Hq,
                         block_table, max_pages, seq_lens, sm_scale, out, k_head_scale, v_head_scale);
}

/* ------------------------------------------------------------------------ */
/* Extend path: dequantise the cached prefix of each sequence into one
 * contiguous FP8 workspace ([LMSYS-summary] Interpretation ¶2).  Reading:
 * each value is E4M3_RNE_sat(fl32(E2M1 x scale x G_h)) at workspace scale 1.0,
 * G_h the tensor scale of kv head h (the fp32 rounding only acts when
 * G_h != 1); rows of sequence b go to
 * workspace rows kv_indptr[b] + j, laid out [row][Hkv][d].                   */
void oracle_dequant_prefix_fp8(const uint8_t *data, const uint8_t *scale,
                               int Hkv, int P, int d,
                               const int32_t *block_table, int max_pages,
                               const int32_t *prefix_lens, const int32_t *kv_indptr,
                               int B, uint8_t *out, const float *head_scale)
{
    for (int b = 0; b < B; ++b) {
        int L = prefix_lens[b];
#pragma omp parallel for schedule(static)
        for (int j = 0; j < L; ++j) {
            int64_t page = block_table[(size_t)b * max_pages + j / P];
            for (int h = 0; h < Hkv; ++h) {
                size_t r = row_index(page, h, j % P, Hkv, P);
                uint8_t *dst = out + (((size_t)kv_indptr[b] + j) * Hkv + h) * d;
                for (int c = 0; c < d; ++c) {
                    float v = (float)nvfp4_row_value(data + r * (size_t)(d / 2),
                                                     scale + r * (size_t)(d / 16), c, head_scale[h]);
                    dst[c] = oracle_e4m3_encode(v);
                }
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* FP8-E4M3 comparison cache ([RTX-PRO-6000] "Unterstuetzung in den Engines":
 * the baseline runs with --kv-cache-dtype fp8_e4m3; "Bytes pro Token": FP8
 * scales of 1.0 when uncalibrated).  Each value is E4M3_RNE_sat(x * 1.0).    */
void oracle_fp8_quantize_append(const float *x, int T, int Hkv, int d,
                                const int32_t *slot_mapping, int P, uint8_t *data)
{
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        int32_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        int64_t page = slot / P;
        int off = slot % P;
        for (int h = 0; h < Hkv; ++h) {
            size_t r = row_index(page, h, off, Hkv, P);
            const float *src = x + ((size_t)t * Hkv + h) * d;
            for (int c = 0; c < d; ++c)
                data[r * (size_t)d + c] = oracle_e4m3_encode(src[c] * 1.0f);
        }
    }
}

void oracle_fp8_paged_decode(const uint8_t *k, const uint8_t *v, int Hkv, int P, int d,
                             const float *q, int B, int Hq,
                             const int32_t *block_table, int max_pages,
                             const int32_t *seq_lens, double sm_scale, double *out)
{
    paged_decode_generic(1, k, NULL, v, NULL, Hkv, P, d, q, B, Hq, block_table,
                         max_pages, seq_lens, sm_scale, out, NULL, NULL);
}

/* ------------------------------------------------------------------------ */
/* Extend attention ([LMSYS-summary] Interpretation ¶2: an extend step attends
 * over the cached prefix, dequantised into the FP8 workspace, plus the new
 * chunk).  For sequence b with prefix length P_b (workspace rows kv_indptr[b]
 * .. + P_b, E4M3 at scale 1.0) and chunk rows q_indptr[b] .. q_indptr[b+1]
 * (queries as floats; the chunk's own K/V as floats, or as E4M3 bytes at
 * scale 1.0), chunk token i and query head hq (kv head hq / g) attend over the
 * P_b prefix keys and chunk keys 0 .. i (causal within the chunk):
 *   s_j = sm_scale * q . k_j,   o = sum_j softmax(s)_j v_j   (all in double)
 * The E4M3 chunk is initial prefill as the same paragraph describes it: the
 * prompt's keys and values arrive in FP8 and attention reads them as they
 * are (prefix length 0 there; any prefix is allowed).                       */
static double chunk_value(int chunk_e4m3, const void *chunk, size_t idx)
{
    if (chunk_e4m3)
        return oracle_e4m3_value(((const uint8_t *)chunk)[idx]);
    return (double)((const float *)chunk)[idx];
}

static void extend_generic(const float *q, const int32_t *q_indptr,
                           const uint8_t *k_prefix, const uint8_t *v_prefix,
                           const int32_t *kv_indptr, const int32_t *prefix_lens,
                           const void *k_chunk, const void *v_chunk, int chunk_e4m3,
                           int B, int Hq, int Hkv, int d, double sm_scale, double *out)
{
    int g = Hq / Hkv;
    for (int b = 0; b < B; ++b) {
        int c0 = q_indptr[b], C = q_indptr[b + 1] - q_indptr[b];
        int P = prefix_lens[b];
        size_t p0 = (size_t)kv_indptr[b];
#pragma omp parallel for schedule(dynamic, 1)
        for (int ti = 0; ti < C * Hq; ++ti) {
            int i = ti / Hq, hq = ti % Hq, h = hq / g;
            const float *qv = q + ((size_t)(c0 + i) * Hq + hq) * d;
            double *o = out + ((size_t)(c0 + i) * Hq + hq) * d;
            int n = P + i + 1;
            double smax = -INFINITY;
            double *sc = (double *)malloc(sizeof(double) * (size_t)n);
            for (int j = 0; j < n; ++j) {
                double dot = 0.0;
                for (int c = 0; c < d; ++c) {
                    double kv = j < P ? oracle_e4m3_value(k_prefix[((p0 + j) * Hkv + h) * d + c])
                                      : chunk_value(chunk_e4m3, k_chunk, ((size_t)(c0 + j - P) * Hkv + h) * d + c);
                    dot += (double)qv[c] * kv;
                }
                sc[j] = dot * sm_scale;
                if (sc[j] > smax)
                    smax = sc[j];
            }
            double denom = 0.0;
            for (int c = 0; c < d; ++c)
                o[c] = 0.0;
            for (int j = 0; j < n; ++j) {
                double pj = exp(sc[j] - smax);
                denom += pj;
                for (int c = 0; c < d; ++c) {
                    double vv = j < P ? oracle_e4m3_value(v_prefix[((p0 + j) * Hkv + h) * d + c])
                                      : chunk_value(chunk_e4m3, v_chunk, ((size_t)(c0 + j - P) * Hkv + h) * d + c);
                    o[c] += pj * vv;
                }
            }
            for (int c = 0; c < d; ++c)
                o[c] /= denom;
            free(sc);
        }
    }
}

void oracle_extend_attention(const float *q, const int32_t *q_indptr,
                             const uint8_t *k_prefix, const uint8_t *v_prefix,
                             const int32_t *kv_indptr, const int32_t *prefix_lens,
                             const float *k_chunk, const float *v_chunk,
                             int B, int Hq, int Hkv, int d, double sm_scale, double *out)
{
    extend_generic(q, q_indptr, k_prefix, v_prefix, kv_indptr, prefix_lens, k_chunk, v_chunk, 0,
                   B, Hq, Hkv, d, sm_scale, out);
}

/* The same with the chunk's K/V as E4M3 bytes [rows][Hkv][d] (scale 1.0). */
void oracle_extend_attention_e4m3_chunk(const float *q, const int32_t *q_indptr,
                                        const uint8_t *k_prefix, const uint8_t *v_prefix,
                                        const int32_t *kv_indptr, const int32_t *prefix_lens,
                                        const uint8_t *k_chunk, const uint8_t *v_chunk,
                                        int B, int Hq, int Hkv, int d, double sm_scale, double *out)
{
    extend_generic(q, q_indptr, k_prefix, v_prefix, kv_indptr, prefix_lens, k_chunk, v_chunk, 1,
                   B, Hq, Hkv, d, sm_scale, out);
}

/* ------------------------------------------------------------------------ */
/* Storage arithmetic ([LMSYS-summary] Interpretation: 8 B packed + 1 B scale
 * per 16 values; [RTX-PRO-6000] "Bytes pro Token": ratio 0.5625 to FP8).     */
int64_t oracle_nvfp4_bytes(int64_t num_values)
{
    return (num_values / 16) * (8 + 1);
}

int64_t oracle_fp8_bytes(int64_t num_values)
{
    return num_values;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads the parallel loops use from now on (n >= 1); for timing the oracle
 * on one core and on all of them.  Changes no result: every parallel loop
 * writes disjoint outputs, each computed in a fixed order. */
void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}
