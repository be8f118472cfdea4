/*
 * Plain CPU oracle for paged decode attention and the paged KV-cache write.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header or table with the CUDA library.
 *
 * What it computes (all arithmetic in double precision unless stated):
 *
 *  - Decoding of stored elements, written from the bit formats: IEEE float32;
 *    bf16 (the upper 16 bits of a float32); fp8-e5m2 (1 sign bit, 5 exponent
 *    bits with bias 15, 2 mantissa bits; exponent 0 is subnormal, 31 is
 *    Inf/NaN); fp8-e4m3 (1 sign bit, 4 exponent bits with bias 7, 3 mantissa
 *    bits; exponent 0 is subnormal, no infinities, the all-ones code is NaN,
 *    largest magnitude 448); INT4 (signed 4-bit integers, two per byte, the
 *    even element in the low nibble).  fp8 and INT4 values are multiplied by
 *    the per-tensor dequant scale (and an optional per-KV-head factor).
 *
 *  - Paged decode attention ("vLLM e PagedAttention: serving high-throughput",
 *    the simplified PagedAttention CUDA-kernel pseudocode; "Inference
 *    optimization" lesson of AI Engineering from Scratch, Step 2,
 *    scaled_dot_product_attention): for sequence s and query head h, the
 *    logical key/value row t < seq_len is read from physical block
 *    block_tables[s][t / block_size] at offset t % block_size of KV head
 *    h / (num_q_heads / num_kv_heads).  The rows are first gathered into
 *    contiguous arrays, then the plain two-pass softmax is applied:
 *        z_t = scale * sum_d q[d] K[t][d];  M = max_t z_t;
 *        w_t = exp(z_t - M);  out[d] = sum_t w_t V[t][d] / sum_t w_t.
 *    The online (running max/sum) recurrence of the pseudocode is an exact
 *    rearrangement of this definition, so the oracle is the definition.
 *    seq_len == 0 gives a zero row.
 *
 *  - Several query tokens per sequence (chunked prefill, speculative
 *    verification): the n queries of a sequence of L tokens are its last n
 *    positions; query i attends rows t <= L - n + i, the causal mask of the
 *    "Inference optimization" lesson, Step 2.  Decode is n = 1.
 *
 *  - Split-sequence attention with a log-sum-exp merge (used only to pin the
 *    merge algebra): the same softmax on each partition of partition_tokens
 *    rows, then M* = max_p m_p, w_p = l_p exp(m_p - M*),
 *    out = sum_p w_p o_p / sum_p w_p.
 *
 *  - The paged cache write ("Inference optimization" lesson, section "Caches
 *    de KV": only the new token's K and V are computed and appended; section
 *    "PagedAttention": fixed 16-token pages anywhere in memory):
 *    new row i with slot = slot_mapping[i] >= 0 lands in block slot / B at
 *    offset slot % B of every KV head.  Values are converted with this file's
 *    own encoders: float32 -> bf16 round-to-nearest-even; float32 ->
 *    fp8-e5m2 as RNE(x / scale) in float32 with saturation to +-57344;
 *    float32 -> fp8-e4m3 the same with saturation to +-448; float32 -> INT4
 *    as RNE(x / scale) clamped to -8..7 (NaN -> 0).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { PKVO_F32 = 0, PKVO_BF16 = 1, PKVO_FP8_E5M2 = 2, PKVO_FP8_E4M3 = 3, PKVO_INT4 = 4 };

/* ------------------------------------------------------------------ decoders */

static double f32_from_bits(uint32_t bits)
{
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static double bf16_value(uint16_t bits)
{
    /* A bf16 is the high half of a float32 with the low half zero. */
    return f32_from_bits((uint32_t)bits << 16);
}

static double e5m2_value(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int expo = (code >> 2) & 0x1f;
    int mant = code & 0x3;
    double mag;
    if (expo == 0) {
        mag = ldexp((double)mant / 4.0, -14);          /* subnormal */
    } else if (expo == 31) {
        mag = (mant == 0) ? INFINITY : NAN;
    } else {
        mag = ldexp(1.0 + (double)mant / 4.0, expo - 15);
    }
    return sign ? -mag : mag;
}

/* fp8-e4m3 ("fn": finite, no infinities): 1 sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits.  Exponent 0 is subnormal (m/8 * 2^-6); the one
 * code with every exponent and mantissa bit set is NaN; the largest finite
 * magnitude is 1.75 * 2^8 = 448. */
static double e4m3_value(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int expo = (code >> 3) & 0xf;
    int mant = code & 0x7;
    double mag;
    if (expo == 0xf && mant == 0x7)
        return NAN;
    if (expo == 0)
        mag = ldexp((double)mant / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)mant / 8.0, expo - 7);
    return sign ? -mag : mag;
}

/* INT4: a signed 4-bit integer (two's complement, -8..7).  Two elements share
 * a byte: element i is the low nibble of byte i / 2 when i is even, the high
 * nibble when it is odd (in the [.., 16] page layout: tokens 2j and 2j+1 of
 * a row share byte j). */
static double int4_value(const void *base, size_t i)
{
    uint8_t byte = ((const uint8_t *)base)[i >> 1];
    int nib = (i & 1) ? (byte >> 4) : (byte & 0xf);
    return (double)(nib >= 8 ? nib - 16 : nib);
}

static double elem_value(const void *base, int dtype, size_t i)
{
    switch (dtype) {
    case PKVO_F32: {
        uint32_t b;
        memcpy(&b, (const uint8_t *)base + 4 * i, 4);
        return f32_from_bits(b);
    }
    case PKVO_BF16: {
        uint16_t b;
        memcpy(&b, (const uint8_t *)base + 2 * i, 2);
        return bf16_value(b);
    }
    case PKVO_FP8_E5M2:
        return e5m2_value(((const uint8_t *)base)[i]);
    case PKVO_FP8_E4M3:
        return e4m3_value(((const uint8_t *)base)[i]);
    case PKVO_INT4:
        return int4_value(base, i);
    default:
        return NAN;
    }
}

/* ------------------------------------------------------------------ encoders */

static uint16_t bf16_encode_rne(float x)
{
    uint32_t u;
    memcpy(&u, &x, 4);
    if (isnan(x))
        return 0x7fff;
    /* Keep the upper half; the lower half decides the rounding. */
    uint32_t upper = u >> 16;
    uint32_t lower = u & 0xffffu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1;  /* carries into the exponent; max finite rounds to Inf */
    return (uint16_t)upper;
}

/* Round a non-negative double holding an exact binary fraction to the nearest
 * integer, ties to even. */
static double round_half_even(double v)
{
    double fl = floor(v);
    double fr = v - fl;
    if (fr > 0.5)
        return fl + 1.0;
    if (fr < 0.5)
        return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

static uint8_t e5m2_encode_rne_satfinite(float x)
{
    if (isnan(x))
        return 0x7f;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    const double max_finite = 57344.0;   /* 1.75 * 2^15 */
    if (isinf(a) || a >= max_finite)
        return sign | 0x7b;
    if (a < ldexp(1.0, -14)) {
        /* Subnormal range: multiples of 2^-16. */
        double n = round_half_even(a * 65536.0);
        if (n >= 4.0)
            return sign | 0x04;                     /* rounds up to 2^-14 */
        return sign | (uint8_t)n;
    }
    int k;
    frexp(a, &k);            /* a = f * 2^k, f in [0.5, 1) */
    int e = k - 1;           /* a in [2^e, 2^(e+1)) */
    double ulp = ldexp(1.0, e - 2);
    double n = round_half_even(a / ulp);   /* in [4, 8] */
    if (n >= 8.0) {
        n = 4.0;
        e += 1;
    }
    if (e > 15)
        return sign | 0x7b;                         /* saturate */
    return sign | (uint8_t)(((e + 15) << 2) | ((int)n - 4));
}

/* Round to the nearest e4m3 value, ties to even; magnitudes beyond 448
 * (infinities included) saturate to +-448; NaN gives the NaN code. */
static uint8_t e4m3_encode_rne_satfinite(float x)
{
    if (isnan(x))
        return 0x7f;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (isinf(a) || a >= 448.0)
        return sign | 0x7e;
    if (a < ldexp(1.0, -6)) {
        /* Subnormal range: multiples of 2^-9. */
        double n = round_half_even(a * 512.0);
        if (n >= 8.0)
            return sign | 0x08;                     /* rounds up to 2^-6 */
        return sign | (uint8_t)n;
    }
    int k;
    frexp(a, &k);
    int e = k - 1;           /* a in [2^e, 2^(e+1)) */
    double ulp = ldexp(1.0, e - 3);
    double n = round_half_even(a / ulp);   /* in [8, 16] */
    if (n >= 16.0) {
        n = 8.0;
        e += 1;
    }
    if (e > 8 || (e == 8 && n > 14.0))
        return sign | 0x7e;                         /* saturate at 448 */
    return sign | (uint8_t)(((e + 7) << 3) | ((int)n - 8));
}

/* Round to the nearest integer, ties to even, clamped to -8..7; NaN gives 0. */
static int int4_encode_rne(float x)
{
    if (isnan(x))
        return 0;
    double a = (double)x;
    if (a >= 7.0)
        return 7;
    if (a <= -8.0)
        return -8;
    double r = (a >= 0) ? round_half_even(a) : -round_half_even(-a);
    return (int)r;
}

static void int4_store(void *base, size_t i, int q)
{
    uint8_t *b = (uint8_t *)base + (i >> 1);
    uint8_t nib = (uint8_t)(q & 0xf);
    if (i & 1)
        *b = (uint8_t)((*b & 0x0f) | (nib << 4));
    else
        *b = (uint8_t)((*b & 0xf0) | nib);
}

/* ------------------------------------------------------- exported decoders */

/* Widen n stored elements of `dtype` to double (no scale applied). */
void pkvo_decode_values(const void *src, int dtype, size_t n, double *dst)
{
    for (size_t i = 0; i < n; ++i)
        dst[i] = elem_value(src, dtype, i);
}

/* Encode n float32 values to `dtype` with this file's encoders.  For fp8 the
 * value stored is RNE_satfinite(x / scale) computed in float32. */
int pkvo_encode_values(const float *src, size_t n, int dtype, float scale, void *dst)
{
    for (size_t i = 0; i < n; ++i) {
        float x = src[i];
        switch (dtype) {
        case PKVO_F32:
            memcpy((uint8_t *)dst + 4 * i, &x, 4);
            break;
        case PKVO_BF16: {
            uint16_t b = bf16_encode_rne(x);
            memcpy((uint8_t *)dst + 2 * i, &b, 2);
            break;
        }
        case PKVO_FP8_E5M2: {
            float xs = x / scale;
            ((uint8_t *)dst)[i] = e5m2_encode_rne_satfinite(xs);
            break;
        }
        case PKVO_FP8_E4M3: {
            float xs = x / scale;
            ((uint8_t *)dst)[i] = e4m3_encode_rne_satfinite(xs);
            break;
        }
        case PKVO_INT4:
            int4_store(dst, i, int4_encode_rne(x / scale));
            break;
        default:
            return 1;
        }
    }
    return 0;
}

/* ------------------------------------------------------------- attention */

typedef struct {
    const void *q;
    int q_dtype;
    const void *k_cache;
    const void *v_cache;
    int kv_dtype;
    double k_scale, v_scale;
    const int32_t *block_tables;
    const int32_t *seq_lens;
    int num_seqs, num_q_heads, num_kv_heads, head_dim, block_size;
    int num_blocks, max_blocks_per_seq;
    double scale;
    const float *k_head_scales;   /* [num_kv_heads] or NULL: per-head factors of fp8 caches */
    const float *v_head_scales;
} pkvo_problem;

static size_t cache_index(const pkvo_problem *P, int32_t blk, int hkv, int d, int off)
{
    return (((size_t)blk * P->num_kv_heads + hkv) * P->head_dim + d) * P->block_size + off;
}

/* Gather the logical rows [0, L) of (s, hkv) into K[L][D], V[L][D].
 * Returns nonzero if a block id is out of range. */
static int gather_rows(const pkvo_problem *P, int s, int hkv, int L, double *K, double *V)
{
    const int D = P->head_dim, B = P->block_size;
    const int fp8 = P->kv_dtype == PKVO_FP8_E5M2 || P->kv_dtype == PKVO_FP8_E4M3 ||
                    P->kv_dtype == PKVO_INT4;
    double ks = fp8 ? P->k_scale : 1.0;
    double vs = fp8 ? P->v_scale : 1.0;
    if (fp8 && P->k_head_scales)
        ks *= (double)P->k_head_scales[hkv];
    if (fp8 && P->v_head_scales)
        vs *= (double)P->v_head_scales[hkv];
    for (int t = 0; t < L; ++t) {
        int32_t blk = P->block_tables[(size_t)s * P->max_blocks_per_seq + t / B];
        if (blk < 0 || blk >= P->num_blocks)
            return 1;
        for (int d = 0; d < D; ++d) {
            size_t idx = cache_index(P, blk, hkv, d, t % B);
            K[(size_t)t * D + d] = elem_value(P->k_cache, P->kv_dtype, idx) * ks;
            V[(size_t)t * D + d] = elem_value(P->v_cache, P->kv_dtype, idx) * vs;
        }
    }
    return 0;
}

/* Two-pass softmax attention of one query row over rows [t0, t1) of the
 * gathered K, V.  Writes the normalised output and the softmax statistics
 * m = max z, l = sum exp(z - m).  An empty range gives o = 0, m = -inf, l = 0. */
static void softmax_attend(const double *qrow, const double *K, const double *V, int D,
                           int t0, int t1, double scale, double *z, double *o,
                           double *m_out, double *l_out)
{
    for (int d = 0; d < D; ++d)
        o[d] = 0.0;
    if (t1 <= t0) {
        *m_out = -INFINITY;
        *l_out = 0.0;
        return;
    }
    double M = -INFINITY;
    for (int t = t0; t < t1; ++t) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d)
            acc += qrow[d] * K[(size_t)t * D + d];
        z[t - t0] = scale * acc;
        if (z[t - t0] > M)
            M = z[t - t0];
    }
    double Z = 0.0;
    for (int t = t0; t < t1; ++t) {
        double w = exp(z[t - t0] - M);
        Z += w;
        for (int d = 0; d < D; ++d)
            o[d] += w * V[(size_t)t * D + d];
    }
    for (int d = 0; d < D; ++d)
        o[d] /= Z;
    *m_out = M;
    *l_out = Z;
}

static void load_q_row(const pkvo_problem *P, int row, int h, double *qrow)
{
    size_t base = ((size_t)row * P->num_q_heads + h) * P->head_dim;
    for (int d = 0; d < P->head_dim; ++d)
        qrow[d] = elem_value(P->q, P->q_dtype, base + d);
}

/* Attention of one query row over the gathered rows [0, t_end), written
 * into dst[D].  partition_tokens > 0 computes each partition of
 * partition_tokens rows separately and merges them with the log-sum-exp
 * weights.  z, o and acc are caller scratch of t_end (>= 1), D and D
 * doubles.  Returns 3 on allocation failure. */
static int attend_row(const double *qrow, const double *K, const double *V, int D, int t_end,
                      double scale, int partition_tokens, double *z, double *o, double *acc,
                      double *dst)
{
    if (partition_tokens <= 0 || t_end <= partition_tokens) {
        double m, l;
        softmax_attend(qrow, K, V, D, 0, t_end, scale, z, o, &m, &l);
        for (int d = 0; d < D; ++d)
            dst[d] = o[d];
        return 0;
    }
    /* Log-sum-exp merge of the partitions. */
    int nparts = (t_end + partition_tokens - 1) / partition_tokens;
    double Mstar = -INFINITY;
    double *mp = malloc(nparts * sizeof(double));
    double *lp = malloc(nparts * sizeof(double));
    double *op = malloc((size_t)nparts * D * sizeof(double));
    if (!mp || !lp || !op) {
        free(mp); free(lp); free(op);
        return 3;
    }
    for (int p = 0; p < nparts; ++p) {
        int t0 = p * partition_tokens;
        int t1 = (t0 + partition_tokens < t_end) ? t0 + partition_tokens : t_end;
        softmax_attend(qrow, K, V, D, t0, t1, scale, z, op + (size_t)p * D, &mp[p], &lp[p]);
        if (mp[p] > Mstar)
            Mstar = mp[p];
    }
    double W = 0.0;
    for (int d = 0; d < D; ++d)
        acc[d] = 0.0;
    for (int p = 0; p < nparts; ++p) {
        double w = lp[p] * exp(mp[p] - Mstar);
        W += w;
        for (int d = 0; d < D; ++d)
            acc[d] += w * op[(size_t)p * D + d];
    }
    for (int d = 0; d < D; ++d)
        dst[d] = acc[d] / W;
    free(mp); free(lp); free(op);
    return 0;
}

/* Attention of the n_q query tokens q_row0 .. q_row0 + n_q - 1 (rows of q
 * [T, Hq, D]) of sequence s for every query head of KV head hkv, written into
 * rows out_row0 .. out_row0 + n_q - 1 of out [*, Hq, D].  Query i sits at
 * logical position L - n_q + i and sees the rows t <= that position.  Decode
 * is n_q = 1, q_row0 = s. */
static int attend_group_rows(const pkvo_problem *P, int s, int hkv, int q_row0, int n_q,
                             int out_row0, int partition_tokens, double *out)
{
    const int D = P->head_dim;
    const int G = P->num_q_heads / P->num_kv_heads;
    int L = P->seq_lens[s];
    int rc = 0;
    if (L < 0 || (size_t)L > (size_t)P->max_blocks_per_seq * P->block_size)
        return 2;
    if (n_q < 0 || n_q > (L > 0 ? L : 1))
        return 2;
    size_t rows = (L > 0) ? (size_t)L : 1;
    double *K = malloc(rows * D * sizeof(double));
    double *V = malloc(rows * D * sizeof(double));
    double *z = malloc(rows * sizeof(double));
    double *qrow = malloc(D * sizeof(double));
    double *o = malloc(D * sizeof(double));
    double *acc = malloc(D * sizeof(double));
    if (!K || !V || !z || !qrow || !o || !acc) {
        rc = 3;
        goto done;
    }
    if (gather_rows(P, s, hkv, L, K, V)) {
        rc = 1;
        goto done;
    }
    for (int i = 0; i < n_q; ++i) {
        const int t_end = (L > 0) ? L - n_q + i + 1 : 0;
        for (int g = 0; g < G; ++g) {
            int h = hkv * G + g;
            double *dst = out + ((size_t)(out_row0 + i) * P->num_q_heads + h) * D;
            load_q_row(P, q_row0 + i, h, qrow);
            rc |= attend_row(qrow, K, V, D, t_end, P->scale, partition_tokens, z, o, acc, dst);
        }
    }
done:
    free(K); free(V); free(z); free(qrow); free(o); free(acc);
    return rc;
}

/* Decode: one query per sequence, row s of q, written to row out_row of out. */
static int attend_group(const pkvo_problem *P, int s, int hkv, int out_row, int partition_tokens,
                        double *out)
{
    return attend_group_rows(P, s, hkv, s, 1, out_row, partition_tokens, out);
}

static int run_attention(const pkvo_problem *P, int partition_tokens, double *out,
                         int num_threads)
{
    if (P->num_kv_heads <= 0 || P->num_q_heads % P->num_kv_heads != 0)
        return 4;
    long units = (long)P->num_seqs * P->num_kv_heads;
    int rc = 0;
#ifdef _OPENMP
    if (num_threads <= 0)
        num_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads) reduction(|:rc)
#endif
    for (long u = 0; u < units; ++u) {
        int s = (int)(u / P->num_kv_heads);
        int hkv = (int)(u % P->num_kv_heads);
        rc |= attend_group(P, s, hkv, s, partition_tokens, out);
    }
    (void)num_threads;
    return rc;
}

/*
 * Paged decode attention over the whole batch; out is [S, Hq, D] doubles.
 * partition_tokens <= 0: one softmax over each sequence.  > 0: the
 * split-sequence form merged with log-sum-exp weights.  num_threads <= 0
 * uses every available thread.  Returns 0, or nonzero for an out-of-range
 * block id (1), an invalid seq_len (2), allocation failure (3) or a head
 * count that does not divide (4).
 */
int pkvo_paged_decode(const void *q, int q_dtype, const void *k_cache, const void *v_cache,
                      int kv_dtype, double k_scale, double v_scale,
                      const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                      int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                      int num_blocks, int max_blocks_per_seq, double scale,
                      int partition_tokens, double *out, int num_threads)
{
    pkvo_problem P = {q, q_dtype, k_cache, v_cache, kv_dtype, k_scale, v_scale,
                      block_tables, seq_lens, num_seqs, num_q_heads, num_kv_heads,
                      head_dim, block_size, num_blocks, max_blocks_per_seq, scale, NULL, NULL};
    return run_attention(&P, partition_tokens, out, num_threads);
}

/*
 * The same decode for fp8 caches with a dequant factor per KV head: element
 * (block, h, d, t) of K stands for code * k_scale * k_head_scales[h] (V
 * likewise).  NULL arrays mean a factor of 1.
 */
int pkvo_paged_decode_head_scaled(const void *q, int q_dtype, const void *k_cache,
                                  const void *v_cache, int kv_dtype, double k_scale,
                                  double v_scale, const float *k_head_scales,
                                  const float *v_head_scales, const int32_t *block_tables,
                                  const int32_t *seq_lens, int num_seqs, int num_q_heads,
                                  int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                  int max_blocks_per_seq, double scale, int partition_tokens,
                                  double *out, int num_threads)
{
    pkvo_problem P = {q, q_dtype, k_cache, v_cache, kv_dtype, k_scale, v_scale,
                      block_tables, seq_lens, num_seqs, num_q_heads, num_kv_heads,
                      head_dim, block_size, num_blocks, max_blocks_per_seq, scale,
                      k_head_scales, v_head_scales};
    return run_attention(&P, partition_tokens, out, num_threads);
}

/*
 * The same attention for a subset of sequences only: out is
 * [num_listed, Hq, D] and row i holds sequence seqs[i].  Used to sample
 * large batches.
 */
int pkvo_paged_decode_seqs(const void *q, int q_dtype, const void *k_cache,
                           const void *v_cache, int kv_dtype, double k_scale, double v_scale,
                           const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                           int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                           int num_blocks, int max_blocks_per_seq, double scale,
                           const int32_t *seqs, int num_listed, double *out, int num_threads)
{
    pkvo_problem P = {q, q_dtype, k_cache, v_cache, kv_dtype, k_scale, v_scale,
                      block_tables, seq_lens, num_seqs, num_q_heads, num_kv_heads,
                      head_dim, block_size, num_blocks, max_blocks_per_seq, scale, NULL, NULL};
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0)
        return 4;
    long units = (long)num_listed * num_kv_heads;
    int rc = 0;
#ifdef _OPENMP
    if (num_threads <= 0)
        num_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads) reduction(|:rc)
#endif
    for (long u = 0; u < units; ++u) {
        int s = seqs[u / num_kv_heads];
        int hkv = (int)(u % num_kv_heads);
        if (s < 0 || s >= num_seqs) {
            rc |= 2;
            continue;
        }
        rc |= attend_group(&P, s, hkv, (int)(u / num_kv_heads), 0, out);
    }
    (void)num_threads;
    return rc;
}

/*
 * Paged attention with several query tokens per sequence (chunked prefill,
 * speculative verification).  q is [T, Hq, D]; the queries of sequence s are
 * rows q_start[s] .. q_start[s+1] - 1, the last n_s = q_start[s+1] - q_start[s]
 * positions of its seq_lens[s] cached tokens (their K/V already written).
 * Query i of the sequence sits at logical position L - n_s + i and attends
 * the rows t <= that position: the causal mask of the "Inference
 * optimization" lesson, Step 2 (scores of keys j >= i + L - n_s + 1 get
 * -1e9, whose weight underflows to exactly zero; the oracle leaves them out).
 * out is [T, Hq, D].  Returns 0, or 1 (block id out of range), 2 (a length
 * or query count out of range), 3 (allocation), 4 (head counts).
 */
int pkvo_paged_prefill(const void *q, int q_dtype, const int32_t *q_start,
                       const void *k_cache, const void *v_cache, int kv_dtype, double k_scale,
                       double v_scale, const int32_t *block_tables, const int32_t *seq_lens,
                       int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                       int block_size, int num_blocks, int max_blocks_per_seq, double scale,
                       int partition_tokens, double *out, int num_threads)
{
    pkvo_problem P = {q, q_dtype, k_cache, v_cache, kv_dtype, k_scale, v_scale,
                      block_tables, seq_lens, num_seqs, num_q_heads, num_kv_heads,
                      head_dim, block_size, num_blocks, max_blocks_per_seq, scale, NULL, NULL};
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0)
        return 4;
    for (int s = 0; s < num_seqs; ++s)
        if (q_start[s + 1] < q_start[s] || q_start[s + 1] - q_start[s] > seq_lens[s])
            return 2;
    long units = (long)num_seqs * num_kv_heads;
    int rc = 0;
#ifdef _OPENMP
    if (num_threads <= 0)
        num_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads) reduction(|:rc)
#endif
    for (long u = 0; u < units; ++u) {
        int s = (int)(u / num_kv_heads);
        int hkv = (int)(u % num_kv_heads);
        rc |= attend_group_rows(&P, s, hkv, q_start[s], q_start[s + 1] - q_start[s],
                                q_start[s], partition_tokens, out);
    }
    (void)num_threads;
    return rc;
}

/* --------------------------------------------------------------- cache write */

/*
 * Scatter num_tokens new K/V rows ([T, Hkv, D] of in_dtype, f32 or bf16) into
 * the host copies of the caches ([N, Hkv, D, B] of kv_dtype).  Slots < 0 are
 * skipped.  Returns 1 if a slot lies past the pool (nothing written for it),
 * 5 for an unsupported dtype.
 */
int pkvo_reshape_and_cache_head_scaled(const void *k, const void *v, int in_dtype,
                                       const int64_t *slot_mapping, int num_tokens,
                                       int num_kv_heads, int head_dim, int block_size,
                                       int num_blocks, void *k_cache, void *v_cache,
                                       int kv_dtype, float k_scale, float v_scale,
                                       const float *k_head_scales, const float *v_head_scales);

int pkvo_reshape_and_cache(const void *k, const void *v, int in_dtype,
                           const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                           int head_dim, int block_size, int num_blocks, void *k_cache,
                           void *v_cache, int kv_dtype, float k_scale, float v_scale)
{
    return pkvo_reshape_and_cache_head_scaled(k, v, in_dtype, slot_mapping, num_tokens,
                                              num_kv_heads, head_dim, block_size, num_blocks,
                                              k_cache, v_cache, kv_dtype, k_scale, v_scale,
                                              NULL, NULL);
}

/*
 * The cache write with a quantisation factor per KV head for fp8 caches: the
 * code stored for head h is RNE_satfinite(x / (k_scale * k_head_scales[h])),
 * the divisor formed in float32 (V likewise).  NULL arrays mean 1.
 */
int pkvo_reshape_and_cache_head_scaled(const void *k, const void *v, int in_dtype,
                                       const int64_t *slot_mapping, int num_tokens,
                                       int num_kv_heads, int head_dim, int block_size,
                                       int num_blocks, void *k_cache, void *v_cache,
                                       int kv_dtype, float k_scale, float v_scale,
                                       const float *k_head_scales, const float *v_head_scales)
{
    if (in_dtype != PKVO_F32 && in_dtype != PKVO_BF16)
        return 5;
    if (kv_dtype != PKVO_F32 && kv_dtype != PKVO_BF16 && kv_dtype != PKVO_FP8_E5M2 &&
        kv_dtype != PKVO_FP8_E4M3 && kv_dtype != PKVO_INT4)
        return 5;
    int rc = 0;
    for (int i = 0; i < num_tokens; ++i) {
        int64_t slot = slot_mapping[i];
        if (slot < 0)
            continue;
        int64_t blk = slot / block_size;
        int off = (int)(slot % block_size);
        if (blk >= num_blocks) {
            rc = 1;
            continue;
        }
        for (int h = 0; h < num_kv_heads; ++h) {
            const float ksh = k_head_scales ? k_scale * k_head_scales[h] : k_scale;
            const float vsh = v_head_scales ? v_scale * v_head_scales[h] : v_scale;
            for (int d = 0; d < head_dim; ++d) {
                size_t src = ((size_t)i * num_kv_heads + h) * head_dim + d;
                size_t dst = (((size_t)blk * num_kv_heads + h) * head_dim + d) * block_size + off;
                /* Inputs are f32 or bf16: both widen to float exactly. */
                float kx = (float)elem_value(k, in_dtype, src);
                float vx = (float)elem_value(v, in_dtype, src);
                if (kv_dtype == PKVO_F32) {
                    memcpy((uint8_t *)k_cache + 4 * dst, &kx, 4);
                    memcpy((uint8_t *)v_cache + 4 * dst, &vx, 4);
                } else if (kv_dtype == PKVO_BF16) {
                    uint16_t kb = bf16_encode_rne(kx), vb = bf16_encode_rne(vx);
                    memcpy((uint8_t *)k_cache + 2 * dst, &kb, 2);
                    memcpy((uint8_t *)v_cache + 2 * dst, &vb, 2);
                } else if (kv_dtype == PKVO_FP8_E5M2) {
                    ((uint8_t *)k_cache)[dst] = e5m2_encode_rne_satfinite(kx / ksh);
                    ((uint8_t *)v_cache)[dst] = e5m2_encode_rne_satfinite(vx / vsh);
                } else if (kv_dtype == PKVO_INT4) {
                    int4_store(k_cache, dst, int4_encode_rne(kx / ksh));
                    int4_store(v_cache, dst, int4_encode_rne(vx / vsh));
                } else {
                    ((uint8_t *)k_cache)[dst] = e4m3_encode_rne_satfinite(kx / ksh);
                    ((uint8_t *)v_cache)[dst] = e4m3_encode_rne_satfinite(vx / vsh);
                }
            }
        }
    }
    return rc;
}

int pkvo_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
