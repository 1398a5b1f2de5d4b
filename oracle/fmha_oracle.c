/*
 * fmha_oracle.c -- plain fp64 CPU oracle for the fused attention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the "obviously correct" statement of
 * what the GPU library computes.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load it.  It shares no code, header, table
 * or helper with the CUDA library, and it never reads anything the CUDA
 * library produced.
 *
 * Sources (web pages of the nvfp4-megamoe-kernel repository, dsv4 directory):
 *  [A] commit e4ee9fd (dsv4) -- the multi-tile C API part
 *      (FA2 online softmax, un-normalised P, final O = sOacc / running_sum)
 *      and the "Architecture" part (MQA: K/V head stride 0).
 *  [B] CURRENT_ISSUE.md "UMMA FMHA -- Full Pipeline + Production", section
 *      "Next steps" item 4 (split-KV merge O = sum exp(lse_i) O_i / sum
 *      exp(lse_i)), section "Key lessons" (the MMA gives the UNSCALED dot
 *      product; 1/sqrt(hd) is applied in the softmax; decode PV is
 *      O[d] = sum_j P[0,j] V[d,j]).
 *  [C] commit 593bc25 (dsv4), scalar reference kernel part (online
 *      softmax with O rescale, sliding-window mask "D3", causal "D4").
 *
 * The method (online softmax over KV tiles, split-KV with an LSE merge)
 * reaches, up to rounding order, the plain definition of softmax attention.
 * So this oracle is that definition, written out in double precision:
 *
 *   s_j   = scale * sum_d q[d] k_j[d]              j in J (the attended keys)
 *   m     = max_j s_j,   l = sum_j exp(s_j - m)
 *   O     = sum_j exp(s_j - m) v_j / l
 *   lse   = m + ln(l)                              natural log, scaled logits
 *
 * Readings taken where the pages are silent (readings, not statements of
 * the pages):
 *  - layouts: Q, O [batch, n_h, T, hd]; K, V [batch, n_kv_h, s_k, hd];
 *    LSE [batch, n_h, T]; all contiguous.
 *  - GQA: query head h reads KV head h / (n_h / n_kv_h); MQA is n_kv_h = 1.
 *  - query row t sits at absolute position p = s_k - T + t (bottom-right
 *    alignment of the T new queries after the cached keys).
 *  - causal: key j attends iff j <= p.
 *  - window w > 0: key j attends iff j > p - w (the last w positions up to
 *    and including p).  w = 0 disables the window.
 *  - a row with no attended key has O = 0 and lse = -inf.
 *  - split-KV: chunk i covers keys [b0 + i*c, b0 + (i+1)*c) where
 *    b0 = first attended key of row t = 0 and c the chunk length; partial i
 *    is the same definition with J restricted to that chunk.
 *  - attention sink: [C] lists "D5c sink" as a TODO and defines nothing.
 *    Reading taken: a per-query-head logit sigma_h (natural-log units, the
 *    same units as the scaled scores s_j) that enters the softmax
 *    denominator only, as one more "key" whose value row is zero:
 *        l   = sum_j exp(s_j - m) + exp(sigma_h - m),  m = max(max_j s_j, sigma_h)
 *        O   = sum_j exp(s_j - m) v_j / l,   lse = m + ln(l)
 *    so a row with no attended key has O = 0 and lse = sigma_h, and
 *    sigma_h = -inf is no sink at all.  For split-KV the partials carry no
 *    sink and the merge adds it once to its denominator.
 *  - NVFP4 output (the "register slot for FP4 pack" of [C]'s TMEM-epilogue
 *    part; the pages' quantiser part names an E2M1 element nibble, an E4M3
 *    scale and round-to-nearest-even, and gives no block size): see
 *    oracle_quantize_nvfp4 below for the format taken.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Element types accepted for q/k/v. */
enum { ORACLE_F64 = 0, ORACLE_BF16 = 1 };

/* bf16 bits -> double.  A bf16 value is the top half of an IEEE binary32, so
 * the widening is exact. */
static double bf16_bits_to_double(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double load_elem(const void* base, size_t i, int dtype)
{
    if (dtype == ORACLE_BF16) return bf16_bits_to_double(((const uint16_t*)base)[i]);
    return ((const double*)base)[i];
}

/* Attended key range [*lo, *hi] (inclusive; empty when *lo > *hi) of query
 * row t of a block of T rows over s_k keys. */
static void attended_range(int t, int T, int s_k, int window, int causal, int* lo, int* hi)
{
    long p = (long)s_k - T + t;
    long l = 0, h = (long)s_k - 1;
    if (causal && p < h) h = p;
    if (window > 0 && p - window + 1 > l) l = p - window + 1;
    *lo = (int)l;
    *hi = (int)h;
}

/* First key of chunk 0 and the number of chunks of length kv_chunk that
 * cover every key any row attends.  Returns the chunk count (>= 1). */
int oracle_split_layout(int T, int s_k, int window, int kv_chunk, int* begin)
{
    int lo, hi;
    attended_range(0, T, s_k, window, 0, &lo, &hi);
    if (lo < 0) lo = 0;
    *begin = lo;
    int span = s_k - lo;
    if (kv_chunk <= 0 || span <= 0) return 1;
    return (span + kv_chunk - 1) / kv_chunk;
}

/* One query row: the plain definition above over keys [j0, j1] (inclusive),
 * with the sink logit `sink` (-INFINITY: none) in the denominator.
 * q_row/k_slab/v_slab are element offsets into the typed buffers. */
static void attend_one_row(const void* q, size_t q_off, const void* k, const void* v,
                           size_t kv_off, int hd, double scale, int j0, int j1,
                           int dtype, double sink, double* o_row, double* lse_out)
{
    int d, j;
    if (j0 > j1) {
        for (d = 0; d < hd; ++d) o_row[d] = 0.0;
        *lse_out = sink;  /* -inf without a sink */
        return;
    }
    int n = j1 - j0 + 1;
    double* s = (double*)malloc(sizeof(double) * (size_t)n);
    double* qd = (double*)malloc(sizeof(double) * (size_t)hd);
    for (d = 0; d < hd; ++d) qd[d] = load_elem(q, q_off + (size_t)d, dtype);

    /* scores s_j = scale * <q, k_j> */
    double m = -INFINITY;
    for (j = 0; j < n; ++j) {
        size_t kj = kv_off + (size_t)(j0 + j) * (size_t)hd;
        double dot = 0.0;
        for (d = 0; d < hd; ++d) dot += qd[d] * load_elem(k, kj + (size_t)d, dtype);
        s[j] = scale * dot;
        if (s[j] > m) m = s[j];
    }
    if (sink > m) m = sink;
    /* softmax denominator l = sum_j exp(s_j - m) (+ exp(sink - m)) */
    double l = 0.0;
    for (j = 0; j < n; ++j) l += exp(s[j] - m);
    if (sink != -INFINITY) l += exp(sink - m);
    /* O = sum_j softmax_j * v_j */
    for (d = 0; d < hd; ++d) o_row[d] = 0.0;
    for (j = 0; j < n; ++j) {
        double w = exp(s[j] - m) / l;
        size_t vj = kv_off + (size_t)(j0 + j) * (size_t)hd;
        for (d = 0; d < hd; ++d) o_row[d] += w * load_elem(v, vj + (size_t)d, dtype);
    }
    *lse_out = m + log(l);
    free(qd);
    free(s);
}

/* Attention for an explicit list of flattened query rows
 * row = ((b * n_h) + h) * T + t.  o: [n_rows, hd], lse: [n_rows].
 * Keys are further restricted to [key_begin, key_end).  sink: [n_h] sink
 * logits, or NULL for none.  Returns 0, or -1 on an invalid shape. */
int oracle_attention_rows_sink(const void* q, const void* k, const void* v, int dtype,
                               const int64_t* rows, int64_t n_rows,
                               int batch, int n_h, int n_kv_h, int T, int s_k, int hd,
                               double scale, int window, int causal,
                               int key_begin, int key_end, const double* sink, double* o, double* lse)
{
    if (batch < 0 || n_h <= 0 || n_kv_h <= 0 || n_h % n_kv_h != 0 || T < 0 || s_k < 0 || hd <= 0)
        return -1;
    const int group = n_h / n_kv_h;
    const int64_t total = (int64_t)batch * n_h * T;
    int64_t i;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 4) reduction(| : bad)
    for (i = 0; i < n_rows; ++i) {
        int64_t r = rows[i];
        if (r < 0 || r >= total) { bad = 1; continue; }
        int t = (int)(r % T);
        int h = (int)((r / T) % n_h);
        int b = (int)(r / ((int64_t)T * n_h));
        int kvh = h / group;                      /* GQA / MQA head sharing */
        int lo, hi;
        attended_range(t, T, s_k, window, causal, &lo, &hi);
        if (lo < key_begin) lo = key_begin;
        if (hi > key_end - 1) hi = key_end - 1;
        size_t q_off = (size_t)r * (size_t)hd;
        size_t kv_off = ((size_t)b * n_kv_h + kvh) * (size_t)s_k * (size_t)hd;
        attend_one_row(q, q_off, k, v, kv_off, hd, scale, lo, hi, dtype,
                       sink ? sink[h] : -INFINITY, o + (size_t)i * hd, lse + i);
    }
    return bad ? -1 : 0;
}

/* oracle_attention_rows_sink without a sink. */
int oracle_attention_rows(const void* q, const void* k, const void* v, int dtype,
                          const int64_t* rows, int64_t n_rows,
                          int batch, int n_h, int n_kv_h, int T, int s_k, int hd,
                          double scale, int window, int causal,
                          int key_begin, int key_end, double* o, double* lse)
{
    return oracle_attention_rows_sink(q, k, v, dtype, rows, n_rows, batch, n_h, n_kv_h, T, s_k, hd, scale,
                                      window, causal, key_begin, key_end, NULL, o, lse);
}

/* Every row, keys restricted to [key_begin, key_end).  o: [batch, n_h, T, hd],
 * lse: [batch, n_h, T].  sink: [n_h] or NULL. */
int oracle_attention_sink(const void* q, const void* k, const void* v, int dtype,
                          int batch, int n_h, int n_kv_h, int T, int s_k, int hd,
                          double scale, int window, int causal, int key_begin, int key_end,
                          const double* sink, double* o, double* lse)
{
    int64_t n = (int64_t)batch * n_h * T, i;
    int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
    for (i = 0; i < n; ++i) rows[i] = i;
    int rc = oracle_attention_rows_sink(q, k, v, dtype, rows, n, batch, n_h, n_kv_h, T, s_k, hd,
                                        scale, window, causal, key_begin, key_end, sink, o, lse);
    free(rows);
    return rc;
}

int oracle_attention(const void* q, const void* k, const void* v, int dtype,
                     int batch, int n_h, int n_kv_h, int T, int s_k, int hd,
                     double scale, int window, int causal, int key_begin, int key_end,
                     double* o, double* lse)
{
    return oracle_attention_sink(q, k, v, dtype, batch, n_h, n_kv_h, T, s_k, hd, scale, window, causal,
                                 key_begin, key_end, NULL, o, lse);
}

/* Split-KV merge [B] "Next steps" item 4:
 *     O = sum_i exp(lse_i) O_i / sum_i exp(lse_i),   lse = ln sum_i exp(lse_i)
 * evaluated with every exponent shifted by max_i lse_i (the same quotient,
 * kept in range).  A partial with lse_i = -inf has weight 0; if every partial
 * is empty the row is O = 0, lse = -inf.
 * With a sink logit sigma (sink_rows[r], per output row; NULL: none) the
 * denominator also holds exp(sigma) once: O = sum_i exp(lse_i) O_i /
 * (sum_i exp(lse_i) + exp(sigma)), lse = ln(sum_i exp(lse_i) + exp(sigma)).
 * o_parts: [n_splits, rows, hd], lse_parts: [n_splits, rows]. */
void oracle_merge_sink(const double* o_parts, const double* lse_parts, int n_splits,
                       int64_t rows, int hd, const double* sink_rows, double* o, double* lse)
{
    int64_t r;
#pragma omp parallel for schedule(static)
    for (r = 0; r < rows; ++r) {
        int i, d;
        const double sg = sink_rows ? sink_rows[r] : -INFINITY;
        double mx = sg;
        for (i = 0; i < n_splits; ++i)
            if (lse_parts[(size_t)i * rows + r] > mx) mx = lse_parts[(size_t)i * rows + r];
        double* orow = o + (size_t)r * hd;
        for (d = 0; d < hd; ++d) orow[d] = 0.0;
        if (mx == -INFINITY) { lse[r] = -INFINITY; continue; }
        double den = 0.0;
        for (i = 0; i < n_splits; ++i) den += exp(lse_parts[(size_t)i * rows + r] - mx);
        if (sg != -INFINITY) den += exp(sg - mx);
        for (i = 0; i < n_splits; ++i) {
            double w = exp(lse_parts[(size_t)i * rows + r] - mx) / den;
            const double* op = o_parts + ((size_t)i * rows + r) * hd;
            for (d = 0; d < hd; ++d) orow[d] += w * op[d];
        }
        lse[r] = mx + log(den);
    }
}

void oracle_merge(const double* o_parts, const double* lse_parts, int n_splits,
                  int64_t rows, int hd, double* o, double* lse)
{
    oracle_merge_sink(o_parts, lse_parts, n_splits, rows, hd, NULL, o, lse);
}

void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}


/* ------------------------------------------------------------------------
 * NVFP4 quantisation of output rows.
 *
 * Format (readings; the pages fix only the element and scale types and the
 * rounding rule):
 *  - each row of hd values is cut into blocks of 16 consecutive elements;
 *  - block scale: s = E4M3(amax / (6 g)), amax = max |x_i| over the block,
 *    g = a global fp32 scale given by the caller (> 0); E4M3 is 1 sign, 4
 *    exponent bits (bias 7), 3 mantissa bits, subnormals below 2^-6, largest
 *    finite value 448 (code 0x7F is NaN and never produced);
 *  - element code: E2M1(x_i / (g s)): magnitude in {0, 0.5, 1, 1.5, 2, 3, 4,
 *    6} by code 0..7 (1 sign, 2 exponent bits, 1 mantissa bit), sign in bit 3
 *    (set only for a negative value whose magnitude code is not 0);
 *  - both roundings: to the nearest representable value, a tie going to the
 *    even code (mantissa bit 0), and values beyond the largest finite value
 *    saturate to it;
 *  - s = 0 (an all-zero block, or amax / (6 g) rounding to 0) gives 0 codes;
 *  - a value is recovered as g * s * e;
 *  - storage: codes[row][hd / 2] bytes, element 2i in the low nibble of
 *    byte i; scales[row][hd / 16] E4M3 bytes.
 * The pages' final threshold list for the E2M1 rounding (0.25, 0.75, 1.25,
 * 1.75, 2.75, 3.75, 5.25) agrees with the midpoints of the E2M1 grid up to
 * 1.75 only (the midpoints of 2|3, 3|4 and 4|6 are 2.5, 3.5 and 5); the
 * plain definition above is taken instead.
 * Precision: amax / (6 g) and x_i / (g s) are evaluated in fp32 (the product
 * 6 g and g s rounded to fp32 first), as the kernels do, so that both sides
 * take every rounding decision on the same fp32 number.
 * ------------------------------------------------------------------------ */

/* value of E4M3 code c (0 .. 0x7E), non-negative */
static double e4m3_value(int c)
{
    int e = c >> 3, m = c & 7;
    if (e == 0) return ldexp((double)m / 8.0, -6);
    return ldexp(1.0 + (double)m / 8.0, e - 7);
}

/* nearest E4M3 code to a >= 0, ties to the even code, saturating at 448 */
static int e4m3_code_rne(double a)
{
    int best = 0;
    for (int c = 1; c <= 0x7E; ++c) {
        double d_new = fabs(a - e4m3_value(c)), d_best = fabs(a - e4m3_value(best));
        if (d_new < d_best || (d_new == d_best && (c & 1) == 0)) best = c;
    }
    return best;
}

static const double kE2M1[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

/* nearest E2M1 magnitude code to a >= 0, ties to the even code, saturating at 6 */
static int e2m1_code_rne(double a)
{
    int best = 0;
    for (int c = 1; c < 8; ++c) {
        double d_new = fabs(a - kE2M1[c]), d_best = fabs(a - kE2M1[best]);
        if (d_new < d_best || (d_new == d_best && (c & 1) == 0)) best = c;
    }
    return best;
}

/* x: rows x hd fp32 values (hd a multiple of 16); g: global scale (> 0).
 * Writes codes [rows][hd / 2] and scales [rows][hd / 16].  Returns 0, or -1
 * for an invalid argument. */
int oracle_quantize_nvfp4(const float* x, long rows, int hd, float g, uint8_t* codes, uint8_t* scales)
{
    if (rows < 0 || hd <= 0 || hd % 16 != 0 || !(g > 0.0f) || isinf(g)) return -1;
    for (long r = 0; r < rows; ++r) {
        for (int blk = 0; blk < hd / 16; ++blk) {
            const float* xb = x + (size_t)r * hd + blk * 16;
            float amax = 0.0f;
            for (int i = 0; i < 16; ++i)
                if (fabsf(xb[i]) > amax) amax = fabsf(xb[i]);
            const float six_g = 6.0f * g;
            const float sv = amax / six_g;
            const int sc = e4m3_code_rne((double)sv);
            const float s = (float)e4m3_value(sc);
            scales[(size_t)r * (hd / 16) + blk] = (uint8_t)sc;
            for (int i = 0; i < 16; i += 2) {
                int nib[2];
                for (int h = 0; h < 2; ++h) {
                    int code = 0;
                    if (s > 0.0f) {
                        const float gs = g * s;
                        const float y = xb[i + h] / gs;
                        code = e2m1_code_rne(fabs((double)y));
                        if (y < 0.0f && code != 0) code |= 8;
                    }
                    nib[h] = code;
                }
                codes[(size_t)r * (hd / 2) + blk * 8 + i / 2] = (uint8_t)(nib[0] | (nib[1] << 4));
            }
        }
    }
    return 0;
}
