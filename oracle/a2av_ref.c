/*
 * CPU oracle for the AlltoAllv + Permute + GroupedMatMul hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may load or call
 * this library; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or helper with the
 * CUDA library: it is written straight from the operator's definition, as
 * plainly as possible, so that a reader can check it against the page by eye.
 *
 * Source: "aclnnAlltoAllvGroupedMatMul" (Huawei CANN operator page),
 *   - "API function": AlltoAllv, Permute and GroupedMatMul for the routed
 *     experts, with an independent MatMul for the shared expert;
 *   - "Formula": permuteOut = Permute(ataOut), gmmY = permuteOut x gmmWeight,
 *     mmY = mmX x mmWeight;
 *   - "Shape variables": A is the sum of recvCounts; e experts per rank.
 * Readings where the page is silent (the order of rows inside an expert after
 * Permute, the layout of recvCounts and gmmWeight) are stated at each
 * function.
 *
 * Element formats: 16-bit floats are passed as raw bit patterns (uint16_t).
 * dtype 0 = bfloat16, dtype 1 = IEEE binary16.  Products are formed and
 * summed in double, k ascending, one output element at a time.
 *
 * Pins: every function here is checked in tests/test_oracle_pins.py against
 * facts fixed by the page or by mathematics (sum rule, bijection, identity
 * cases, numpy float64 matmul, exact integer cases, hand-worked fixtures).
 *
 * Return codes: 0 = ok, 1 = bad argument, 2 = recvCounts inconsistent with A.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define REF_OK 0
#define REF_BAD_ARG 1
#define REF_BAD_COUNTS 2

/* ---- 16-bit float decoding, from the format definitions ---------------- */

/* bfloat16: the upper half of an IEEE binary32 word. */
static double bf16_value(uint16_t bits)
{
    uint32_t word = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &word, sizeof f);
    return (double)f;
}

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
 * bits; exponent 0 encodes zero and subnormals, exponent 31 inf and NaN. */
static double fp16_value(uint16_t bits)
{
    int sign = bits >> 15;
    int expo = (bits >> 10) & 0x1f;
    int frac = bits & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)frac, -24);                 /* frac * 2^-14 / 2^10 */
    else if (expo == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + frac), expo - 25);  /* (1 + frac/2^10) * 2^(expo-15) */
    return sign ? -v : v;
}

static double bf16_table[65536];
static double fp16_table[65536];
static int tables_ready = 0;

static void build_tables(void)
{
    if (tables_ready)
        return;
    for (int i = 0; i < 65536; ++i) {
        bf16_table[i] = bf16_value((uint16_t)i);
        fp16_table[i] = fp16_value((uint16_t)i);
    }
    tables_ready = 1;
}

static const double *table_for(int dtype)
{
    build_tables();
    return dtype == 0 ? bf16_table : fp16_table;
}

/* Decode n 16-bit values to double (exposed so tests can pin the decoders). */
int a2av_ref_decode(int dtype, const uint16_t *bits, int64_t n, double *out)
{
    if ((dtype != 0 && dtype != 1) || n < 0 || (n && (!bits || !out)))
        return REF_BAD_ARG;
    const double *t = table_for(dtype);
    for (int64_t i = 0; i < n; ++i)
        out[i] = t[bits[i]];
    return REF_OK;
}

/* ---- Permute bookkeeping ----------------------------------------------- */

/*
 * Offsets of the (source rank w, local expert j) segments.
 *
 * ataOut arrives rank-major: all rows from source 0 (its rows for expert 0,
 * then expert 1, ...), then all rows from source 1, and so on; segment
 * (w, j) holds recvCounts[w*e + j] rows (page: "Formula", ataOut =
 * AlltoAllv(gmmX); "Shape variables": A = sum of recvCounts).
 *
 * permuteOut is expert-major: all rows of expert 0, then expert 1, ...
 * Inside one expert the rows keep their arrival order: source rank
 * ascending, and the order within a segment unchanged (the page names the
 * step Permute without fixing the order inside a group; this stable order is
 * the reading taken).
 *
 *   src_off[w*e+j]  first ataOut row of segment (w, j)
 *   dst_off[w*e+j]  first permuteOut row of segment (w, j)
 *   group_rows[j]   rows of expert j, summed over sources
 *   group_off[j]    first permuteOut row of expert j; group_off[e] = A
 */
int a2av_ref_plan(int32_t W, int32_t e, const int32_t *recvCounts, int64_t A,
                  int64_t *src_off, int64_t *dst_off, int64_t *group_rows,
                  int64_t *group_off)
{
    if (W < 1 || e < 1 || !recvCounts || !src_off || !dst_off || !group_rows || !group_off)
        return REF_BAD_ARG;

    int64_t total = 0;
    for (int32_t w = 0; w < W; ++w) {
        for (int32_t j = 0; j < e; ++j) {
            int32_t c = recvCounts[w * e + j];
            if (c < 0)
                return REF_BAD_COUNTS;
            src_off[w * e + j] = total;
            total += c;
        }
    }
    if (total != A)
        return REF_BAD_COUNTS;

    for (int32_t j = 0; j < e; ++j) {
        group_rows[j] = 0;
        for (int32_t w = 0; w < W; ++w)
            group_rows[j] += recvCounts[w * e + j];
    }
    group_off[0] = 0;
    for (int32_t j = 0; j < e; ++j)
        group_off[j + 1] = group_off[j] + group_rows[j];

    for (int32_t j = 0; j < e; ++j) {
        int64_t at = group_off[j];
        for (int32_t w = 0; w < W; ++w) {
            dst_off[w * e + j] = at;
            at += recvCounts[w * e + j];
        }
    }
    return REF_OK;
}

/*
 * permuteOut = Permute(ataOut) (page: "Formula", routed experts): copy every
 * row of every segment from its rank-major place to its expert-major place.
 * A bit copy of H1 16-bit elements per row.
 */
int a2av_ref_permute(int32_t W, int32_t e, const int32_t *recvCounts, int64_t A,
                     int64_t H1, const uint16_t *ataOut, uint16_t *permuteOut)
{
    if (W < 1 || e < 1 || H1 < 1 || A < 0 || (A && (!ataOut || !permuteOut)))
        return REF_BAD_ARG;
    int64_t E = (int64_t)W * e;
    int64_t *src_off = malloc(sizeof(int64_t) * E);
    int64_t *dst_off = malloc(sizeof(int64_t) * E);
    int64_t *group_rows = malloc(sizeof(int64_t) * e);
    int64_t *group_off = malloc(sizeof(int64_t) * (e + 1));
    int rc = a2av_ref_plan(W, e, recvCounts, A, src_off, dst_off, group_rows, group_off);
    if (rc == REF_OK) {
        for (int32_t j = 0; j < e; ++j)
            for (int32_t w = 0; w < W; ++w)
                for (int64_t r = 0; r < recvCounts[w * e + j]; ++r)
                    memcpy(permuteOut + (dst_off[w * e + j] + r) * H1,
                           ataOut + (src_off[w * e + j] + r) * H1,
                           sizeof(uint16_t) * (size_t)H1);
    }
    free(src_off);
    free(dst_off);
    free(group_rows);
    free(group_off);
    return rc;
}

/* ---- Products ----------------------------------------------------------- */

/*
 * out[r][n] = sum_k x[row][k] * w[k][n] in double, k ascending, for the
 * listed rows of x ([*, K] row-major) and w ([K, N] row-major).
 */
static void rows_times_matrix(const double *dec, const uint16_t *x, const uint16_t *w,
                              int64_t K, int64_t N, const int64_t *rows,
                              int64_t nrows, const int64_t *row_weight_index,
                              double *out)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        const uint16_t *xr = x + rows[r] * K;
        const uint16_t *wm = w + (row_weight_index ? row_weight_index[r] : 0) * K * N;
        double *o = out + r * N;
        for (int64_t n = 0; n < N; ++n)
            o[n] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double a = dec[xr[k]];
            const uint16_t *wk = wm + k * N;
            for (int64_t n = 0; n < N; ++n)
                o[n] += a * dec[wk[n]];
        }
    }
}

/*
 * gmmY = permuteOut x gmmWeight (page: "Formula", routed experts), as a
 * grouped product: row i of permuteOut belongs to expert j when
 * group_off[j] <= i < group_off[j+1], and is multiplied by gmmWeight[j],
 * an [H1, N1] row-major matrix (gmmWeight is [e, H1, N1]).  Row i of gmmY
 * pairs with row i of permuteOut (expert-major, no un-permute).
 *
 * Computes only the listed rows (all of them when rows == NULL).
 * out is [nrows, N1] double.
 */
int a2av_ref_grouped_matmul(int32_t e, const int64_t *group_rows, int64_t A,
                            int64_t H1, int64_t N1, int32_t dtype,
                            const uint16_t *permuteOut, const uint16_t *gmmWeight,
                            const int64_t *rows, int64_t nrows, double *out)
{
    if (e < 1 || !group_rows || A < 0 || H1 < 1 || N1 < 1 || (dtype != 0 && dtype != 1))
        return REF_BAD_ARG;
    int64_t sum = 0;
    for (int32_t j = 0; j < e; ++j) {
        if (group_rows[j] < 0)
            return REF_BAD_COUNTS;
        sum += group_rows[j];
    }
    if (sum != A)
        return REF_BAD_COUNTS;
    if (!rows)
        nrows = A;
    if (nrows == 0)
        return REF_OK;
    if (!permuteOut || !gmmWeight || !out || nrows < 0)
        return REF_BAD_ARG;

    int64_t *row_list = malloc(sizeof(int64_t) * nrows);
    int64_t *expert = malloc(sizeof(int64_t) * nrows);
    int bad = 0;
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = rows ? rows[r] : r;
        row_list[r] = i;
        if (i < 0 || i >= A) {
            bad = 1;
            break;
        }
        int64_t start = 0;
        int32_t j = 0;
        while (i >= start + group_rows[j]) {
            start += group_rows[j];
            ++j;
        }
        expert[r] = j;
    }
    if (!bad)
        rows_times_matrix(table_for(dtype), permuteOut, gmmWeight, H1, N1,
                          row_list, nrows, expert, out);
    free(row_list);
    free(expert);
    return bad ? REF_BAD_ARG : REF_OK;
}

/*
 * mmY = mmX x mmWeight (page: "Formula", shared experts): mmX [BS, H2],
 * mmWeight [H2, N2], both row-major.  Only the listed rows (all when
 * rows == NULL); out is [nrows, N2] double.
 */
int a2av_ref_matmul(int64_t BS, int64_t H2, int64_t N2, int32_t dtype,
                    const uint16_t *mmX, const uint16_t *mmWeight,
                    const int64_t *rows, int64_t nrows, double *out)
{
    if (BS < 0 || H2 < 1 || N2 < 1 || (dtype != 0 && dtype != 1))
        return REF_BAD_ARG;
    if (!rows)
        nrows = BS;
    if (nrows == 0)
        return REF_OK;
    if (!mmX || !mmWeight || !out || nrows < 0)
        return REF_BAD_ARG;
    int64_t *row_list = malloc(sizeof(int64_t) * nrows);
    int bad = 0;
    for (int64_t r = 0; r < nrows; ++r) {
        row_list[r] = rows ? rows[r] : r;
        if (row_list[r] < 0 || row_list[r] >= BS)
            bad = 1;
    }
    if (!bad)
        rows_times_matrix(table_for(dtype), mmX, mmWeight, H2, N2, row_list, nrows,
                          NULL, out);
    free(row_list);
    return bad ? REF_BAD_ARG : REF_OK;
}

/* Threads the product loops use (the CPU baseline reports it). */
/* Threads the OpenMP loops use from here on (n >= 1); the results do not
 * depend on it: every output row is one sequential float64 sum.  Returns the
 * new count.  (For timing the oracle on one core beside all of them.) */
int a2av_ref_set_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1)
        omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

int a2av_ref_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- AMP dynamic loss scale (page "aclnnAmpUpdateScale") ---------------
 *
 * "Formula" of that page, with its four explanatory notes and the
 * "Inf/NaN priority" and "overflow protection" constraints:
 *   found_inf != 0                      -> scale * backoff_factor, tracker = 0
 *   else tracker + 1 == growth_interval -> new = scale * growth_factor;
 *                                          scale = new if new is finite (else
 *                                          unchanged); tracker = 0 either way
 *   else                                -> scale unchanged, tracker + 1
 * The page requires current_scale and found_inf of one floating type; this
 * oracle takes float32 for both (the products are float32 products).
 * Returns REF_BAD_ARG for growth_interval < 1 (page: [1, 2147483647]).
 */
int a2av_ref_amp_update_scale(float *scale, int32_t *growth_tracker, float found_inf,
                              float growth_factor, float backoff_factor, int32_t growth_interval)
{
    if (!scale || !growth_tracker || growth_interval < 1)
        return REF_BAD_ARG;
    if (found_inf != 0.0f) {            /* NaN != 0 is true: NaN counts as found */
        *scale = *scale * backoff_factor;
        *growth_tracker = 0;
    } else if (*growth_tracker + 1 == growth_interval) {
        float grown = *scale * growth_factor;
        if (isfinite(grown))
            *scale = grown;
        *growth_tracker = 0;
    } else {
        *growth_tracker = *growth_tracker + 1;
    }
    return REF_OK;
}

/* 1 when any of the n values (dtype 0 bf16, 1 fp16, 2 fp32) is inf or NaN. */
int a2av_ref_any_nonfinite(int dtype, const void *x, int64_t n, int32_t *found)
{
    if (!found || n < 0 || (n && !x) || dtype < 0 || dtype > 2)
        return REF_BAD_ARG;
    *found = 0;
    for (int64_t i = 0; i < n && !*found; ++i) {
        double v;
        if (dtype == 2) {
            float f;
            memcpy(&f, (const char *)x + 4 * i, 4);
            v = f;
        } else {
            uint16_t b;
            memcpy(&b, (const char *)x + 2 * i, 2);
            v = dtype == 0 ? bf16_value(b) : fp16_value(b);
        }
        if (!isfinite(v))
            *found = 1;
    }
    return REF_OK;
}

/* ---- Quantised reduce (page "aclnnQuantReduceScatter") -----------------
 *
 * "Formula": output = Reduce(AllToAllScales * AllToAllData), the Reduce
 * running over the data received from the different ranks.  On this rank,
 * after the AllToAll, data[w] and scales[w] are what source rank w sent:
 *     out[i][h] = sum over w of value(data[w][i][h]) * scale(w, i, h)
 * "Constraints": mx quantisation = FLOAT8_E4M3FN / FLOAT8_E5M2 data with
 * FLOAT8_E8M0 scales, one per 32 elements along H (scalesDataSize =
 * BS * H / 32 bytes); pertoken-pergroup = INT8 / FLOAT8 data with float
 * scales, one per 128 elements along H (BS * H / 128 * 4 bytes).
 * Summed in double, w ascending.
 *
 * qtype: 0 E4M3FN, 1 E5M2, 2 INT8.  mode: 0 mx (E8M0 per 32), 1 float per 128.
 */

/* FLOAT8_E4M3FN: 1 sign, 4 exponent (bias 7), 3 fraction bits; no
 * infinities; S.1111.111 is NaN; exponent 0 encodes zero and subnormals. */
static double e4m3_value(uint8_t b)
{
    int sign = b >> 7, expo = (b >> 3) & 0xf, frac = b & 7;
    double v;
    if (expo == 15 && frac == 7)
        v = NAN;
    else if (expo == 0)
        v = ldexp((double)frac, -9);                   /* frac/8 * 2^(1-7) */
    else
        v = ldexp((double)(8 + frac), expo - 10);      /* (1 + frac/8) * 2^(expo-7) */
    return sign ? -v : v;
}

/* FLOAT8_E5M2: 1 sign, 5 exponent (bias 15), 2 fraction bits, IEEE rules. */
static double e5m2_value(uint8_t b)
{
    int sign = b >> 7, expo = (b >> 2) & 0x1f, frac = b & 3;
    double v;
    if (expo == 31)
        v = frac ? NAN : INFINITY;
    else if (expo == 0)
        v = ldexp((double)frac, -16);                  /* frac/4 * 2^(1-15) */
    else
        v = ldexp((double)(4 + frac), expo - 17);      /* (1 + frac/4) * 2^(expo-15) */
    return sign ? -v : v;
}

/* FLOAT8_E8M0: an unsigned power of two 2^(e - 127); 0xFF is NaN. */
static double e8m0_value(uint8_t e)
{
    return e == 0xff ? NAN : ldexp(1.0, (int)e - 127);
}

static double q_value(int qtype, uint8_t b)
{
    if (qtype == 0)
        return e4m3_value(b);
    if (qtype == 1)
        return e5m2_value(b);
    return (double)(int8_t)b;
}

/* Decode n bytes of one 8-bit format (0 E4M3FN, 1 E5M2, 2 INT8, 3 E8M0). */
int a2av_ref_decode8(int kind, const uint8_t *bits, int64_t n, double *out)
{
    if (kind < 0 || kind > 3 || n < 0 || (n && (!bits || !out)))
        return REF_BAD_ARG;
    for (int64_t i = 0; i < n; ++i)
        out[i] = kind == 3 ? e8m0_value(bits[i]) : q_value(kind, bits[i]);
    return REF_OK;
}

int a2av_ref_quant_reduce(int32_t W, int64_t rows, int64_t H, int32_t qtype, int32_t mode,
                          const uint8_t *data, const void *scales, double *out)
{
    if (W < 1 || rows < 0 || H < 1 || qtype < 0 || qtype > 2 || mode < 0 || mode > 1)
        return REF_BAD_ARG;
    if (mode == 0 && qtype == 2)
        return REF_BAD_ARG;                            /* mx takes FLOAT8 data only */
    const int64_t group = mode == 0 ? 32 : 128;
    if (H % group)
        return REF_BAD_ARG;
    if (rows && (!data || !scales || !out))
        return REF_BAD_ARG;
    const int64_t ng = H / group;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < rows; ++i) {
        for (int64_t h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int32_t w = 0; w < W; ++w) {
                const int64_t row = (int64_t)w * rows + i;
                double s;
                if (mode == 0) {
                    s = e8m0_value(((const uint8_t *)scales)[row * ng + h / group]);
                } else {
                    float f;
                    memcpy(&f, (const char *)scales + 4 * (row * ng + h / group), 4);
                    s = f;
                }
                acc += q_value(qtype, data[row * H + h]) * s;
            }
            out[i * H + h] = acc;
        }
    }
    return REF_OK;
}

/* ---- MX (block-scaled FP8) grouped product ----------------------------
 *
 * The GroupedMatMul of "aclnnAlltoAllvGroupedMatMul" ("Formula": gmmY =
 * permuteOut x gmmWeight) with its operands in the mx quantisation that the
 * "aclnnQuantReduceScatter" page's "Constraints" define: FLOAT8_E4M3FN or
 * FLOAT8_E5M2 codes, one FLOAT8_E8M0 scale per 32 consecutive elements of a
 * row (scalesDataSize = rows * H / 32 bytes).  Both operands are blocked
 * along the contraction dimension K, so
 *
 *   out[i][n] = sum_k  value(a[i][k]) * 2^(sa[i][k/32] - 127)
 *                    * value(w[n][k]) * 2^(sw[n][k/32] - 127)
 *
 * for row i of group j, with w = that group's weight.  Layouts (row-major):
 *   a   [A, K] codes,  sa [A, K/32] E8M0          (rows expert-major)
 *   w   [e, N, K] codes (each output column's K codes contiguous),
 *   sw  [e, N, K/32] E8M0.
 * Each element is decoded to its exact value, products are formed and summed
 * in double, k ascending.  `rows` (length nrows) selects output rows as in
 * a2av_ref_grouped_matmul (NULL: all A rows); out is [nrows, N].
 * qa, qw: 0 = E4M3FN, 1 = E5M2.
 */
int a2av_ref_mx_grouped_matmul(int32_t e, const int64_t *group_rows, int64_t A, int64_t K, int64_t N,
                               int32_t qa, int32_t qw, const uint8_t *a, const uint8_t *sa,
                               const uint8_t *w, const uint8_t *sw, const int64_t *rows, int64_t nrows,
                               double *out)
{
    if (e < 1 || !group_rows || A < 0 || K < 32 || K % 32 || N < 1 || qa < 0 || qa > 1 || qw < 0 || qw > 1)
        return REF_BAD_ARG;
    int64_t sum = 0;
    for (int32_t j = 0; j < e; ++j) {
        if (group_rows[j] < 0)
            return REF_BAD_COUNTS;
        sum += group_rows[j];
    }
    if (sum != A)
        return REF_BAD_COUNTS;
    if (!rows)
        nrows = A;
    if (nrows == 0)
        return REF_OK;
    if (!a || !sa || !w || !sw || !out || nrows < 0)
        return REF_BAD_ARG;
    const int64_t nb = K / 32;
    int bad = 0;
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t i = rows ? rows[r] : r;
        if (i < 0 || i >= A)
            bad = 1;
    }
    if (bad)
        return REF_BAD_ARG;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t i = rows ? rows[r] : r;
        int64_t start = 0;
        int32_t j = 0;
        while (i >= start + group_rows[j]) {
            start += group_rows[j];
            ++j;
        }
        double *x = malloc(sizeof(double) * K);
        for (int64_t k = 0; k < K; ++k)
            x[k] = q_value(qa, a[i * K + k]) * e8m0_value(sa[i * nb + k / 32]);
        const uint8_t *wj = w + (int64_t)j * N * K;
        const uint8_t *sj = sw + (int64_t)j * N * nb;
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += x[k] * (q_value(qw, wj[n * K + k]) * e8m0_value(sj[n * nb + k / 32]));
            out[r * N + n] = acc;
        }
        free(x);
    }
    return REF_OK;
}
