/*
 * nvfp4_oracle.c -- plain, slow, scalar CPU oracle for the rollout-side NVFP4 W4A4 linear
 * layer with Residual Activation Compensation (RAC).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or load this file;
 * only the test-suite, the smoke check and the benchmark's CPU-baseline leg use it.  It
 * shares no code, header, table or constant generator with the CUDA library.
 *
 * Source of the method: "QUADS: Stabilizing NVFP4 Reinforcement Learning for MoE via
 * QUantization-error Alignment across Dual Sides" (arXiv 2607.15810), cited below as QUADS.
 *   - §2.2 "FP8": E4M3 format, maximum magnitude 448.
 *   - §2.2 "FP4", Eq. (4): E2M1 elements on the grid {0,0.5,1,1.5,2,3,4,6} per sign,
 *     16 consecutive elements share one E4M3 block scale, plus one FP32 per-tensor scale.
 *   - §3.1 Eq. (7), (9): weight and activation QDQ operators Q_W, Q_A.
 *   - §3.2 Eq. (12), (15)-(16): the trainer's weight QDQ equals the rollout quantizer.
 *   - §3.3 Eq. (20)-(24): activation residual, RAC reconstruction, channel score, top-k.
 *
 * Readings of points the paper leaves open (each is stated where it is used):
 *   R1 E2M1 subnormal: exponent field 0 encodes 0 and 0.5 (bias 1), as the printed grid requires.
 *   R2 E2M1 rounding: nearest grid value, ties to the even magnitude index, |v| > 6 -> 6,
 *      and the sign bit of the input is kept (a negative value that rounds to 0 gives 0x8).
 *   R3 E4M3 rounding: nearest finite value, ties to the even code, anything above 448 -> 448.
 *   R4 Per-tensor scale: S_enc = fl(2688 / amax) (2688 = 448 * 6), S_dec = fl(1 / S_enc);
 *      amax == 0 gives S_enc = S_dec = 1.
 *   R5 Block scale: sb = e4m3(fl(fl(amax_b / 6) * S_enc)); element code
 *      q = e2m1(fl(x * fl(S_enc / sb))); sb == 0 gives code 0 (0x8 for a negative sign bit).
 *      The quotient fl(S_enc / sb) saturates at FLT_MAX like S_enc itself (R4): it can overflow
 *      only when S_enc was clamped (amax below 2688 / FLT_MAX) and sb < 1, and saturation keeps
 *      every product finite (x = 0 then encodes as a signed zero, never as the code of a NaN).
 *   R6 Dequantization: fl(V[q] * fl(sb * S_dec)).
 *   R7 Residual r = fl(x - DQ(Q(x))) (= -dX_q of Eq. (20)).  The channel score of Eq. (23) is
 *      the exact integer sum over rows of q^2 with q = rint(|r| * 2^(20 - E)) (nearest integer,
 *      ties to even), E = ilogb(amax) + 2.  Since |r| < 2^(E-1), q < 2^19 and the uint64 sum is
 *      exact and independent of summation order for up to 2^19 rows.  It ranks channels as the
 *      L2 norm does except between channels whose sums of r^2 differ by less than about
 *      M * amax^2 * 2^-17.
 *   R8 Top-k of Eq. (24) with an absolute channel count k; ties broken to the lower channel
 *      index; the selected indices are emitted in ascending order.
 *   R9 Second pass: the residual on the selected channels, gathered in ascending index order,
 *      is quantized with blocks of 16 gathered channels and the activation's own S_enc.
 *   R10 Weight tail: the weight columns that multiply the correction are the dequantized
 *      stored weights on the selected channels, re-quantized with the weight's own S_enc.
 *   R16 FP8 W8A8 baseline (§2.2 "FP8": "each tile of values carries its own alpha in
 *      Eq. (4)", tile sizes unstated): activation tiles of 1 x 128 (one row, 128 consecutive
 *      channels), weight tiles of 128 x 128 (128 output rows x 128 input channels); a tile cut
 *      by the matrix edge covers what is left.
 *   R17 FP8 tile scale alpha = 2^e, e the smallest integer with 448 * 2^e >= amax of the tile,
 *      clamped to [-127, 127] (an all-zero tile gets -127): a power of two, stored as the byte
 *      e + 127 (UE8M0).
 *   R18 FP8 element: E4M3 of x * 2^-e, nearest value, ties to the even code, sign kept (a
 *      negative value that rounds to zero gives 0x80); |x * 2^-e| <= 448 by R17.  The
 *      dequantized value V * 2^e is exact.
 *
 * Arithmetic: IEEE binary32 with round-to-nearest-even for every step the method performs in
 * FP32 (compile with -ffp-contract=off so that no multiply-add is fused); fp64 / exact
 * integers for reductions and the GEMM reference.
 */
#define _POSIX_C_SOURCE 200809L
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------------------------------
 * bf16 (the activation and weight storage type of the rollout path)
 * ---------------------------------------------------------------------------------------- */
static float bf16_value(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a binary32 value to the nearest bfloat16, ties to even (finite inputs). */
uint16_t oracle_bf16_round(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u) return (uint16_t)((u >> 16) | ((u & 0xffff) ? 0x40 : 0));
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

float oracle_bf16_value(uint16_t h) { return bf16_value(h); }

/* ------------------------------------------------------------------------------------------
 * E2M1 element format.  QUADS §2.2 "FP4": 1 sign, 2 exponent, 1 mantissa bit, Eq. (4) with
 * the subnormal of reading R1.  The code is sign << 3 | exponent << 1 | mantissa.
 * ---------------------------------------------------------------------------------------- */
double oracle_e2m1_value(uint8_t code)
{
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

/* Reading R2: nearest of the eight magnitudes, ties to the even magnitude index, sign kept. */
uint8_t oracle_e2m1_encode(float v)
{
    uint8_t sign = signbit(v) ? 8 : 0;
    double a = fabs((double)v);
    int best = 0;
    if (isinf(a)) {
        best = 7;
    } else {
        double bestd = INFINITY;
        for (int i = 0; i < 8; ++i) {
            double d = fabs(a - oracle_e2m1_value((uint8_t)i));
            if (d < bestd || (d == bestd && (i % 2) == 0)) {
                best = i;
                bestd = d;
            }
        }
    }
    return (uint8_t)(sign | best);
}

/* ------------------------------------------------------------------------------------------
 * E4M3 block-scale format.  QUADS §2.2 "FP8": b = 8, e = 4, three mantissa bits, maximum 448.
 * Bias 7, subnormals are multiples of 2^-9, S.1111.111 is NaN (no infinity).
 * ---------------------------------------------------------------------------------------- */
double oracle_e4m3_value(uint8_t b)
{
    int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
    if (e == 15 && m == 7) return NAN;
    double mag = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* Nearest finite non-negative E4M3 code to a >= 0, ties to the even code (readings R3, R18). */
static uint8_t e4m3_nearest(double a)
{
    int best = 0;
    double bestd = INFINITY;
    for (int c = 0; c <= 0x7e; ++c) {
        double d = fabs(a - oracle_e4m3_value((uint8_t)c));
        if (d < bestd || (d == bestd && (c % 2) == 0)) {
            best = c;
            bestd = d;
        }
    }
    return (uint8_t)best;
}

/* Reading R3: for t >= 0, nearest finite non-negative E4M3 value, ties to the even code. */
uint8_t oracle_e4m3_encode(float t) { return e4m3_nearest((double)t); }

/* ------------------------------------------------------------------------------------------
 * Per-tensor FP32 scale (QUADS §2.2 "FP4", the second scaling level; formula: reading R4).
 * ---------------------------------------------------------------------------------------- */
typedef struct {
    float amax;
    float s_enc;
    float s_dec;
    int32_t shift_e; /* E of reading R7 */
} oracle_tscale;

static oracle_tscale tscale_from_amax(float amax)
{
    oracle_tscale ts;
    ts.amax = amax;
    if (amax == 0.0f) {
        ts.s_enc = 1.0f;
        ts.s_dec = 1.0f;
        ts.shift_e = 0;
        return ts;
    }
    float s = 2688.0f / amax;
    if (isinf(s)) s = 3.4028234663852886e38f;
    ts.s_enc = s;
    ts.s_dec = 1.0f / s;
    ts.shift_e = ilogbf(amax) + 2;
    return ts;
}

void oracle_tensor_scale(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx,
                         oracle_tscale* out)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < rows; ++i)
        for (int64_t j = 0; j < cols; ++j) {
            float a = fabsf(bf16_value(x[i * ldx + j]));
            if (a > amax) amax = a;
        }
    *out = tscale_from_amax(amax);
}

void oracle_tensor_scale_from_amax(float amax, oracle_tscale* out) { *out = tscale_from_amax(amax); }

/* ------------------------------------------------------------------------------------------
 * One 16-element block (reading R5).  v: 16 binary32 values.  codes: 16 unpacked 4-bit codes.
 * ---------------------------------------------------------------------------------------- */
static void quantize_block16(const float* v, float s_enc, uint8_t* codes, uint8_t* sb_out)
{
    float amax_b = 0.0f;
    for (int i = 0; i < 16; ++i) {
        float a = fabsf(v[i]);
        if (a > amax_b) amax_b = a;
    }
    float t = amax_b / 6.0f;
    t = t * s_enc;
    uint8_t sb = oracle_e4m3_encode(t);
    *sb_out = sb;
    if (sb == 0) {
        for (int i = 0; i < 16; ++i) codes[i] = signbit(v[i]) ? 8 : 0;
        return;
    }
    float e_b = s_enc / (float)oracle_e4m3_value(sb);
    if (isinf(e_b)) e_b = 3.4028234663852886e38f; /* reading R5: saturates, as S_enc does (R4) */
    for (int i = 0; i < 16; ++i) {
        float y = v[i] * e_b;
        codes[i] = oracle_e2m1_encode(y);
    }
}

/* Reading R6. */
static float dequant_elem(uint8_t code, uint8_t sb, float s_dec)
{
    float d_b = (float)oracle_e4m3_value(sb) * s_dec;
    return (float)oracle_e2m1_value(code) * d_b;
}

static void put_code(uint8_t* row, int64_t j, uint8_t c)
{
    if (j % 2 == 0)
        row[j / 2] = (uint8_t)((row[j / 2] & 0xf0) | (c & 0x0f));
    else
        row[j / 2] = (uint8_t)((row[j / 2] & 0x0f) | (uint8_t)(c << 4));
}

static uint8_t get_code(const uint8_t* row, int64_t j)
{
    return (j % 2 == 0) ? (row[j / 2] & 0x0f) : (row[j / 2] >> 4);
}

uint8_t oracle_get_code(const uint8_t* row, int64_t j) { return get_code(row, j); }

/* ------------------------------------------------------------------------------------------
 * Q_A / Q_W (QUADS Eq. (7), (9), (12)): codes [rows][cols/2] with element 2i in the low
 * nibble, block scales [rows][cols/16], for a bf16 matrix with leading dimension ldx.
 * ---------------------------------------------------------------------------------------- */
void oracle_quantize(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx,
                     const oracle_tscale* ts, uint8_t* codes, int64_t ld_codes, uint8_t* scales,
                     int64_t ld_scales)
{
    float v[16];
    uint8_t q[16], sb;
    for (int64_t i = 0; i < rows; ++i)
        for (int64_t b = 0; b < cols / 16; ++b) {
            for (int l = 0; l < 16; ++l) v[l] = bf16_value(x[i * ldx + b * 16 + l]);
            quantize_block16(v, ts->s_enc, q, &sb);
            scales[i * ld_scales + b] = sb;
            for (int l = 0; l < 16; ++l) put_code(codes + i * ld_codes, b * 16 + l, q[l]);
        }
}

/* DQ of an NVFP4 matrix into fp32 (reading R6); used for W-hat of the trainer path. */
void oracle_dequantize(const uint8_t* codes, int64_t ld_codes, const uint8_t* scales,
                       int64_t ld_scales, int64_t rows, int64_t cols, float s_dec, float* out,
                       int64_t ld_out)
{
    for (int64_t i = 0; i < rows; ++i)
        for (int64_t j = 0; j < cols; ++j)
            out[i * ld_out + j] =
                dequant_elem(get_code(codes + i * ld_codes, j), scales[i * ld_scales + j / 16], s_dec);
}

/* ------------------------------------------------------------------------------------------
 * Residual R = X - DQ(Q(X)) (QUADS Eq. (20), sign of reading R7), binary32, [rows][cols].
 * ---------------------------------------------------------------------------------------- */
void oracle_residual(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx,
                     const oracle_tscale* ts, float* r, int64_t ld_r)
{
    float v[16];
    uint8_t q[16], sb;
    for (int64_t i = 0; i < rows; ++i)
        for (int64_t b = 0; b < cols / 16; ++b) {
            for (int l = 0; l < 16; ++l) v[l] = bf16_value(x[i * ldx + b * 16 + l]);
            quantize_block16(v, ts->s_enc, q, &sb);
            for (int l = 0; l < 16; ++l) r[i * ld_r + b * 16 + l] = v[l] - dequant_elem(q[l], sb, ts->s_dec);
        }
}

/* Channel score of QUADS Eq. (23) in the exact integer form of reading R7. */
void oracle_scores(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx,
                   const oracle_tscale* ts, uint64_t* scores)
{
    float* r = (float*)malloc(sizeof(float) * (size_t)cols);
    for (int64_t j = 0; j < cols; ++j) scores[j] = 0;
    for (int64_t i = 0; i < rows; ++i) {
        oracle_residual(x + i * ldx, 1, cols, ldx, ts, r, cols);
        for (int64_t j = 0; j < cols; ++j) {
            double q = rint(ldexp(fabs((double)r[j]), 20 - ts->shift_e));
            scores[j] += (uint64_t)q * (uint64_t)q;
        }
    }
    free(r);
}

/* ------------------------------------------------------------------------------------------
 * Channel selection S = TopK (QUADS Eq. (24)), reading R8.
 * ---------------------------------------------------------------------------------------- */
static const uint64_t* g_sort_scores;
static int cmp_desc_score_asc_index(const void* pa, const void* pb)
{
    int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
    uint64_t sa = g_sort_scores[a], sb = g_sort_scores[b];
    if (sa != sb) return sa > sb ? -1 : 1;
    return a < b ? -1 : (a > b ? 1 : 0);
}
static int cmp_int32(const void* pa, const void* pb)
{
    int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
    return a < b ? -1 : (a > b ? 1 : 0);
}

void oracle_topk(const uint64_t* scores, int64_t n, int32_t k, int32_t* idx)
{
    int32_t* order = (int32_t*)malloc(sizeof(int32_t) * (size_t)n);
    for (int64_t j = 0; j < n; ++j) order[j] = (int32_t)j;
    g_sort_scores = scores;
    qsort(order, (size_t)n, sizeof(int32_t), cmp_desc_score_asc_index);
    for (int32_t i = 0; i < k; ++i) idx[i] = order[i];
    qsort(idx, (size_t)k, sizeof(int32_t), cmp_int32);
    free(order);
}

/* ------------------------------------------------------------------------------------------
 * RAC second pass (QUADS Eq. (21), reading R9): the residual on the selected channels,
 * quantized into k extra K-columns.  tail codes [rows][k/2], tail scales [rows][k/16].
 * ---------------------------------------------------------------------------------------- */
void oracle_rac_tail(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx,
                     const oracle_tscale* ts, const int32_t* idx, int32_t k, uint8_t* tcodes,
                     int64_t ld_tcodes, uint8_t* tscales, int64_t ld_tscales)
{
    float* r = (float*)malloc(sizeof(float) * (size_t)cols);
    float v[16];
    uint8_t q[16], sb;
    for (int64_t i = 0; i < rows; ++i) {
        oracle_residual(x + i * ldx, 1, cols, ldx, ts, r, cols);
        for (int32_t b = 0; b < k / 16; ++b) {
            for (int l = 0; l < 16; ++l) v[l] = r[idx[b * 16 + l]];
            quantize_block16(v, ts->s_enc, q, &sb);
            tscales[i * ld_tscales + b] = sb;
            for (int l = 0; l < 16; ++l) put_code(tcodes + i * ld_tcodes, b * 16 + l, q[l]);
        }
    }
    free(r);
}

/* Weight tail (reading R10): W'_S = Q(DQ(W_q)[:, S]) with the weight's S_enc. */
void oracle_weight_tail(const uint8_t* wcodes, int64_t ld_wcodes, const uint8_t* wscales,
                        int64_t ld_wscales, int64_t rows, const oracle_tscale* wts,
                        const int32_t* idx, int32_t k, uint8_t* tcodes, int64_t ld_tcodes,
                        uint8_t* tscales, int64_t ld_tscales)
{
    float v[16];
    uint8_t q[16], sb;
    for (int64_t n = 0; n < rows; ++n)
        for (int32_t b = 0; b < k / 16; ++b) {
            for (int l = 0; l < 16; ++l) {
                int32_t j = idx[b * 16 + l];
                v[l] = dequant_elem(get_code(wcodes + n * ld_wcodes, j), wscales[n * ld_wscales + j / 16],
                                    wts->s_dec);
            }
            quantize_block16(v, wts->s_enc, q, &sb);
            tscales[n * ld_tscales + b] = sb;
            for (int l = 0; l < 16; ++l) put_code(tcodes + n * ld_tcodes, b * 16 + l, q[l]);
        }
}

/* ------------------------------------------------------------------------------------------
 * Block-scaled FP4 GEMM reference (QUADS §3.3 "Targeted residual compensation": the main and
 * the correction terms run as one native W4A4 product over K + k columns).
 *
 * y[m,n] = S_dec,a * S_dec,b * sum_c V[a_mc] sa_m,c/16 * V[b_nc] sb_n,c/16, evaluated exactly:
 * 2V is an integer in [-12, 12] and 2^9 * sb is an integer <= 229376, so the sum is an exact
 * int64 (|term| < 2^43, at most 2^13 terms); the only rounding is the final fp64 scaling.
 * Evaluated at the (m, n) pairs given (row indices into A, row indices into B).
 * ---------------------------------------------------------------------------------------- */
typedef struct gemm_job {
    const uint8_t *a_codes, *a_scales, *b_codes, *b_scales;
    int64_t lda, ld_as, ldb, ld_bs, ktot;
    double s_dec_a, s_dec_b;
    const int64_t *mi, *ni;
    int64_t p0, p1;
    double* y;
} gemm_job;

static void gemm_pair_range(const gemm_job* j)
{
    const uint8_t *a_codes = j->a_codes, *a_scales = j->a_scales, *b_codes = j->b_codes, *b_scales = j->b_scales;
    const int64_t lda = j->lda, ld_as = j->ld_as, ldb = j->ldb, ld_bs = j->ld_bs, ktot = j->ktot;
    const int64_t *mi = j->mi, *ni = j->ni;
    double* y = j->y;
    for (int64_t p = j->p0; p < j->p1; ++p) {
        const uint8_t* ar = a_codes + mi[p] * lda;
        const uint8_t* br = b_codes + ni[p] * ldb;
        const uint8_t* as = a_scales + mi[p] * ld_as;
        const uint8_t* bs = b_scales + ni[p] * ld_bs;
        int64_t acc = 0;
        for (int64_t c = 0; c < ktot; ++c) {
            int64_t va = (int64_t)llround(2.0 * oracle_e2m1_value(get_code(ar, c)));
            int64_t vb = (int64_t)llround(2.0 * oracle_e2m1_value(get_code(br, c)));
            int64_t sa = (int64_t)llround(ldexp(oracle_e4m3_value(as[c / 16]), 9));
            int64_t sbv = (int64_t)llround(ldexp(oracle_e4m3_value(bs[c / 16]), 9));
            acc += va * vb * sa * sbv;
        }
        y[p] = ldexp((double)acc, -20) * j->s_dec_a * j->s_dec_b;
    }
}

static void* gemm_thread(void* arg)
{
    gemm_pair_range((const gemm_job*)arg);
    return NULL;
}

/* Host threads the pairs are spread over (1 by default).  Every pair is computed by one thread
 * with the same arithmetic, so the result does not depend on the count. */
static int g_threads = 1;

void oracle_set_threads(int n) { g_threads = n < 1 ? 1 : (n > 1024 ? 1024 : n); }

int oracle_hardware_threads(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n < 1 ? 1 : (int)n;
}

void oracle_gemm_pairs(const uint8_t* a_codes, int64_t lda, const uint8_t* a_scales, int64_t ld_as,
                       const uint8_t* b_codes, int64_t ldb, const uint8_t* b_scales, int64_t ld_bs,
                       int64_t ktot, double s_dec_a, double s_dec_b, const int64_t* mi,
                       const int64_t* ni, int64_t npairs, double* y)
{
    gemm_job base = {a_codes, a_scales, b_codes, b_scales, lda, ld_as, ldb, ld_bs, ktot, s_dec_a, s_dec_b,
                     mi, ni, 0, npairs, y};
    int nt = g_threads;
    if ((int64_t)nt > npairs / 16) nt = (int)(npairs / 16);
    if (nt <= 1) {
        gemm_pair_range(&base);
        return;
    }
    gemm_job jobs[1024];
    pthread_t tids[1024];
    int created[1024];
    for (int t = 0; t < nt; ++t) {
        jobs[t] = base;
        jobs[t].p0 = npairs * t / nt;
        jobs[t].p1 = npairs * (t + 1) / nt;
        created[t] = t > 0 && pthread_create(&tids[t], NULL, gemm_thread, &jobs[t]) == 0;
        if (t > 0 && !created[t]) gemm_pair_range(&jobs[t]);  /* no thread: compute it here */
    }
    gemm_pair_range(&jobs[0]);
    for (int t = 1; t < nt; ++t)
        if (created[t]) pthread_join(tids[t], NULL);
}

/* The same product as plain fp64 arithmetic on the dequantized operands (cross-check). */
void oracle_gemm_pairs_fp64(const uint8_t* a_codes, int64_t lda, const uint8_t* a_scales,
                            int64_t ld_as, const uint8_t* b_codes, int64_t ldb,
                            const uint8_t* b_scales, int64_t ld_bs, int64_t ktot, double s_dec_a,
                            double s_dec_b, const int64_t* mi, const int64_t* ni, int64_t npairs,
                            double* y)
{
    for (int64_t p = 0; p < npairs; ++p) {
        double acc = 0.0;
        for (int64_t c = 0; c < ktot; ++c) {
            double a = oracle_e2m1_value(get_code(a_codes + mi[p] * lda, c)) *
                       oracle_e4m3_value(a_scales[mi[p] * ld_as + c / 16]) * s_dec_a;
            double b = oracle_e2m1_value(get_code(b_codes + ni[p] * ldb, c)) *
                       oracle_e4m3_value(b_scales[ni[p] * ld_bs + c / 16]) * s_dec_b;
            acc += a * b;
        }
        y[p] = acc;
    }
}

/* ------------------------------------------------------------------------------------------
 * MoE routing plumbing (not described by the paper; the expert layer of its MoE model).
 * Dispatch: stable counting sort of the (token, slot) pairs by expert, ascending (token, slot)
 * inside an expert.  grp_off[G+1] are unpadded offsets, row_src[r] = token * topk + slot.
 * ---------------------------------------------------------------------------------------- */
void oracle_moe_dispatch(const int32_t* topk_ids, int64_t tokens, int32_t topk, int32_t groups,
                         int64_t* grp_off, int32_t* row_src)
{
    int64_t* fill = (int64_t*)calloc((size_t)groups + 1, sizeof(int64_t));
    for (int32_t g = 0; g <= groups; ++g) grp_off[g] = 0;
    for (int64_t t = 0; t < tokens * topk; ++t) grp_off[topk_ids[t] + 1] += 1;
    for (int32_t g = 0; g < groups; ++g) grp_off[g + 1] += grp_off[g];
    for (int64_t t = 0; t < tokens; ++t)
        for (int32_t s = 0; s < topk; ++s) {
            int32_t e = topk_ids[t * topk + s];
            row_src[grp_off[e] + fill[e]] = (int32_t)(t * topk + s);
            fill[e] += 1;
        }
    free(fill);
}

/* SwiGLU of the expert MLP: silu(g) * u with silu(g) = g / (1 + exp(-g)), fp64. */
double oracle_swiglu(double g, double u) { return g / (1.0 + exp(-g)) * u; }

/* Combine: out[t] = bf16( sum over slots, in slot order, of y[pos(t, s)] in binary32 ). */
void oracle_moe_combine(const uint16_t* y, int64_t ldy, const int64_t* pos, int64_t tokens,
                        int32_t topk, int64_t hidden, uint16_t* out, int64_t ldo)
{
    for (int64_t t = 0; t < tokens; ++t)
        for (int64_t h = 0; h < hidden; ++h) {
            float acc = 0.0f;
            for (int32_t s = 0; s < topk; ++s) acc += bf16_value(y[pos[t * topk + s] * ldy + h]);
            out[t * ldo + h] = oracle_bf16_round(acc);
        }
}

/* ------------------------------------------------------------------------------------------
 * Array forms of the element codecs, for exhaustive checks from Python.
 * ---------------------------------------------------------------------------------------- */
void oracle_e2m1_encode_array(const float* v, int64_t n, uint8_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e2m1_encode(v[i]);
}

void oracle_e4m3_encode_array(const float* t, int64_t n, uint8_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(t[i]);
}

void oracle_bf16_round_array(const float* f, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_round(f[i]);
}

/* One block of reading R5 from Python: v[16] -> codes[16] (unpacked) and the scale byte. */
void oracle_quantize_block16(const float* v, float s_enc, uint8_t* codes, uint8_t* sb)
{
    quantize_block16(v, s_enc, codes, sb);
}

/* ------------------------------------------------------------------------------------------
 * FP8 W8A8 with fine-grained tile scaling, the comparison baseline of QUADS §2.2 "FP8" and
 * §4.4.2 (readings R16-R18).
 * ---------------------------------------------------------------------------------------- */

/* Reading R17, by search: the smallest e in [-127, 127] with 448 * 2^e >= amax. */
int32_t oracle_fp8_scale_exponent(double amax)
{
    if (!(amax > 0.0)) return -127;
    int32_t e = -127;
    while (e < 127 && ldexp(448.0, e) < amax) ++e;
    return e;
}

/* Reading R18 for a value already divided by its tile scale: sign bit, then the nearest
 * magnitude code. */
uint8_t oracle_fp8_encode(double v)
{
    uint8_t mag = e4m3_nearest(fabs(v));
    return (uint8_t)(signbit(v) ? (mag | 0x80u) : mag);
}

/* Tiles of tile_rows x 128 (tile_rows 1: activations, 128: weights), row-major codes
 * [rows][ld_codes] and one UE8M0 byte per tile in scales[row tile][column tile]. */
void oracle_fp8_quantize(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx, int32_t tile_rows,
                         uint8_t* codes, int64_t ld_codes, uint8_t* scales, int64_t ld_scales)
{
    for (int64_t r0 = 0; r0 < rows; r0 += tile_rows)
        for (int64_t c0 = 0; c0 < cols; c0 += 128) {
            const int64_t r1 = r0 + tile_rows < rows ? r0 + tile_rows : rows;
            const int64_t c1 = c0 + 128 < cols ? c0 + 128 : cols;
            double amax = 0.0;
            for (int64_t i = r0; i < r1; ++i)
                for (int64_t j = c0; j < c1; ++j) {
                    const double a = fabs((double)bf16_value(x[i * ldx + j]));
                    if (a > amax) amax = a;
                }
            const int32_t e = oracle_fp8_scale_exponent(amax);
            scales[(r0 / tile_rows) * ld_scales + c0 / 128] = (uint8_t)(e + 127);
            for (int64_t i = r0; i < r1; ++i)
                for (int64_t j = c0; j < c1; ++j)
                    codes[i * ld_codes + j] = oracle_fp8_encode(ldexp((double)bf16_value(x[i * ldx + j]), -e));
        }
}

/* V * 2^e in fp64, out [rows][ld_out]. */
void oracle_fp8_dequantize(const uint8_t* codes, int64_t ld_codes, const uint8_t* scales, int64_t ld_scales,
                           int64_t rows, int64_t cols, int32_t tile_rows, double* out, int64_t ld_out)
{
    for (int64_t i = 0; i < rows; ++i)
        for (int64_t j = 0; j < cols; ++j) {
            const int32_t e = (int32_t)scales[(i / tile_rows) * ld_scales + j / 128] - 127;
            out[i * ld_out + j] = ldexp(oracle_e4m3_value(codes[i * ld_codes + j]), e);
        }
}
