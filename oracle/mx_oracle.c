/*
 * mx_oracle.c -- the plain, slow, single-threaded CPU oracle for the
 * block-float decode-in-kernel matmul (MXFP4 / MXFP8 / NVFP4 weights,
 * bf16 activations).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only the test suite, the package's smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no code, header, table or
 * constant with the CUDA library.
 *
 * Sources followed (cited by page title and section):
 *  - "MLxcel 0.8 release" (backend.ai blog), section "Decoding block-float
 *    formats in software" (블록 부동소수점 형식을 소프트웨어로 디코드하기), and the
 *    talk "High-performance LLM/VLM inference on AMD Strix Halo with mlxcel
 *    engine", slide 12 "Software Decode for Block Float Formats":
 *    MXFP4, MXFP8 and NVFP4 share one scale per block; weights are decoded
 *    inside the kernel and then multiplied; an E2M1 value is 1 sign bit,
 *    2 exponent bits and 1 mantissa bit, and the decode is exact.
 *  - Where the pages are silent (E8M0 and E4M3 definitions, block sizes,
 *    packing order, the NVFP4 per-tensor scale) the oracle follows the
 *    plain readings listed in the repository's design notes: OCP MX v1.0
 *    (E8M0 = 2^(e-127), 0xFF = NaN; MX block = 32), NVFP4 (E4M3 scale per
 *    16 elements times one fp32 per-tensor scale), E4M3 "FN" (bias 7, no
 *    infinities, S.1111.111 = NaN), element k of a row in byte k/2 with
 *    even k in the low nibble, scales row-major [N][K/block].
 *
 * Arithmetic: every decoded weight is the exact real value of
 * code x scale, rounded once to fp32 (it is exact for every finite case
 * except overflow and the NVFP4 per-tensor multiply, which is one
 * round-to-nearest-even fp32 multiply).  Products are accumulated in fp64
 * in increasing k order.  Build with -O2 -ffp-contract=off and no
 * fast-math, so the C compiler keeps every operation as written.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_FMT_MXFP4 = 0, OR_FMT_MXFP8 = 1, OR_FMT_NVFP4 = 2 };

/* ---------------------------------------------------------------- formats */

/* E2M1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.
 * Exponent 0 is the subnormal range 0.5*m; otherwise 2^(e-1)*(1+m/2).
 * Bias 1 is what makes the pages' fp16 bit placement exact: fp16 has bias
 * 15, and the single corrective multiply is by 2^14 = 2^(15-1). */
double or_e2m1(unsigned code)
{
#ifdef OR_PLANT_E2M1_BIAS0
    const int bias = 0;
#else
    const int bias = 1;
#endif
    unsigned s = (code >> 3) & 1u;
    unsigned e = (code >> 1) & 3u;
    unsigned m = code & 1u;
    double mag = (e == 0) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, (int)e - bias);
#ifdef OR_PLANT_E2M1_NOSIGN
    s = 0;
#endif
    return s ? -mag : mag;
}

/* E8M0 block scale: 2^(e-127) for e in 0..254, NaN for 0xFF. */
double or_e8m0(unsigned e)
{
    e &= 0xFFu;
    if (e == 0xFFu) return NAN;
#ifdef OR_PLANT_E8M0_BIAS128
    return ldexp(1.0, (int)e - 128);
#else
    return ldexp(1.0, (int)e - 127);
#endif
}

/* E4M3 (the "FN" variant): bit 7 sign, bits 6..3 exponent (bias 7),
 * bits 2..0 mantissa.  Exponent 0 is subnormal 2^-6 * m/8.  No infinities;
 * exponent 15 with mantissa 7 is NaN, so the largest finite value is
 * 1.75 * 2^8 = 448. */
double or_e4m3(unsigned b)
{
    b &= 0xFFu;
    unsigned s = (b >> 7) & 1u;
    unsigned e = (b >> 3) & 15u;
    unsigned m = b & 7u;
    if (e == 15u && m == 7u) return NAN;
    double mag = (e == 0) ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return s ? -mag : mag;
}

/* bf16 bit pattern -> exact value (bf16 is the top half of an fp32). */
double or_bf16(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a real (held exactly in a double) to bf16, nearest-even, with
 * gradual underflow and overflow to infinity.  bf16 keeps 8 significant
 * bits and fp32's exponent range: normal quantum 2^(e-7) for |v| in
 * [2^e, 2^(e+1)), subnormal quantum 2^-133 below 2^-126. */
uint16_t or_round_bf16(double v)
{
    if (isnan(v)) return 0x7FC0u;
    double a = fabs(v);
    double r;
    if (a == 0.0 || isinf(v)) {
        r = a;
    } else {
        int e;
        (void)frexp(a, &e);             /* a = f * 2^e with f in [0.5, 1) */
        int qexp = (e - 1) - 7;         /* quantum of an 8-significant-bit value */
        if (qexp < -133) qexp = -133;   /* subnormal range */
        double n = nearbyint(ldexp(a, -qexp)); /* default rounding: to nearest, ties to even */
        r = ldexp(n, qexp);
        if (r >= ldexp(1.0, 128)) r = INFINITY;
    }
    float f = (float)r;                 /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    u >>= 16;
    if (signbit(v)) u |= 0x8000u;
    return (uint16_t)u;
}

/* ------------------------------------------------------------- dequantise */

static int block_of(int fmt) { return fmt == OR_FMT_NVFP4 ? 16 : 32; }

/* Code of element k in row n of a [N][K] weight (no scale). */
static double code_value(int fmt, const uint8_t *codes, int64_t n, int64_t k, int64_t K)
{
    if (fmt == OR_FMT_MXFP8) {
        return or_e4m3(codes[n * K + k]);
    }
    uint8_t byte = codes[n * (K / 2) + k / 2];
#ifdef OR_PLANT_NIBBLE_SWAP
    unsigned nib = (k % 2 == 0) ? (byte >> 4) : (byte & 0xFu);
#else
    unsigned nib = (k % 2 == 0) ? (byte & 0xFu) : (byte >> 4);
#endif
    return or_e2m1(nib);
}

/* Block scale of element k in row n (without the NVFP4 tensor scale);
 * scales are row-major [N][K/block]. */
static double block_scale(int fmt, const uint8_t *scales, int64_t n, int64_t k, int64_t N,
                          int64_t K)
{
    int blk = block_of(fmt);
#ifdef OR_PLANT_SCALE_COLMAJOR
    uint8_t s = scales[(k / blk) * N + n];
#else
    (void)N;
    uint8_t s = scales[n * (K / blk) + k / blk];
#endif
    return fmt == OR_FMT_NVFP4 ? or_e4m3(s) : or_e8m0(s);
}

/* NVFP4 per-tensor fp32 scale, stored little-endian right after the
 * [N][K/16] block-scale bytes. */
static float tensor_scale(const uint8_t *scales, int64_t N, int64_t K)
{
    float g;
    memcpy(&g, scales + N * (K / 16), sizeof g);
    return g;
}

/* One decoded weight, as fp32.  MXFP4 / MXFP8: fp32(code * 2^(e-127)),
 * exact unless it overflows.  NVFP4: fp32(fp32(code * s) * g), where
 * code * s is exact (at most 6 significant bits) and the multiply by the
 * fp32 tensor scale g rounds once. */
static float weight(int fmt, const uint8_t *codes, const uint8_t *scales, float g,
                    int64_t n, int64_t k, int64_t N, int64_t K)
{
    double v = code_value(fmt, codes, n, k, K) * block_scale(fmt, scales, n, k, N, K);
    float w = (float)v;
    if (fmt == OR_FMT_NVFP4) {
        /* the exact product of two fp32 values fits a double; one rounding */
        w = (float)((double)w * (double)g);
    }
    return w;
}

/* W[n][k] for the whole [N][K] matrix, fp32. */
int or_dequant(int fmt, const uint8_t *codes, const uint8_t *scales, float *W,
               int64_t N, int64_t K)
{
    if (fmt < 0 || fmt > 2 || N < 0 || K < 0 || K % block_of(fmt) != 0) return -1;
    float g = fmt == OR_FMT_NVFP4 ? tensor_scale(scales, N, K) : 1.0f;
    for (int64_t n = 0; n < N; n++)
        for (int64_t k = 0; k < K; k++)
            W[n * K + k] = weight(fmt, codes, scales, g, n, k, N, K);
    return 0;
}

/* ------------------------------------------------------------------- qmv */

/* Dot product of one decoded weight row with one bf16 activation row,
 * accumulated in fp64 in increasing k. */
static double row_dot(const float *wrow, const uint16_t *xrow, int64_t K)
{
    double acc = 0.0;
#ifdef OR_PLANT_DROP_LAST
    K -= 1;
#endif
    for (int64_t k = 0; k < K; k++)
        acc += (double)wrow[k] * or_bf16(xrow[k]);
    return acc;
}

static void dequant_row(int fmt, const uint8_t *codes, const uint8_t *scales, float g,
                        int64_t n, int64_t N, int64_t K, float *wrow)
{
    for (int64_t k = 0; k < K; k++) wrow[k] = weight(fmt, codes, scales, g, n, k, N, K);
}

/* Entries r0 .. r1-1 of the row list: y[m][r] = sum_k x[m][k] * W[rows[r]][k]
 * (rows[r] = r when rows == NULL), y fp64 [M][nrows]. */
static int qmv_row_range(int fmt, const uint8_t *codes, const uint8_t *scales, const uint16_t *x,
                         double *y, int64_t M, int64_t N, int64_t K, const int64_t *rows, int64_t nrows,
                         int64_t r0, int64_t r1)
{
    float g = fmt == OR_FMT_NVFP4 ? tensor_scale(scales, N, K) : 1.0f;
    float *wrow = (float *)malloc((size_t)K * sizeof(float));
    if (!wrow) return -2;
    for (int64_t r = r0; r < r1; r++) {
        int64_t n = rows ? rows[r] : r;
        if (n < 0 || n >= N) { free(wrow); return -1; }
        dequant_row(fmt, codes, scales, g, n, N, K, wrow);
        for (int64_t m = 0; m < M; m++) y[m * nrows + r] = row_dot(wrow, x + m * K, K);
    }
    free(wrow);
    return 0;
}

/* y[m][r] = sum_k x[m][k] * W[rows[r]][k] for a chosen list of weight rows
 * (all rows when rows == NULL).  x is bf16 [M][K]; y is fp64 [M][nrows]. */
int or_qmv_rows(int fmt, const uint8_t *codes, const uint8_t *scales, const uint16_t *x,
                double *y, int64_t M, int64_t N, int64_t K, const int64_t *rows, int64_t nrows)
{
    if (fmt < 0 || fmt > 2 || M < 0 || N < 0 || K <= 0 || K % block_of(fmt) != 0) return -1;
    if (rows == NULL) nrows = N;
    return qmv_row_range(fmt, codes, scales, x, y, M, N, K, rows, nrows, 0, nrows);
}

/* The same on several host threads: the row list is cut into nthreads
 * contiguous ranges, each computed by the routine above (same operations in
 * the same order per row, so the result is bit for bit that of or_qmv_rows).
 * Used to time the oracle on every core of a host; nthreads < 1 means 1. */
struct or_rows_job {
    int fmt;
    const uint8_t *codes, *scales;
    const uint16_t *x;
    double *y;
    int64_t M, N, K, nrows, r0, r1;
    const int64_t *rows;
    int rc;
};

static void *or_rows_worker(void *arg)
{
    struct or_rows_job *j = (struct or_rows_job *)arg;
    j->rc = qmv_row_range(j->fmt, j->codes, j->scales, j->x, j->y, j->M, j->N, j->K, j->rows, j->nrows, j->r0,
                          j->r1);
    return NULL;
}

int or_qmv_rows_mt(int fmt, const uint8_t *codes, const uint8_t *scales, const uint16_t *x, double *y,
                   int64_t M, int64_t N, int64_t K, const int64_t *rows, int64_t nrows, int nthreads)
{
    if (fmt < 0 || fmt > 2 || M < 0 || N < 0 || K <= 0 || K % block_of(fmt) != 0) return -1;
    if (rows == NULL) nrows = N;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (nthreads > nrows) nthreads = nrows > 0 ? (int)nrows : 1;
    pthread_t tid[256];
    int created[256];
    struct or_rows_job job[256];
    for (int t = 0; t < nthreads; t++) {
        job[t] = (struct or_rows_job){fmt, codes, scales, x, y, M, N, K, nrows,
                                      nrows * t / nthreads, nrows * (t + 1) / nthreads, rows, 0};
        created[t] = 0;
    }
    /* range 0 runs on the calling thread; a range whose thread cannot be
     * started runs there too */
    for (int t = 1; t < nthreads; t++)
        created[t] = pthread_create(&tid[t], NULL, or_rows_worker, &job[t]) == 0;
    or_rows_worker(&job[0]);
    for (int t = 1; t < nthreads; t++) {
        if (created[t]) pthread_join(tid[t], NULL);
        else or_rows_worker(&job[t]);
    }
    int rc = 0;
    for (int t = 0; t < nthreads; t++)
        if (job[t].rc != 0) rc = job[t].rc;
    return rc;
}

/* Decode GEMV: y[m][n] = sum_k x[m][k] * W[n][k], y fp64 [M][N]. */
int or_qmv(int fmt, const uint8_t *codes, const uint8_t *scales, const uint16_t *x,
           double *y, int64_t M, int64_t N, int64_t K)
{
    return or_qmv_rows(fmt, codes, scales, x, y, M, N, K, NULL, N);
}

/* Prefill GEMM, same definition over all M rows; also usable on chosen
 * (m, n) points so that full-size outputs can be spot-checked:
 * y[p] = sum_k x[ms[p]][k] * W[ns[p]][k]. */
int or_qmm_points(int fmt, const uint8_t *codes, const uint8_t *scales, const uint16_t *x,
                  int64_t M, int64_t N, int64_t K, const int64_t *ms, const int64_t *ns,
                  int64_t npts, double *y)
{
    if (fmt < 0 || fmt > 2 || M <= 0 || N <= 0 || K <= 0 || K % block_of(fmt) != 0) return -1;
    float g = fmt == OR_FMT_NVFP4 ? tensor_scale(scales, N, K) : 1.0f;
    float *wrow = (float *)malloc((size_t)K * sizeof(float));
    if (!wrow) return -2;
    int64_t cur = -1;
    for (int64_t p = 0; p < npts; p++) {
        if (ms[p] < 0 || ms[p] >= M || ns[p] < 0 || ns[p] >= N) { free(wrow); return -1; }
        if (ns[p] != cur) { dequant_row(fmt, codes, scales, g, ns[p], N, K, wrow); cur = ns[p]; }
        y[p] = row_dot(wrow, x + ms[p] * K, K);
    }
    free(wrow);
    return 0;
}

/* ------------------------------------------------------------------- MoE */

/* MoE decode GEMV over routed experts:
 *   y[t][j][n] = sum_k x[t][k] * W_{ids[t][j]}[n][k]
 * Expert e's codes start at e * N * (bytes per row) and its block scales at
 * e * N * (K / block); for NVFP4 the E per-tensor fp32 scales follow the
 * whole [E][N][K/16] scale block, one per expert.  Returns -3 (and leaves
 * that slot's outputs untouched) for an id outside [0, E). */
int or_moe_qmv(int fmt, const uint8_t *ecodes, const uint8_t *escales, const uint16_t *x,
               const int32_t *ids, double *y, int64_t T, int64_t E, int64_t topk,
               int64_t N, int64_t K)
{
    if (fmt < 0 || fmt > 2 || T < 0 || E <= 0 || topk <= 0 || N <= 0 || K <= 0 ||
        K % block_of(fmt) != 0)
        return -1;
    int blk = block_of(fmt);
    int64_t row_bytes = fmt == OR_FMT_MXFP8 ? K : K / 2;
    int64_t code_stride = N * row_bytes;
    int64_t scale_stride = N * (K / blk);
    float *wrow = (float *)malloc((size_t)K * sizeof(float));
    if (!wrow) return -2;
    int rc = 0;
    for (int64_t t = 0; t < T; t++) {
        for (int64_t j = 0; j < topk; j++) {
            int64_t e = ids[t * topk + j];
            if (e < 0 || e >= E) { rc = -3; continue; }
            const uint8_t *c = ecodes + e * code_stride;
            const uint8_t *s = escales + e * scale_stride;
            float g = 1.0f;
            if (fmt == OR_FMT_NVFP4) memcpy(&g, escales + E * scale_stride + 4 * e, sizeof g);
            for (int64_t n = 0; n < N; n++) {
                dequant_row(fmt, c, s, g, n, N, K, wrow);
                y[(t * topk + j) * N + n] = row_dot(wrow, x + t * K, K);
            }
        }
    }
    free(wrow);
    return rc;
}

/* ------------------------------------------------- MoE FFN glue (SwiGLU) */

/* h[q][i] = bf16_rne( silu(gate) * up ), gate = gu[q][i], up = gu[q][I + i],
 * silu(v) = v / (1 + exp(-v)), all in fp64 before the single bf16 rounding.
 * gu is [Q][2I] (gate rows then up rows, as one concatenated projection);
 * h is bf16 bits [Q][I]. */
int or_swiglu_bf16(const double *gu, uint16_t *h, int64_t Q, int64_t I)
{
    for (int64_t q = 0; q < Q; q++) {
        for (int64_t i = 0; i < I; i++) {
            double g = gu[q * 2 * I + i];
            double u = gu[q * 2 * I + I + i];
            double s = g / (1.0 + exp(-g));
            h[q * I + i] = or_round_bf16(s * u);
        }
    }
    return 0;
}

/* out[t][n] = sum_j r[t][j] * yd[t*topk + j][n], fp64, increasing j. */
int or_moe_combine(const double *yd, const float *r, double *out, int64_t T, int64_t topk,
                   int64_t N)
{
    for (int64_t t = 0; t < T; t++) {
        for (int64_t n = 0; n < N; n++) {
            double acc = 0.0;
            for (int64_t j = 0; j < topk; j++)
                acc += (double)r[t * topk + j] * yd[(t * topk + j) * N + n];
            out[t * N + n] = acc;
        }
    }
    return 0;
}

/* ------------------------------------------------------------- quantise */

/* bf16 activations -> block-float codes and scales: the reverse of the
 * decode above.  The pages say only that block-float quantisation runs on
 * the GPU's hardware NVFP4 / MXFP4 converter on Blackwell (manual page
 * "Building from source", CUDA build options, "GPU architecture
 * auto-detection") and that FP8 block checkpoints are re-quantised to MXFP8
 * (manual, ROCm status table).  The procedure is the plain reading of the
 * format definitions:
 *  - MXFP4 / MXFP8 (OCP MX v1.0 conversion): per block of 32, shared
 *    exponent e = floor(log2(amax)) - emax_elem (emax_elem = 2 for E2M1,
 *    8 for E4M3), clamped to [-127, 127], amax = 0 giving -127; scale byte
 *    e + 127; each element x / 2^e rounded to nearest-even in the element
 *    format, saturating at the largest finite value.  A block holding a NaN
 *    or an infinity gets scale 0xFF (NaN) and zero codes.
 *  - NVFP4: g = fp32(G / 2688) with G the largest finite |x| of the whole
 *    tensor (g = 1 when G = 0), stored after the scales as the tensor scale;
 *    per block of 16, s = E4M3(fp32(amax / fp32(6 g))) (nearest-even,
 *    saturating) and each element fp32(x / fp32(s g)) rounded to E2M1 (all
 *    codes zero when s g = 0); a block holding a NaN or an infinity gets
 *    scale 0x7F (NaN) and zero codes.
 *  - A zero result is stored as +0 (code 0), whatever the sign of x.
 * The fp32 steps of NVFP4 are written as separate float operations so that
 * each is one IEEE round-to-nearest-even operation. */

/* Nearest-even code of |v| among the 8 E2M1 magnitudes, saturating at 6. */
static unsigned e2m1_round(double a)
{
    unsigned best = 0;
    double bd = INFINITY;
    for (unsigned c = 0; c < 8; ++c) {
        const double d = fabs(or_e2m1(c) - a);
#ifdef OR_PLANT_Q_TIES_UP
        if (d < bd || d == bd) {
#else
        if (d < bd || (d == bd && (c & 1u) == 0)) {
#endif
            bd = d;
            best = c;
        }
    }
    return best;
}

/* Nearest-even code of |v| among the 127 finite E4M3 magnitudes, saturating
 * at 448. */
static unsigned e4m3_round(double a)
{
    unsigned best = 0;
    double bd = INFINITY;
    for (unsigned c = 0; c < 0x7F; ++c) {
        const double d = fabs(or_e4m3(c) - a);
        if (d < bd || (d == bd && (c & 1u) == 0)) {
            bd = d;
            best = c;
        }
    }
    return best;
}

/* Signed code: the magnitude's code with the sign bit set for negative v,
 * except that a zero magnitude is +0. */
static unsigned signed_code(int fmt, double v)
{
    const unsigned mag = fmt == OR_FMT_MXFP8 ? e4m3_round(fabs(v)) : e2m1_round(fabs(v));
    if (mag == 0 || !(v < 0)) return mag;
    return mag | (fmt == OR_FMT_MXFP8 ? 0x80u : 0x8u);
}

static void put_code(int fmt, uint8_t *codes, int64_t m, int64_t k, int64_t K, unsigned c)
{
    if (fmt == OR_FMT_MXFP8) {
        codes[m * K + k] = (uint8_t)c;
    } else {
        uint8_t *b = &codes[m * (K / 2) + k / 2];
#ifdef OR_PLANT_Q_NIBBLE_SWAP
        if (k % 2 == 1) *b = (uint8_t)((*b & 0xF0u) | c);
#else
        if (k % 2 == 0) *b = (uint8_t)((*b & 0xF0u) | c);
#endif
        else *b = (uint8_t)((*b & 0x0Fu) | (c << 4));
    }
}

int or_quantize(int fmt, const uint16_t *x, uint8_t *codes, uint8_t *scales, int64_t M, int64_t K)
{
    const int B = block_of(fmt);
    if (M <= 0 || K <= 0 || K % B) return -1;
    memset(codes, 0, (size_t)(fmt == OR_FMT_MXFP8 ? M * K : M * K / 2));
    float g = 1.0f;
    if (fmt == OR_FMT_NVFP4) {
        double G = 0.0;
        for (int64_t i = 0; i < M * K; ++i) {
            const double a = fabs(or_bf16(x[i]));
            if (isfinite(a) && a > G) G = a;
        }
        if (G > 0) g = (float)G / 2688.0f;  /* G is a bf16 value: exact in float */
        memcpy(scales + M * (K / 16), &g, 4);
    }
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t b0 = 0; b0 < K; b0 += B) {
            double amax = 0.0;
            int finite = 1;
            for (int64_t k = b0; k < b0 + B; ++k) {
                const double v = or_bf16(x[m * K + k]);
                if (!isfinite(v)) finite = 0;
                else if (fabs(v) > amax) amax = fabs(v);
            }
            uint8_t *sb = &scales[m * (K / B) + b0 / B];
            if (!finite) {
                *sb = fmt == OR_FMT_NVFP4 ? 0x7F : 0xFF;
                continue;  /* codes stay zero */
            }
            if (fmt == OR_FMT_NVFP4) {
                const float d = 6.0f * g;
                const float t = (float)amax / d;
                const unsigned s = e4m3_round(t);
                *sb = (uint8_t)s;
                const float den = (float)or_e4m3(s) * g;
                if (den == 0.0f) continue;
                for (int64_t k = b0; k < b0 + B; ++k) {
                    const float v = (float)or_bf16(x[m * K + k]) / den;
                    put_code(fmt, codes, m, k, K, signed_code(fmt, v));
                }
            } else {
                const int emax = fmt == OR_FMT_MXFP8 ? 8 : 2;
                int e = -127;
                if (amax > 0) {
                    int ex;
                    frexp(amax, &ex);   /* amax = f * 2^ex, f in [0.5, 1): floor(log2(amax)) = ex - 1 */
#ifdef OR_PLANT_Q_EMAX
                    e = ex - emax;
#else
                    e = ex - 1 - emax;
#endif
                    if (e < -127) e = -127;
                    if (e > 127) e = 127;
                }
                *sb = (uint8_t)(e + 127);
                for (int64_t k = b0; k < b0 + B; ++k) {
                    const double v = ldexp(or_bf16(x[m * K + k]), -e);  /* exact */
                    put_code(fmt, codes, m, k, K, signed_code(fmt, v));
                }
            }
        }
    }
    return 0;
}

/* ------------------------------------------- product over quantised activations */

/* y[m][n] = sum_k X^[m][k] * W^[n][k], fp64, increasing k, where both X^ and
 * W^ are decoded block-float tensors of the same format (X^ from x codes
 * [M][K(/2)] and scales [M][K/block] (+ tensor scale), W^ as in or_qmv): the
 * reference for a matmul whose activations were quantised first (the
 * on-device quantiser above feeding a block-scaled tensor-core product).
 * Parity of such a kernel is checked against this, on the same quantised
 * operands. */
int or_qmm_qx(int fmt, const uint8_t *codes, const uint8_t *scales, const uint8_t *xcodes,
              const uint8_t *xscales, double *y, int64_t M, int64_t N, int64_t K)
{
    if (M <= 0 || N <= 0 || K <= 0 || K % block_of(fmt)) return -1;
    float *X = (float *)malloc((size_t)(M * K) * sizeof(float));
    float *W = (float *)malloc((size_t)K * sizeof(float));
    if (!X || !W) {
        free(X);
        free(W);
        return -2;
    }
    const float gx = fmt == OR_FMT_NVFP4 ? tensor_scale(xscales, M, K) : 1.0f;
    const float gw = fmt == OR_FMT_NVFP4 ? tensor_scale(scales, N, K) : 1.0f;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k) X[m * K + k] = weight(fmt, xcodes, xscales, gx, m, k, M, K);
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t k = 0; k < K; ++k) W[k] = weight(fmt, codes, scales, gw, n, k, N, K);
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) acc += (double)X[m * K + k] * (double)W[k];
            y[m * N + n] = acc;
        }
    }
    free(X);
    free(W);
    return 0;
}
