/*
 * nvfp4_oracle.c -- plain CPU reference for the NVFP4 grouped GEMM.
 *
 * TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only the test suite, the
 * smoke check and the benchmark's CPU-baseline leg may load or call this
 * library.  It shares no code, header, table or constant with the CUDA path.
 *
 * What it computes (kernelbot nvfp4-group-gemm, submission 474067: the
 * header comment of the CUDA source names FP4 E2M1 inputs, FP8 E4M3FN scale
 * factors and an FP16 output; tcgen05_mma_nvfp4 issues
 * kind::mxf4nvf4.block_scale.block16, i.e. one scale per 16 K-elements; the
 * first MMA of every tile runs with enable_input_d = 0, so there is no C
 * input):
 *
 *   C[m][n] = fp16_rne( sum_{k<K} e2m1(A[m][k]) * e4m3fn(SFA[m][k/16])
 *                                * e2m1(B[n][k]) * e4m3fn(SFB[n][k/16]) )
 *
 * A is [M][K/2] bytes, B is [N][K/2] bytes (K-major, two E2M1 codes per byte,
 * element 2i in the low nibble of byte i).  SFA is [M][K/16] bytes and SFB is
 * [N][K/16] bytes, both plain row-major.  The sum is taken in float64.  For
 * the value ranges of the benchmark configurations this sum is exact (every
 * product is a multiple of 2^-20 and the partial sums stay far below 2^33),
 * so the result is the correctly rounded FP16 value of the exact real sum.
 *
 * The scale-factor relayout (the tiled layout the GPU kernel consumes) is
 * defined here as a pure byte permutation; see nvfp4_oracle_sf_relayout.
 *
 * Every function is a direct transcription of the definitions above; nothing
 * is blocked, fused or reordered beyond an optional split of output rows
 * across threads.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------------ */
/* Element decoders, from the bit definitions of the two formats.            */
/* ------------------------------------------------------------------------ */

/* FP4 E2M1 (OCP Microscaling Formats v1.0, FP4 E2M1): bit 3 = sign,
 * bits 2..1 = exponent (bias 1), bit 0 = mantissa.  Exponent 0 is
 * subnormal: value = m * 2^-1.  No inf, no NaN. */
double nvfp4_oracle_e2m1(unsigned code)
{
    unsigned s = (code >> 3) & 1u;
    unsigned e = (code >> 1) & 3u;
    unsigned m = code & 1u;
    double mag;
    if (e == 0)
        mag = 0.5 * (double)m;
    else
        mag = ldexp(1.0 + 0.5 * (double)m, (int)e - 1);
    return s ? -mag : mag;
}

/* FP8 E4M3FN (OCP 8-bit floating point, E4M3 with the "FN" encoding):
 * bit 7 = sign, bits 6..3 = exponent (bias 7), bits 2..0 = mantissa.
 * Exponent 0 is subnormal: value = m/8 * 2^-6.  S.1111.111 is NaN; there is
 * no infinity, so S.1111.000 .. S.1111.110 are ordinary finite values. */
double nvfp4_oracle_e4m3fn(unsigned byte)
{
    unsigned s = (byte >> 7) & 1u;
    unsigned e = (byte >> 3) & 15u;
    unsigned m = byte & 7u;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return s ? -mag : mag;
}

/* Round a double to IEEE binary16 with round-to-nearest-even, returning the
 * bit pattern.  Handles subnormals, overflow to +-inf (|x| >= 65520 rounds
 * up past the largest finite 65504) and NaN (returned as 0x7E00). */
uint16_t nvfp4_oracle_fp16_rne(double x)
{
    if (isnan(x))
        return 0x7E00u;
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (isinf(a))
        return (uint16_t)(sign | 0x7C00u);
    if (a == 0.0)
        return sign;

    /* quantum of the binade a lies in: 11 significant bits for normals,
     * fixed 2^-24 below the smallest normal 2^-14 */
    int ex;
    (void)frexp(a, &ex);            /* a = f * 2^ex, f in [0.5, 1) */
    int qexp = ex - 11;
    if (qexp < -24)
        qexp = -24;
    double r = ldexp(a, -qexp);     /* exact: power-of-two scaling */
    double fl = floor(r);
    double diff = r - fl;           /* exact */
    double n = fl;
    if (diff > 0.5 || (diff == 0.5 && fmod(fl, 2.0) != 0.0))
        n = fl + 1.0;
    double v = ldexp(n, qexp);      /* the rounded magnitude, exact */

    if (v >= 65536.0)
        return (uint16_t)(sign | 0x7C00u);
    if (v < ldexp(1.0, -14)) {
        /* subnormal (or zero): integer multiple of 2^-24 */
        unsigned mant = (unsigned)ldexp(v, 24);
        return (uint16_t)(sign | mant);
    }
    int e2;
    double f = frexp(v, &e2);       /* v = f * 2^e2, f in [0.5, 1) */
    unsigned efield = (unsigned)(e2 + 14);
    unsigned mant = (unsigned)((f * 2.0 - 1.0) * 1024.0);
    return (uint16_t)(sign | (efield << 10) | mant);
}

/* ------------------------------------------------------------------------ */
/* Operand access.                                                            */
/* ------------------------------------------------------------------------ */

/* E2M1 code of element k of a K-major row of packed bytes: element 2i is the
 * low nibble of byte i, element 2i+1 the high nibble. */
static unsigned fp4_code(const uint8_t *row, int k)
{
    uint8_t byte = row[k >> 1];
    return (k & 1) ? (unsigned)(byte >> 4) : (unsigned)(byte & 0x0Fu);
}

/* Dequantised row: out[k] = e2m1(row[k]) * e4m3fn(sf_row[k/16]).  Each
 * product has at most 6 significant bits, so it is exact in float64. */
static void dequant_row(const uint8_t *row, const uint8_t *sf_row, int K,
                        double *out)
{
    for (int k = 0; k < K; ++k)
        out[k] = nvfp4_oracle_e2m1(fp4_code(row, k)) *
                 nvfp4_oracle_e4m3fn(sf_row[k / 16]);
}

/* ------------------------------------------------------------------------ */
/* One group, float64 accumulation.                                           */
/* ------------------------------------------------------------------------ */

typedef struct {
    const uint8_t *A, *SFA;
    const double *Bdq;      /* [N][K] dequantised B, shared read-only        */
    uint16_t *C;            /* [M][N] FP16 bits, may be NULL                 */
    double *acc;            /* [M][N] float64 sums before rounding, may be NULL */
    int M, N, K;
    const int32_t *rows;    /* output rows of this worker                    */
    int nrows;
} gemm_job;

static void *gemm_worker(void *arg)
{
    gemm_job *j = (gemm_job *)arg;
    const int K = j->K;
    double *arow = (double *)malloc(sizeof(double) * (size_t)K);
    if (!arow)
        return (void *)1;
    for (int i = 0; i < j->nrows; ++i) {
        const int m = j->rows[i];
        dequant_row(j->A + (size_t)m * (K / 2), j->SFA + (size_t)m * (K / 16), K, arow);
        for (int n = 0; n < j->N; ++n) {
            const double *brow = j->Bdq + (size_t)n * K;
            double sum = 0.0;
            for (int k = 0; k < K; ++k)
                sum += arow[k] * brow[k];
            size_t idx = (size_t)m * j->N + n;
            if (j->acc)
                j->acc[idx] = sum;
            if (j->C)
                j->C[idx] = nvfp4_oracle_fp16_rne(sum);
        }
    }
    free(arow);
    return NULL;
}

static int resolve_threads(int n_threads, int rows)
{
    if (n_threads <= 0) {
        long c = sysconf(_SC_NPROCESSORS_ONLN);
        n_threads = c > 0 ? (int)c : 1;
    }
    if (n_threads > rows)
        n_threads = rows;
    if (n_threads < 1)
        n_threads = 1;
    if (n_threads > 256)
        n_threads = 256;
    return n_threads;
}

typedef struct {
    const uint8_t *X, *SFX;
    double *out;
    int K, r0, r1;
} dequant_job;

static void *dequant_worker(void *arg)
{
    dequant_job *j = (dequant_job *)arg;
    for (int r = j->r0; r < j->r1; ++r)
        dequant_row(j->X + (size_t)r * (j->K / 2), j->SFX + (size_t)r * (j->K / 16), j->K,
                    j->out + (size_t)r * j->K);
    return NULL;
}

/* out[r][k] = dequantised element k of row r, rows split across T threads */
static void dequant_rows_parallel(const uint8_t *X, const uint8_t *SFX, int rows, int K,
                                  double *out, int T)
{
    dequant_job jobs[256];
    pthread_t tids[256];
    int started[256];
    for (int t = 0; t < T; ++t) {
        jobs[t] = (dequant_job){X, SFX, out, K, (int)((long)rows * t / T),
                                (int)((long)rows * (t + 1) / T)};
        started[t] = (t > 0) && pthread_create(&tids[t], NULL, dequant_worker, &jobs[t]) == 0;
        if (t > 0 && !started[t])
            dequant_worker(&jobs[t]);
    }
    dequant_worker(&jobs[0]);
    for (int t = 1; t < T; ++t)
        if (started[t])
            pthread_join(tids[t], NULL);
}

/* The listed rows of C for one group.  C and acc are full [M][N] buffers;
 * only the listed rows are written.  B is dequantised once (N*K doubles,
 * rows split across threads), then each row of A is dequantised and dotted
 * with every row of B, k in ascending order.  n_threads <= 0 uses every online core.  Returns 0 on
 * success, -1 on bad arguments or allocation failure. */
int nvfp4_oracle_gemm_rows(const uint8_t *A, const uint8_t *SFA,
                           const uint8_t *B, const uint8_t *SFB,
                           uint16_t *C, double *acc,
                           int M, int N, int K, const int32_t *rows, int nrows,
                           int n_threads)
{
    if (M < 0 || N < 0 || K < 0 || (K % 16) != 0 || nrows < 0)
        return -1;
    for (int i = 0; i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= M)
            return -1;
    if (nrows == 0 || N == 0)
        return 0;
    double *Bdq = (double *)malloc(sizeof(double) * (size_t)N * (size_t)K);
    if (!Bdq)
        return -1;
    dequant_rows_parallel(B, SFB, N, K, Bdq, resolve_threads(n_threads, N));
    int T = resolve_threads(n_threads, nrows);
    gemm_job jobs[256];
    pthread_t tids[256];
    int started[256];
    int rc = 0;
    for (int t = 0; t < T; ++t) {
        int i0 = (int)((long)nrows * t / T), i1 = (int)((long)nrows * (t + 1) / T);
        jobs[t] = (gemm_job){A, SFA, Bdq, C, acc, M, N, K, rows + i0, i1 - i0};
        started[t] = (t > 0) && pthread_create(&tids[t], NULL, gemm_worker, &jobs[t]) == 0;
        if (t > 0 && !started[t] && gemm_worker(&jobs[t]) != NULL)
            rc = -1;
    }
    if (gemm_worker(&jobs[0]) != NULL)
        rc = -1;
    for (int t = 1; t < T; ++t) {
        if (started[t]) {
            void *ret = NULL;
            pthread_join(tids[t], &ret);
            if (ret != NULL)
                rc = -1;
        }
    }
    free(Bdq);
    return rc;
}

/* C rows [m_begin, m_end) of one group (see nvfp4_oracle_gemm_rows). */
int nvfp4_oracle_gemm(const uint8_t *A, const uint8_t *SFA,
                      const uint8_t *B, const uint8_t *SFB,
                      uint16_t *C, double *acc,
                      int M, int N, int K, int m_begin, int m_end,
                      int n_threads)
{
    if (m_begin < 0 || m_end > M || m_begin > m_end)
        return -1;
    int nrows = m_end - m_begin;
    if (nrows == 0)
        return 0;
    int32_t *rows = (int32_t *)malloc(sizeof(int32_t) * (size_t)nrows);
    if (!rows)
        return -1;
    for (int i = 0; i < nrows; ++i)
        rows[i] = m_begin + i;
    int rc = nvfp4_oracle_gemm_rows(A, SFA, B, SFB, C, acc, M, N, K, rows, nrows, n_threads);
    free(rows);
    return rc;
}

/* Sampled outputs: out[i] = C[ms[i]][ns[i]] for one group (FP16 bits). */
int nvfp4_oracle_gemm_elements(const uint8_t *A, const uint8_t *SFA,
                               const uint8_t *B, const uint8_t *SFB,
                               int M, int N, int K,
                               const int32_t *ms, const int32_t *ns, int count,
                               uint16_t *out)
{
    if (K % 16 != 0)
        return -1;
    for (int i = 0; i < count; ++i) {
        int m = ms[i], n = ns[i];
        if (m < 0 || m >= M || n < 0 || n >= N)
            return -1;
        const uint8_t *arow = A + (size_t)m * (K / 2);
        const uint8_t *brow = B + (size_t)n * (K / 2);
        const uint8_t *sa = SFA + (size_t)m * (K / 16);
        const uint8_t *sb = SFB + (size_t)n * (K / 16);
        double sum = 0.0;
        for (int k = 0; k < K; ++k)
            sum += nvfp4_oracle_e2m1(fp4_code(arow, k)) * nvfp4_oracle_e4m3fn(sa[k / 16]) *
                   nvfp4_oracle_e2m1(fp4_code(brow, k)) * nvfp4_oracle_e4m3fn(sb[k / 16]);
        out[i] = nvfp4_oracle_fp16_rne(sum);
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Exact fixed-point accumulation (an independent pin on the float64 sum).   */
/* ------------------------------------------------------------------------ */

/* E2M1 magnitude in units of 2^-1: 0, 1, 2, 3, 4, 6, 8, 12. */
static int64_t e2m1_halves(unsigned code, int *neg)
{
    unsigned e = (code >> 1) & 3u, m = code & 1u;
    *neg = (int)((code >> 3) & 1u);
    if (e == 0)
        return (int64_t)m;                          /* m * 0.5 = m halves  */
    return (int64_t)(2 + m) << (e - 1);             /* (1 + m/2) 2^(e-1)   */
}

/* E4M3FN as an integer significand times 2^exp (exp in [-9, 5]).
 * Returns -1 for NaN. */
static int e4m3_int(unsigned byte, int64_t *sig, int *exp2, int *neg)
{
    unsigned e = (byte >> 3) & 15u, m = byte & 7u;
    *neg = (int)((byte >> 7) & 1u);
    if (e == 15 && m == 7)
        return -1;
    if (e == 0) {
        *sig = (int64_t)m;                          /* m/8 * 2^-6          */
        *exp2 = -9;
    } else {
        *sig = (int64_t)(8 + m);                    /* (1+m/8) 2^(e-7)     */
        *exp2 = (int)e - 10;
    }
    return 0;
}

/* acc_units[m][n] = sum of the products in units of 2^-20, as an exact
 * int64.  Every finite product a*sa*b*sb is an integer multiple of 2^-20
 * (halves * halves * 2^-9 * 2^-9), and |product| < 2^43, so sums of up to
 * 2^19 terms cannot overflow.  Returns -1 on a NaN scale or bad sizes. */
int nvfp4_oracle_gemm_fixed(const uint8_t *A, const uint8_t *SFA,
                            const uint8_t *B, const uint8_t *SFB,
                            int64_t *acc_units, int M, int N, int K)
{
    if (M < 0 || N < 0 || K < 0 || K % 16 != 0 || K > (1 << 19))
        return -1;
    for (int m = 0; m < M; ++m) {
        for (int n = 0; n < N; ++n) {
            int64_t sum = 0;
            for (int k = 0; k < K; ++k) {
                int na, nb, nsa, nsb, ea, eb;
                int64_t sa, sb;
                int64_t a = e2m1_halves(fp4_code(A + (size_t)m * (K / 2), k), &na);
                int64_t b = e2m1_halves(fp4_code(B + (size_t)n * (K / 2), k), &nb);
                if (e4m3_int(SFA[(size_t)m * (K / 16) + k / 16], &sa, &ea, &nsa) ||
                    e4m3_int(SFB[(size_t)n * (K / 16) + k / 16], &sb, &eb, &nsb))
                    return -1;
                /* value = a/2 * sa*2^ea * b/2 * sb*2^eb
                 *       = a*b*sa*sb * 2^(ea+eb-2);  in units of 2^-20: */
                int shift = ea + eb - 2 + 20;       /* >= 0 */
                int64_t p = (a * b * sa * sb) << shift;
                if (na ^ nb ^ nsa ^ nsb)
                    p = -p;
                sum += p;
            }
            acc_units[(size_t)m * N + n] = sum;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Scale-factor relayout: plain row-major [rows][K/16] -> tiled atoms.       */
/* ------------------------------------------------------------------------ */

/* The tiled layout groups scales into 512-byte atoms, one per
 * (128-row block rb, 64-element K block kb), stored in the order
 * [rb][kb] (kernelbot nvfp4-group-gemm submission 474067, TMA producer warp
 * of group_gemm_persistent_kernel: the scale source address is
 * base + ((row_block * K/64) + k_block) * 512).  Inside an atom, the scale of
 * row r (0..127 within the block) and 16-element K sub-block j (0..3 within
 * the 64-element block) sits at byte (r % 32) * 16 + (r / 32) * 4 + j: 32
 * rows of 16 bytes, each holding the four row-quarters' four scales, which is
 * the shape a 32x128b tensor-memory copy replicated to four warps moves.
 * Rows at or beyond `rows` in the last block are zero. */
size_t nvfp4_oracle_sf_tiled_bytes(int rows, int K)
{
    if (rows <= 0 || K <= 0)
        return 0;
    size_t rb = (size_t)(rows + 127) / 128;
    return rb * (size_t)(K / 64) * 512u;
}

int nvfp4_oracle_sf_relayout(const uint8_t *src, uint8_t *dst, int rows, int K)
{
    if (rows < 0 || K < 0 || K % 64 != 0)
        return -1;
    int kblocks = K / 64;
    int rblocks = (rows + 127) / 128;
    for (int rb = 0; rb < rblocks; ++rb)
        for (int kb = 0; kb < kblocks; ++kb) {
            uint8_t *atom = dst + ((size_t)rb * kblocks + kb) * 512;
            for (int r = 0; r < 128; ++r)
                for (int j = 0; j < 4; ++j) {
                    int row = rb * 128 + r;
                    int col = kb * 4 + j;           /* scale index = k/16  */
                    uint8_t v = row < rows ? src[(size_t)row * (K / 16) + col] : 0;
                    atom[(r % 32) * 16 + (r / 32) * 4 + j] = v;
                }
        }
    return 0;
}

/* Inverse of the relayout for rows < `rows` (padding is dropped). */
int nvfp4_oracle_sf_unrelayout(const uint8_t *tiled, uint8_t *dst, int rows, int K)
{
    if (rows < 0 || K < 0 || K % 64 != 0)
        return -1;
    int kblocks = K / 64;
    for (int row = 0; row < rows; ++row)
        for (int col = 0; col < K / 16; ++col) {
            int rb = row / 128, r = row % 128, kb = col / 4, j = col % 4;
            const uint8_t *atom = tiled + ((size_t)rb * kblocks + kb) * 512;
            dst[(size_t)row * (K / 16) + col] = atom[(r % 32) * 16 + (r / 32) * 4 + j];
        }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* NVFP4 quantisation, the step that produces the GEMM's operands: every    */
/* 16-element block of a row gets the scale E4M3FN(absmax / 6) and every    */
/* element the E2M1 code of x / scale (the generator of the "quantized"     */
/* configuration of the grouped GEMM: values quantised per 16-block to E2M1 */
/* with an absmax/6 scale rounded to E4M3FN).  Both rounding decisions are  */
/* taken on IEEE single-precision values (absmax / 6 and x / scale rounded  */
/* to nearest), the precision the GPU kernel computes in.                   */
/* ------------------------------------------------------------------------ */

/* IEEE binary16 bits -> float (exact: every half is a float) */
static float half_bits_to_float(uint16_t h)
{
    const unsigned s = (h >> 15) & 1u, e = (h >> 10) & 31u, m = h & 1023u;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                       /* subnormal */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp(1.0 + (double)m / 1024.0, (int)e - 15);
    return (float)(s ? -v : v);
}

/* bfloat16 bits -> float (exact: the upper half of a float's bits) */
static float bf16_bits_to_float(uint16_t h)
{
    const uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof(f));
    return f;
}

/* E4M3FN code of a finite float >= 0: the nearest finite E4M3FN value, ties
 * to the even code (mantissa bit 0 clear); everything above 448 becomes 448
 * (0x7E), the largest finite value; 0 and negative inputs give 0. */
unsigned nvfp4_oracle_e4m3_rne(float v)
{
    if (!(v > 0.0f))
        return 0;
    if (v >= 448.0f)          /* saturation (also keeps the distances below exact) */
        return 0x7E;
    const double x = (double)v;
    unsigned best = 0;
    double best_d = x;                                    /* distance to 0 */
    for (unsigned c = 1; c < 0x7F; ++c) {                 /* 0x7F is NaN */
        const double d = fabs(x - nvfp4_oracle_e4m3fn(c));
        if (d < best_d || (d == best_d && (c & 1u) == 0 && (best & 1u) == 1)) {
            best = c;
            best_d = d;
        }
    }
    return best;
}

/* E2M1 code of a finite float: the magnitude is the nearest of
 * {0, .5, 1, 1.5, 2, 3, 4, 6} (ties to the even code, 6 for anything larger),
 * the sign goes to bit 3 unless the magnitude is 0 (zero is always 0x0). */
unsigned nvfp4_oracle_e2m1_rne(float q)
{
    const double a = fabs((double)q);
    if (a >= 6.0)             /* saturation (also keeps the distances below exact) */
        return q < 0.0f ? 0xFu : 0x7u;
    unsigned best = 0;
    double best_d = a;
    for (unsigned c = 1; c < 8; ++c) {
        const double d = fabs(a - nvfp4_oracle_e2m1(c));
        if (d < best_d || (d == best_d && (c & 1u) == 0 && (best & 1u) == 1)) {
            best = c;
            best_d = d;
        }
    }
    return (best != 0 && q < 0.0f) ? (best | 8u) : best;
}

/* x: [rows][K] FP16 (is_bf16 = 0) or BF16 (is_bf16 = 1) bits, finite;
 * codes: [rows][K/2] bytes, element 2i in the low nibble; sf: [rows][K/16]
 * E4M3FN bytes (row-major).  A block whose scale rounds to 0 (absmax < 6 *
 * 2^-10, all zeros included) gets scale 0 and codes 0.  K % 16 == 0. */
int nvfp4_oracle_quantize(const uint16_t *x, int is_bf16, int rows, int K, uint8_t *codes,
                          uint8_t *sf)
{
    if (rows < 0 || K <= 0 || K % 16 != 0 || !x || !codes || !sf)
        return -1;
    for (int r = 0; r < rows; ++r) {
        for (int b = 0; b < K / 16; ++b) {
            float v[16];
            float amax = 0.0f;
            for (int i = 0; i < 16; ++i) {
                const uint16_t h = x[(size_t)r * K + (size_t)b * 16 + i];
                v[i] = is_bf16 ? bf16_bits_to_float(h) : half_bits_to_float(h);
                const float a = fabsf(v[i]);
                if (a > amax)
                    amax = a;
            }
            const float s32 = amax / 6.0f;
            const unsigned sc = nvfp4_oracle_e4m3_rne(s32);
            const float sdec = (float)nvfp4_oracle_e4m3fn(sc);
            sf[(size_t)r * (K / 16) + b] = (uint8_t)sc;
            for (int i = 0; i < 16; i += 2) {
                const unsigned lo = sdec > 0.0f ? nvfp4_oracle_e2m1_rne(v[i] / sdec) : 0u;
                const unsigned hi = sdec > 0.0f ? nvfp4_oracle_e2m1_rne(v[i + 1] / sdec) : 0u;
                codes[(size_t)r * (K / 2) + (size_t)b * 8 + i / 2] = (uint8_t)(lo | (hi << 4));
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Fused epilogue options of the grouped GEMM (an MoE layer's per-tensor    */
/* scale, BF16 output and the SwiGLU of a gate/up projection), applied to   */
/* the exact float64 sums.                                                   */
/* ------------------------------------------------------------------------ */

/* Round a double to bfloat16 (8 exponent bits, 8 significant bits) with
 * round-to-nearest-even, returning the bit pattern: subnormals (multiples of
 * 2^-133), overflow to +-inf, NaN as 0x7FC0. */
uint16_t nvfp4_oracle_bf16_rne(double x)
{
    if (isnan(x))
        return 0x7FC0u;
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (isinf(a))
        return (uint16_t)(sign | 0x7F80u);
    if (a == 0.0)
        return sign;
    int ex;
    (void)frexp(a, &ex);            /* a = f * 2^ex, f in [0.5, 1) */
    int qexp = ex - 8;
    if (qexp < -133)
        qexp = -133;
    double r = ldexp(a, -qexp);
    double fl = floor(r);
    double diff = r - fl;
    double n = fl;
    if (diff > 0.5 || (diff == 0.5 && fmod(fl, 2.0) != 0.0))
        n = fl + 1.0;
    double v = ldexp(n, qexp);
    if (v >= ldexp(1.0, 128))
        return (uint16_t)(sign | 0x7F80u);
    if (v < ldexp(1.0, -126)) {
        unsigned mant = (unsigned)ldexp(v, 133);
        return (uint16_t)(sign | mant);
    }
    int e2;
    double f = frexp(v, &e2);       /* v = f * 2^e2 */
    unsigned efield = (unsigned)(e2 + 126);
    unsigned mant = (unsigned)((f * 2.0 - 1.0) * 128.0);
    return (uint16_t)(sign | (efield << 7) | mant);
}

/* SiLU in float64: x * sigmoid(x) = x / (1 + e^-x) */
double nvfp4_oracle_silu(double x)
{
    return x / (1.0 + exp(-x));
}

/* acc: the exact sums [M][N] of one group (float64).  Plain: out[m][n] =
 * alpha * acc[m][n], [M][N].  SwiGLU (N % 256 == 0): the B rows come in
 * 256-row blocks, 128 gate rows then the 128 up rows of the same outputs,
 * and out[m][128 j + c] = silu(alpha * acc[m][256 j + c]) *
 * (alpha * acc[m][256 j + 128 + c]), [M][N/2].  Rounded once, to BF16 if
 * bf16 else FP16. */
int nvfp4_oracle_epilogue(const double *acc, int M, int N, double alpha, int swiglu, int bf16,
                          uint16_t *out)
{
    if (M < 0 || N <= 0 || !acc || !out || (swiglu && N % 256 != 0))
        return -1;
    const int nout = swiglu ? N / 2 : N;
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < nout; ++n) {
            double v;
            if (swiglu) {
                const int j = n / 128, c = n % 128;
                const double g = alpha * acc[(size_t)m * N + 256 * j + c];
                const double u = alpha * acc[(size_t)m * N + 256 * j + 128 + c];
                v = nvfp4_oracle_silu(g) * u;
            } else {
                v = alpha * acc[(size_t)m * N + n];
            }
            out[(size_t)m * nout + n] = bf16 ? nvfp4_oracle_bf16_rne(v) : nvfp4_oracle_fp16_rne(v);
        }
    return 0;
}
