/*
 * Plain CPU oracle for the block-scaled (MX) dense matrix multiply
 *
 *     D = alpha * (A scaled by SA) * (B scaled by SB) + beta * C
 *
 * TEST INFRASTRUCTURE ONLY, like oracle.c: only the test suite, the package
 * smoke check and the benchmark's CPU-baseline leg load liboracle.so, and this
 * file shares no source with the CUDA library.
 *
 * Where it comes from. "TorchInductor ganha suporte a GEMMs de alta
 * performance com CuteDSL" names scaled_mm among the GEMMs its backend covers
 * (the enablement paragraph) and reports MXFP8 results (the results
 * paragraph), but it defines no element or scale format. The formats are
 * those of the OCP Microscaling (MX) Formats Specification v1.0, read here as:
 *  - an MX block is 32 consecutive elements along K that share one scale;
 *  - the scale is E8M0: an unsigned 8-bit exponent e with value 2^(e - 127);
 *    e = 255 is NaN;
 *  - an FP8 element is E4M3 (bias 7, no infinities, S.1111.111 is NaN,
 *    largest finite 448) or E5M2 (bias 15, IEEE-style infinities and NaNs,
 *    largest finite 57344), both with subnormals;
 *  - an element's value is scale * element, and the dot product of two MX
 *    blocks is scale_A * scale_B * (sum of the 32 element products).
 * The GEMM is that dot product taken over the K/32 blocks of a row of A and
 * a column of B:
 *     acc[i,n] = sum over blocks b (ascending) of
 *                (SA[i,b] * SB[n,b]) * (sum over k in b (ascending) of A[i,k] * B[k,n])
 * in fp64, then D = alpha*acc + beta*C (two separate fp64 operations) and one
 * round-to-nearest-even rounding to the output dtype, as in oracle.c.
 * In fp64 every element product is exact (FP8 significands have at most 4
 * bits), and so is every scale product (a power of two between 2^-254 and
 * 2^254); the only roundings are those of the fp64 sums and the final one.
 * (With NVFP4's E4M3 scales, below, a scale product has at most 8 significant
 * bits and an element product at most 4: still exact.)
 *
 * Layouts (the oracle's own, plain ones): A is [M, K] bytes, row-major with
 * row stride lda; B is given transposed, Bt = [N, K] bytes, row-major with
 * row stride ldb (B[k,n] = Bt[n,k]); SA is [M, K/32] and SB is [N, K/32] scale
 * bytes, row-major with row strides ldsa and ldsb. K must be a multiple of 32.
 *
 * FP4. The same page names FP4 GEMMs, NVFP4 and MXF4, and reports NVFP4
 * results on decode shapes. Read here as:
 *  - an FP4 element is E2M1 (OCP MX specification): sign, two exponent bits
 *    with bias 1, one mantissa bit, a subnormal 0.5 at exponent field 0, no
 *    infinities or NaNs; the values are 0, 0.5, 1, 1.5, 2, 3, 4 and 6 and
 *    their negatives;
 *  - two elements share a byte, the even-numbered one (along K) in the low
 *    four bits, so a row of K elements is K/2 bytes;
 *  - MXFP4 (OCP MX): blocks of 32 elements, E8M0 scales, as above;
 *  - NVFP4 (NVIDIA's FP4 format): blocks of 16 elements, each with an E4M3
 *    scale, decoded as E4M3 above; the format's per-tensor scale is a plain
 *    multiplier of the product and is the caller's alpha here.
 * The block dot product and the GEMM are as above, over K/16 or K/32 blocks.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_FP8_E4M3 0
#define ORACLE_FP8_E5M2 1
#define ORACLE_SCALE_E8M0 2
#define ORACLE_FP4_E2M1 3
#define ORACLE_MX_BLOCK 32

/* Defined in oracle.c. */
uint16_t oracle_round_bf16(double x);
float oracle_round_f32(double x);

/* E4M3: s eeee mmm; exponent field 0 holds subnormals m/8 * 2^-6. */
double oracle_decode_e4m3(uint8_t x) {
    const int s = x >> 7;
    const int e = (x >> 3) & 0xF;
    const int m = x & 0x7;
    if (e == 15 && m == 7) return NAN;
    const double v = e == 0 ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
    return s ? -v : v;
}

/* E5M2: s eeeee mm; exponent field 31 holds infinities (m == 0) and NaNs. */
double oracle_decode_e5m2(uint8_t x) {
    const int s = x >> 7;
    const int e = (x >> 2) & 0x1F;
    const int m = x & 0x3;
    if (e == 31) return m == 0 ? (s ? -INFINITY : INFINITY) : NAN;
    const double v = e == 0 ? ldexp((double)m, -16) : ldexp((double)(4 + m), e - 17);
    return s ? -v : v;
}

/* E8M0: 2^(e - 127), e = 255 is NaN. */
double oracle_decode_e8m0(uint8_t x) { return x == 255 ? NAN : ldexp(1.0, (int)x - 127); }

/* E2M1: s ee m (low four bits of x); exponent field 0 holds the subnormal m/2. */
double oracle_decode_e2m1(uint8_t x) {
    const int s = (x >> 3) & 1;
    const int e = (x >> 1) & 0x3;
    const int m = x & 0x1;
    const double v = e == 0 ? 0.5 * m : ldexp((double)(2 + m), e - 2);
    return s ? -v : v;
}

static double oracle_decode_fp8(int fmt, uint8_t x) {
    return fmt == ORACLE_FP8_E5M2 ? oracle_decode_e5m2(x) : oracle_decode_e4m3(x);
}

/* Element k of a row of codes in format fmt (FP4 packs two per byte, element
 * 2i in the low four bits of byte i). */
static double oracle_element(int fmt, const uint8_t *row, int64_t k) {
    if (fmt == ORACLE_FP4_E2M1) return oracle_decode_e2m1((uint8_t)((row[k / 2] >> (4 * (k % 2))) & 0xF));
    return oracle_decode_fp8(fmt, row[k]);
}

static double oracle_scale(int sfmt, uint8_t x) {
    return sfmt == ORACLE_SCALE_E8M0 ? oracle_decode_e8m0(x) : oracle_decode_e4m3(x);
}

/* Batch decoders, for the pins. fmt: 0 E4M3, 1 E5M2, 2 E8M0, 3 E2M1 (the low
 * four bits of each byte). */
void oracle_decode_mx_array(int fmt, const uint8_t *in, double *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i)
        out[i] = fmt == ORACLE_SCALE_E8M0 ? oracle_decode_e8m0(in[i])
                 : fmt == ORACLE_FP4_E2M1 ? oracle_decode_e2m1((uint8_t)(in[i] & 0xF))
                                           : oracle_decode_fp8(fmt, in[i]);
}

typedef struct {
    int64_t N, K, nb, block;
    const uint8_t *A;
    int64_t lda;
    int fmt_a;
    int sfmt;
    const uint8_t *SA;
    int64_t ldsa;
    const double *Bd;  /* decoded B, [K, N] */
    const double *SBd; /* decoded SB, [nb, N] */
    const void *C;
    int64_t ldc;
    double alpha, beta;
    int out_dtype;
    const int64_t *rows;
    int64_t row_begin, row_end;
    void *D;
    int64_t ldd;
    double *pre;
    int64_t ldpre;
    int status;
} oracle_mx_job;

static void *oracle_mx_worker(void *arg) {
    oracle_mx_job *j = (oracle_mx_job *)arg;
    const size_t n1 = (size_t)(j->N > 0 ? j->N : 1);
    double *acc = (double *)malloc(n1 * sizeof(double));
    double *part = (double *)malloc(n1 * sizeof(double));
    if (!acc || !part) {
        free(acc);
        free(part);
        j->status = -1;
        return NULL;
    }
    for (int64_t r = j->row_begin; r < j->row_end; ++r) {
        const int64_t i = j->rows[r];
        for (int64_t n = 0; n < j->N; ++n) acc[n] = 0.0;
        for (int64_t b = 0; b < j->nb; ++b) {
            /* part[n] = sum over the block's k, ascending, of A[i,k] * B[k,n] */
            for (int64_t n = 0; n < j->N; ++n) part[n] = 0.0;
            for (int64_t k = b * j->block; k < (b + 1) * j->block; ++k) {
                const double a = oracle_element(j->fmt_a, j->A + i * j->lda, k);
                const double *brow = j->Bd + k * j->N;
                for (int64_t n = 0; n < j->N; ++n) part[n] += a * brow[n];
            }
            /* acc[n] += (SA[i,b] * SB[n,b]) * part[n] */
            const double sa = oracle_scale(j->sfmt, j->SA[i * j->ldsa + b]);
            const double *sb = j->SBd + b * j->N;
            for (int64_t n = 0; n < j->N; ++n) acc[n] += (sa * sb[n]) * part[n];
        }
        for (int64_t n = 0; n < j->N; ++n) {
            double v = j->alpha * acc[n];
            if (j->beta != 0.0) {
                double c;
                if (j->out_dtype == 0) {
                    const uint32_t u = (uint32_t)((const uint16_t *)j->C)[i * j->ldc + n] << 16;
                    float f;
                    memcpy(&f, &u, sizeof f);
                    c = (double)f;
                } else {
                    c = (double)((const float *)j->C)[i * j->ldc + n];
                }
                v = v + j->beta * c;
            }
            if (j->pre) j->pre[r * j->ldpre + n] = v;
            if (j->out_dtype == 0)
                ((uint16_t *)j->D)[r * j->ldd + n] = oracle_round_bf16(v);
            else
                ((float *)j->D)[r * j->ldd + n] = oracle_round_f32(v);
        }
    }
    free(acc);
    free(part);
    j->status = 0;
    return NULL;
}

/*
 * Output rows rows[0..nrows) of the block-scaled GEMM described at the top of
 * this file. fmt_a, fmt_b: 0 E4M3, 1 E5M2, 3 E2M1 (FP4, two per byte); sfmt:
 * 2 E8M0 or 0 E4M3; block: 32 or 16 elements per scale. Row strides are in
 * bytes; a row of K FP4 elements is K/2 bytes. C is of the output dtype (0
 * bf16, 1 fp32), [M, N] with row stride ldc, not read when beta == 0. D is
 * packed [nrows, ldd]; pre (optional) [nrows, ldpre] receives the fp64 value
 * before rounding. Returns 0, or -1 on a bad argument or an allocation failure.
 */
int oracle_bs_gemm_rows(int64_t M, int64_t N, int64_t K, const uint8_t *A, int64_t lda, int fmt_a,
                        const uint8_t *SA, int64_t ldsa, const uint8_t *Bt, int64_t ldb, int fmt_b,
                        const uint8_t *SB, int64_t ldsb, int sfmt, int block, const void *C, int64_t ldc,
                        double alpha, double beta, int out_dtype, const int64_t *rows, int64_t nrows, void *D,
                        int64_t ldd, double *pre, int64_t ldpre, int nthreads) {
    if (block != 16 && block != 32) return -1;
    if (M < 0 || N < 0 || K < 0 || nrows < 0 || K % block != 0) return -1;
    if (out_dtype != 0 && out_dtype != 1) return -1;
    if (sfmt != ORACLE_SCALE_E8M0 && sfmt != ORACLE_FP8_E4M3) return -1;
    if ((fmt_a != ORACLE_FP8_E4M3 && fmt_a != ORACLE_FP8_E5M2 && fmt_a != ORACLE_FP4_E2M1) ||
        (fmt_b != ORACLE_FP8_E4M3 && fmt_b != ORACLE_FP8_E5M2 && fmt_b != ORACLE_FP4_E2M1))
        return -1;
    if (nrows == 0 || N == 0) return 0;
    const int64_t nb = K / block;
    const int64_t row_a = fmt_a == ORACLE_FP4_E2M1 ? K / 2 : K;
    const int64_t row_b = fmt_b == ORACLE_FP4_E2M1 ? K / 2 : K;
    if (!rows || !D || ldd < N) return -1;
    if (K > 0 && (!A || !Bt || !SA || !SB || lda < row_a || ldb < row_b || ldsa < nb || ldsb < nb)) return -1;
    if (beta != 0.0 && (!C || ldc < N)) return -1;
    if (pre && ldpre < N) return -1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= M) return -1;

    /* B and its scales decoded once, B laid out [K, N] so that the inner loop
     * runs over contiguous columns. */
    double *Bd = (double *)malloc((size_t)(K > 0 ? K : 1) * (size_t)N * sizeof(double));
    double *SBd = (double *)malloc((size_t)(nb > 0 ? nb : 1) * (size_t)N * sizeof(double));
    if (!Bd || !SBd) {
        free(Bd);
        free(SBd);
        return -1;
    }
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t k = 0; k < K; ++k) Bd[k * N + n] = oracle_element(fmt_b, Bt + n * ldb, k);
        for (int64_t b = 0; b < nb; ++b) SBd[b * N + n] = oracle_scale(sfmt, SB[n * ldsb + b]);
    }

    if (nthreads < 1) nthreads = 1;
    if (nthreads > nrows) nthreads = (int)nrows;
    oracle_mx_job *jobs = (oracle_mx_job *)calloc((size_t)nthreads, sizeof(oracle_mx_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    char *spawned = (char *)calloc((size_t)nthreads, 1);
    if (!jobs || !tids || !spawned) {
        free(jobs);
        free(tids);
        free(spawned);
        free(Bd);
        free(SBd);
        return -1;
    }
    for (int t = 0; t < nthreads; ++t) {
        oracle_mx_job *j = &jobs[t];
        j->N = N; j->K = K; j->nb = nb; j->block = block;
        j->A = A; j->lda = lda; j->fmt_a = fmt_a; j->sfmt = sfmt; j->SA = SA; j->ldsa = ldsa;
        j->Bd = Bd; j->SBd = SBd;
        j->C = C; j->ldc = ldc; j->alpha = alpha; j->beta = beta; j->out_dtype = out_dtype;
        j->rows = rows; j->D = D; j->ldd = ldd; j->pre = pre; j->ldpre = ldpre;
        j->row_begin = nrows * t / nthreads;
        j->row_end = nrows * (t + 1) / nthreads;
        j->status = -1;
        if (t > 0) spawned[t] = pthread_create(&tids[t], NULL, oracle_mx_worker, j) == 0;
    }
    oracle_mx_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t) {
        if (spawned[t])
            pthread_join(tids[t], NULL);
        else
            oracle_mx_worker(&jobs[t]);
    }
    int rc = 0;
    for (int t = 0; t < nthreads; ++t)
        if (jobs[t].status != 0) rc = -1;
    free(jobs);
    free(tids);
    free(spawned);
    free(Bd);
    free(SBd);
    return rc;
}

/* The MX (FP8 elements, E8M0 scales, blocks of 32) form of oracle_bs_gemm_rows. */
int oracle_mx_gemm_rows(int64_t M, int64_t N, int64_t K, const uint8_t *A, int64_t lda, int fmt_a,
                        const uint8_t *SA, int64_t ldsa, const uint8_t *Bt, int64_t ldb, int fmt_b,
                        const uint8_t *SB, int64_t ldsb, const void *C, int64_t ldc, double alpha,
                        double beta, int out_dtype, const int64_t *rows, int64_t nrows, void *D,
                        int64_t ldd, double *pre, int64_t ldpre, int nthreads) {
    if ((fmt_a != ORACLE_FP8_E4M3 && fmt_a != ORACLE_FP8_E5M2) ||
        (fmt_b != ORACLE_FP8_E4M3 && fmt_b != ORACLE_FP8_E5M2))
        return -1;
    return oracle_bs_gemm_rows(M, N, K, A, lda, fmt_a, SA, ldsa, Bt, ldb, fmt_b, SB, ldsb, ORACLE_SCALE_E8M0,
                               ORACLE_MX_BLOCK, C, ldc, alpha, beta, out_dtype, rows, nrows, D, ldd, pre, ldpre,
                               nthreads);
}
