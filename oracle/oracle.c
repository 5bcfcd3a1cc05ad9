/*
 * Plain CPU oracle for the tile-partitioned dense matrix multiply
 *
 *     D = alpha * A * B + beta * C
 *
 * TEST INFRASTRUCTURE ONLY. This file is compiled into liboracle.so, which only
 * the test suite, the package smoke check and the benchmark's CPU-baseline leg
 * load. The product path (the CUDA library and its Python binding) never links,
 * imports or calls it, and the two share no source: not a header, not a
 * conversion helper, not a constant.
 *
 * What it computes, and where that comes from:
 *  - "TorchInductor ganha suporte a GEMMs de alta performance com CuteDSL"
 *    (the paragraph on where transformer cycles go): the GEMMs of attention
 *    projections and fully-connected layers are the operation.
 *  - Same page, epilogue-fusion roadmap paragraph: the epilogue loads an
 *    auxiliary tensor and adds it element-wise; here that is beta * C.
 *  - "cuTile Rust explained", sections "Ownership crosses the launch boundary"
 *    and "The useful boundary": each tile program owns one disjoint output
 *    sub-tensor and reads shared immutable inputs. Ownership does not change
 *    the arithmetic, so the oracle is the untiled definition itself.
 *  The pages never write the formula, the dtypes or a rounding rule. The
 *  reading taken here: A, B are bf16; every product is formed exactly in fp64
 *  (a bf16 x bf16 product has at most 16 significant bits); products are summed
 *  in fp64 in ascending k; then alpha*acc and beta*C are formed in fp64 as two
 *  separate operations (no contraction: built with -ffp-contract=off); the
 *  result is rounded ONCE, round-to-nearest-even, to the output dtype (fp32 or
 *  bf16). fp64 -> bf16 goes directly, never through fp32, so there is no double
 *  rounding. When beta == 0 C is not read (it may be NULL).
 *
 * Loop order is i-k-j with one fp64 accumulator per output element of the row,
 * which keeps the per-element summation order k = 0, 1, ..., K-1.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OUT_BF16 0
#define ORACLE_OUT_F32 1

/* bf16 is the upper half of an IEEE binary32 pattern. */
static double oracle_decode_bf16(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double oracle_decode_f32(const void *p) {
    float f;
    memcpy(&f, p, sizeof f);
    return (double)f;
}

/*
 * fp64 -> bf16, round to nearest, ties to even, in one step.
 * bf16 has 8 significand bits (7 stored) and fp32's exponent range, so its
 * quantum at binade e (2^e <= |x| < 2^(e+1)) is 2^(e-7), with e clamped to the
 * smallest normal exponent -126 (below it the quantum stays 2^-133:
 * subnormals). Scaling by a power of two is exact, nearbyint() rounds to an
 * integer under the default ties-to-even mode, and scaling back is exact.
 * A result of magnitude >= 2^128 is outside bf16's finite range: +-inf.
 * NaN maps to the canonical quiet NaN 0x7FC0. Signed zeros are kept.
 */
uint16_t oracle_round_bf16(double x) {
    if (isnan(x)) return 0x7FC0u;
    const uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isinf(x)) return (uint16_t)(sign | 0x7F80u);
    if (x == 0.0) return sign;
    int e = ilogb(x);
    if (e < -126) e = -126;
    const double r = nearbyint(ldexp(x, 7 - e));
    const double y = ldexp(r, e - 7);
    if (fabs(y) >= 0x1p128) return (uint16_t)(sign | 0x7F80u);
    /* y is a bf16 value, so its binary32 encoding ends in 16 zero bits. */
    const float f = (float)y;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)((u >> 16) | sign); /* sign kept for -0 from a tiny negative */
}

/* fp64 -> fp32: C's conversion, which is IEEE round-to-nearest-even. */
float oracle_round_f32(double x) { return (float)x; }

/* Batch forms used by the exhaustive rounding pin. */
void oracle_round_bf16_from_f32_bits(const uint32_t *in, uint16_t *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) {
        float f;
        memcpy(&f, &in[i], sizeof f);
        out[i] = oracle_round_bf16((double)f);
    }
}

void oracle_round_bf16_array(const double *in, uint16_t *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_round_bf16(in[i]);
}

/*
 * Fused epilogue (the EFC capabilities listed in the epilogue-fusion roadmap
 * paragraph of "TorchInductor ganha suporte a GEMMs de alta performance com
 * CuteDSL": auxiliary tensor loads, element-wise add and mul, activations
 * ReLU, sigmoid and tanh). The order, a reading of the page, is
 *     v = alpha*acc + beta*C;  v = v + bias[n];  v = act(v);  v = v * aux[m,n]
 * all in fp64 (libm exp and tanh), then one rounding to the output dtype.
 */
#define ORACLE_ACT_NONE 0
#define ORACLE_ACT_RELU 1
#define ORACLE_ACT_SIGMOID 2
#define ORACLE_ACT_TANH 3

static double oracle_activation(int act, double v) {
    switch (act) {
    case ORACLE_ACT_RELU: return v > 0.0 ? v : 0.0;
    case ORACLE_ACT_SIGMOID: return 1.0 / (1.0 + exp(-v));
    case ORACLE_ACT_TANH: return tanh(v);
    default: return v;
    }
}

typedef struct {
    const void *bias; /* NULL or [N] of bias_dtype */
    int bias_dtype;
    int act;
    const void *aux; /* NULL or [M, N] of the output dtype, row stride ldaux */
    int64_t ldaux;
} oracle_epilogue;

typedef struct {
    int64_t N, K;
    const uint16_t *A;
    int64_t lda;
    const uint16_t *B;
    int64_t ldb;
    const void *C;
    int64_t ldc;
    double alpha, beta;
    int out_dtype;
    const int64_t *rows;
    int64_t row_begin, row_end; /* indices into rows[] */
    void *D;
    int64_t ldd; /* row stride of D, in elements; D row r holds output row rows[r] */
    double *pre;
    int64_t ldpre; /* row stride of pre; NULL pre = not wanted */
    const oracle_epilogue *epi; /* NULL = plain alpha*acc + beta*C */
    int status;
} oracle_job;

static double oracle_decode_out(int out_dtype, const void *base, int64_t idx) {
    if (out_dtype == ORACLE_OUT_BF16) return oracle_decode_bf16(((const uint16_t *)base)[idx]);
    return oracle_decode_f32((const float *)base + idx);
}

static void *oracle_rows_worker(void *arg) {
    oracle_job *j = (oracle_job *)arg;
    double *acc = (double *)malloc((size_t)(j->N > 0 ? j->N : 1) * sizeof(double));
    if (!acc) {
        j->status = -1;
        return NULL;
    }
    for (int64_t r = j->row_begin; r < j->row_end; ++r) {
        const int64_t i = j->rows[r];
        for (int64_t n = 0; n < j->N; ++n) acc[n] = 0.0;
        /* acc[n] = sum over k ascending of A[i,k] * B[k,n], each product exact. */
        for (int64_t k = 0; k < j->K; ++k) {
            const double a = oracle_decode_bf16(j->A[i * j->lda + k]);
            const uint16_t *brow = j->B + k * j->ldb;
            for (int64_t n = 0; n < j->N; ++n) acc[n] += a * oracle_decode_bf16(brow[n]);
        }
        for (int64_t n = 0; n < j->N; ++n) {
            double v = j->alpha * acc[n];
            if (j->beta != 0.0) {
                double c;
                if (j->out_dtype == ORACLE_OUT_BF16)
                    c = oracle_decode_bf16(((const uint16_t *)j->C)[i * j->ldc + n]);
                else
                    c = oracle_decode_f32((const float *)j->C + i * j->ldc + n);
                v = v + j->beta * c;
            }
            if (j->epi) {
                const oracle_epilogue *e = j->epi;
                if (e->bias) v = v + oracle_decode_out(e->bias_dtype, e->bias, n);
                v = oracle_activation(e->act, v);
                if (e->aux) v = v * oracle_decode_out(j->out_dtype, e->aux, i * e->ldaux + n);
            }
            if (j->pre) j->pre[r * j->ldpre + n] = v;
            if (j->out_dtype == ORACLE_OUT_BF16)
                ((uint16_t *)j->D)[r * j->ldd + n] = oracle_round_bf16(v);
            else
                ((float *)j->D)[r * j->ldd + n] = oracle_round_f32(v);
        }
    }
    free(acc);
    j->status = 0;
    return NULL;
}

/*
 * Computes the output rows listed in rows[0..nrows) of D = alpha*A*B + beta*C.
 *   A: bf16 bits, row-major [M, K] with row stride lda (elements)
 *   B: bf16 bits, row-major [K, N] with row stride ldb
 *   C: out_dtype, row-major [M, N] with row stride ldc; not read if beta == 0
 *   D: out_dtype, packed [nrows, ldd]; D row r receives output row rows[r]
 *   pre: optional fp64 [nrows, ldpre], the value before the final rounding
 * nthreads <= 0 means one thread. Returns 0, or -1 on a bad argument or an
 * allocation failure.
 */
static int oracle_gemm_rows_impl(int64_t M, int64_t N, int64_t K, const uint16_t *A, int64_t lda,
                                 const uint16_t *B, int64_t ldb, const void *C, int64_t ldc,
                                 double alpha, double beta, int out_dtype, const int64_t *rows,
                                 int64_t nrows, void *D, int64_t ldd, double *pre, int64_t ldpre,
                                 int nthreads, const oracle_epilogue *epi) {
    if (M < 0 || N < 0 || K < 0 || nrows < 0) return -1;
    if (out_dtype != ORACLE_OUT_BF16 && out_dtype != ORACLE_OUT_F32) return -1;
    if (nrows == 0 || N == 0) return 0;
    if (!rows || !D || ldd < N) return -1;
    if (K > 0 && (!A || !B || lda < K || ldb < N)) return -1;
    if (beta != 0.0 && (!C || ldc < N)) return -1;
    if (pre && ldpre < N) return -1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= M) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > nrows) nthreads = (int)nrows;

    oracle_job *jobs = (oracle_job *)calloc((size_t)nthreads, sizeof(oracle_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    char *spawned = (char *)calloc((size_t)nthreads, 1);
    if (!jobs || !tids || !spawned) {
        free(jobs);
        free(tids);
        free(spawned);
        return -1;
    }
    for (int t = 0; t < nthreads; ++t) {
        oracle_job *j = &jobs[t];
        j->N = N; j->K = K; j->A = A; j->lda = lda; j->B = B; j->ldb = ldb;
        j->C = C; j->ldc = ldc; j->alpha = alpha; j->beta = beta; j->out_dtype = out_dtype;
        j->rows = rows; j->D = D; j->ldd = ldd; j->pre = pre; j->ldpre = ldpre; j->epi = epi;
        j->row_begin = nrows * t / nthreads;
        j->row_end = nrows * (t + 1) / nthreads;
        j->status = -1;
        /* the calling thread takes share 0; a share whose thread cannot start runs here */
        if (t > 0) spawned[t] = pthread_create(&tids[t], NULL, oracle_rows_worker, j) == 0;
    }
    oracle_rows_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t) {
        if (spawned[t])
            pthread_join(tids[t], NULL);
        else
            oracle_rows_worker(&jobs[t]);
    }
    int rc = 0;
    for (int t = 0; t < nthreads; ++t)
        if (jobs[t].status != 0) rc = -1;
    free(jobs);
    free(tids);
    free(spawned);
    return rc;
}

int oracle_gemm_rows(int64_t M, int64_t N, int64_t K, const uint16_t *A, int64_t lda,
                     const uint16_t *B, int64_t ldb, const void *C, int64_t ldc, double alpha,
                     double beta, int out_dtype, const int64_t *rows, int64_t nrows, void *D,
                     int64_t ldd, double *pre, int64_t ldpre, int nthreads) {
    return oracle_gemm_rows_impl(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, out_dtype, rows,
                                 nrows, D, ldd, pre, ldpre, nthreads, NULL);
}

/* oracle_gemm_rows plus the fused epilogue described above oracle_activation. */
int oracle_gemm_rows_epilogue(int64_t M, int64_t N, int64_t K, const uint16_t *A, int64_t lda,
                              const uint16_t *B, int64_t ldb, const void *C, int64_t ldc,
                              double alpha, double beta, int out_dtype, const int64_t *rows,
                              int64_t nrows, void *D, int64_t ldd, double *pre, int64_t ldpre,
                              int nthreads, const void *bias, int bias_dtype, int act,
                              const void *aux, int64_t ldaux) {
    if (act < ORACLE_ACT_NONE || act > ORACLE_ACT_TANH) return -1;
    if (bias && bias_dtype != ORACLE_OUT_BF16 && bias_dtype != ORACLE_OUT_F32) return -1;
    if (aux && ldaux < N) return -1;
    oracle_epilogue e = {bias, bias_dtype, act, aux, ldaux};
    return oracle_gemm_rows_impl(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, out_dtype, rows,
                                 nrows, D, ldd, pre, ldpre, nthreads, &e);
}

/* The activation alone, for its pins. */
double oracle_act(int act, double v) { return oracle_activation(act, v); }
