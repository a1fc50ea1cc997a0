/*
 * oracle.c -- plain, slow, obviously correct CPU statement of what the hot path
 * computes.  TEST INFRASTRUCTURE ONLY: nothing in the product library links,
 * loads or calls this file.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA path.
 *
 * Everything accumulates in IEEE double.  Every product formed here is exact in
 * double: fp32*fp32 needs at most 48 significant bits, and
 * fp16 scale * fp32 codebook entry * fp16 activation at most 11+24+11 = 46.
 * Each output also gets T = sum_k |term_k|, the scale of the acceptance bound
 * |y - y_ref| <= 1e-5 * T.
 *
 * Sources (page title, section):
 *  - "I built a GPT-2 in the browser, then made it 2.6x-12.1x faster",
 *    section "The kernel sweep": the matmul as one output cell per (row,
 *    column), walking the inner dimension and summing products.
 *  - "More Stumbling, This Time in the Browser", section "Four answers per
 *    worker": row = token, column = output feature, each cell walks the inner
 *    dimension multiplying activation by weight and adding.
 *  - "Kernel 0112", section "What is being measured": 12,288 x 1,536 weights
 *    stored in 2 bits each times a vector of 1,536 inputs; section "How it is
 *    measured": a plain CPU computation of the outputs is the reference answer.
 *
 * Readings where the pages are silent:
 *  - storage is row-major; transA means op(A) = A^T with A stored K x M,
 *    transB means op(B) = B^T with B stored N x K; C is overwritten.
 *  - 2-bit field of element k in a packed row: byte floor(k/4), bits
 *    2*(k mod 4) and 2*(k mod 4)+1 (little-endian along K); a row has
 *    ceil(cols/4) bytes and unused high fields of its last byte are ignored.
 *  - a field selects one of 4 codebook entries; the per-row fp16 scale
 *    multiplies the entry.
 *  - 4-bit codes (the 16-entry codebook of "Kernel 0112", section "What the
 *    kernel costs in a whole token": the 4-bit weight-reading kernels, and of
 *    "More Stumbling, This Time in the Browser": the packed NF4 path): element
 *    k of a packed row is in byte floor(k/2), bits 4*(k mod 2)..4*(k mod 2)+3
 *    (low nibble first, little-endian along K like the 2-bit codes); a row has
 *    ceil(cols/2) bytes; the field selects one of 16 codebook entries.
 *
 * Loop nesting: each output's sum runs over k = 0..K-1 in increasing order.
 * The nesting of the i/j loops only changes which output is visited when, not
 * the order of any sum.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* IEEE 754 binary16 -> double, from the format's definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * exponent 0: subnormal, value = fraction * 2^-24; exponent 31: inf / NaN. */
double orc_half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);
    } else if (e == 31) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + f), e - 25);
    }
    return sign ? -v : v;
}

/* field value of element k of one packed row */
int orc_code2(const uint8_t *row, int64_t k) {
    uint8_t byte = row[k / 4];
    int shift = 2 * (int)(k % 4);
    return (byte >> shift) & 3;
}

int64_t orc_row_bytes(int64_t cols) { return (cols + 3) / 4; }

/* out[r*cols + k] = field of element (r, k) */
void orc_unpack2(const uint8_t *codes, int64_t rows, int64_t cols, uint8_t *out) {
    int64_t rb = orc_row_bytes(cols);
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t k = 0; k < cols; ++k)
            out[r * cols + k] = (uint8_t)orc_code2(codes + r * rb, k);
}

/* inverse of orc_unpack2; fields must be in 0..3; unused bits of a row's last byte are 0 */
void orc_pack2(const uint8_t *fields, int64_t rows, int64_t cols, uint8_t *codes) {
    int64_t rb = orc_row_bytes(cols);
    memset(codes, 0, (size_t)(rows * rb));
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t k = 0; k < cols; ++k) {
            uint8_t v = fields[r * cols + k] & 3;
            codes[r * rb + k / 4] |= (uint8_t)(v << (2 * (k % 4)));
        }
}

/* 4-bit field of element k of one packed row: byte floor(k/2), low nibble first */
int orc_code4(const uint8_t *row, int64_t k) {
    uint8_t byte = row[k / 2];
    int shift = 4 * (int)(k % 2);
    return (byte >> shift) & 15;
}

int64_t orc_row_bytes4(int64_t cols) { return (cols + 1) / 2; }

/* out[r*cols + k] = 4-bit field of element (r, k) */
void orc_unpack4(const uint8_t *codes, int64_t rows, int64_t cols, uint8_t *out) {
    int64_t rb = orc_row_bytes4(cols);
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t k = 0; k < cols; ++k)
            out[r * cols + k] = (uint8_t)orc_code4(codes + r * rb, k);
}

/* inverse of orc_unpack4; fields must be in 0..15; an odd row's unused high nibble is 0 */
void orc_pack4(const uint8_t *fields, int64_t rows, int64_t cols, uint8_t *codes) {
    int64_t rb = orc_row_bytes4(cols);
    memset(codes, 0, (size_t)(rows * rb));
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t k = 0; k < cols; ++k) {
            uint8_t v = fields[r * cols + k] & 15;
            codes[r * rb + k / 2] |= (uint8_t)(v << (4 * (k % 2)));
        }
}

/* field of element k of a packed row with `bits` bits per field (2 or 4) */
static int packed_code(const uint8_t *row, int64_t k, int bits) {
    return bits == 4 ? orc_code4(row, k) : orc_code2(row, k);
}

static int64_t packed_row_bytes(int64_t cols, int bits) {
    return bits == 4 ? orc_row_bytes4(cols) : orc_row_bytes(cols);
}

/* ------------------------------------------------------------------------ */
/* Dense GEMM: C[i][j] = sum_k opA(i,k) * opB(k,j)                          */
/* ------------------------------------------------------------------------ */

static inline double opA(const float *A, int64_t lda, int transA, int64_t i, int64_t k) {
    return transA ? (double)A[k * lda + i] : (double)A[i * lda + k];
}
static inline double opB(const float *B, int64_t ldb, int transB, int64_t k, int64_t j) {
    return transB ? (double)B[j * ldb + k] : (double)B[k * ldb + j];
}

typedef struct {
    int transA, transB;
    int64_t M, N, K;
    const float *A;
    int64_t lda;
    const float *B;
    int64_t ldb;
    double *C, *T;
    int64_t i0, i1;
} gemm_job;

static void gemm_rows(const gemm_job *g) {
    for (int64_t i = g->i0; i < g->i1; ++i) {
        double *c = g->C + i * g->N;
        double *t = g->T + i * g->N;
        if (g->transB) {
            /* i, j, k: both op(A) row i and stored row j of B run along k */
            for (int64_t j = 0; j < g->N; ++j) {
                double s = 0.0, a = 0.0;
                for (int64_t k = 0; k < g->K; ++k) {
                    double p = opA(g->A, g->lda, g->transA, i, k) * opB(g->B, g->ldb, 1, k, j);
                    s += p;
                    a += fabs(p);
                }
                c[j] = s;
                t[j] = a;
            }
        } else {
            /* i, k, j: stored row k of B runs along j; every c[j] still sums k upward */
            for (int64_t j = 0; j < g->N; ++j) { c[j] = 0.0; t[j] = 0.0; }
            for (int64_t k = 0; k < g->K; ++k) {
                double a = opA(g->A, g->lda, g->transA, i, k);
                const float *brow = g->B + k * g->ldb;
                for (int64_t j = 0; j < g->N; ++j) {
                    double p = a * (double)brow[j];
                    c[j] += p;
                    t[j] += fabs(p);
                }
            }
        }
    }
}

static void *gemm_thread(void *arg) {
    gemm_rows((const gemm_job *)arg);
    return NULL;
}

/* C and T are M x N, row-major, dense. */
void orc_gemm(int transA, int transB, int64_t M, int64_t N, int64_t K,
              const float *A, int64_t lda, const float *B, int64_t ldb,
              double *C, double *T, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > M) nthreads = (int)(M > 0 ? M : 1);
    gemm_job *jobs = (gemm_job *)calloc((size_t)nthreads, sizeof(gemm_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    for (int t = 0; t < nthreads; ++t) {
        gemm_job g = {transA, transB, M, N, K, A, lda, B, ldb, C, T,
                      M * t / nthreads, M * (t + 1) / nthreads};
        jobs[t] = g;
    }
    for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, gemm_thread, &jobs[t]);
    gemm_rows(&jobs[0]);
    for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
    free(jobs);
    free(th);
}

/* Selected outputs only: C[n] = C(ii[n], jj[n]). */
void orc_gemm_at(int transA, int transB, int64_t K,
                 const float *A, int64_t lda, const float *B, int64_t ldb,
                 int64_t n, const int64_t *ii, const int64_t *jj, double *C, double *T) {
    for (int64_t q = 0; q < n; ++q) {
        double s = 0.0, a = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double p = opA(A, lda, transA, ii[q], k) * opB(B, ldb, transB, k, jj[q]);
            s += p;
            a += fabs(p);
        }
        C[q] = s;
        T[q] = a;
    }
}

/* ------------------------------------------------------------------------ */
/* Packed 2-bit (or 4-bit) weights:                                         */
/*   Y[m][r] = sum_k scale_r * codebook[field(r,k)] * X[m][k]               */
/* codes: rows x ceil(cols/4) bytes (4-bit: ceil(cols/2)); scales: rows fp16; */
/* X: M x cols fp16.  A GEMV is the M = 1 case.                             */
/* ------------------------------------------------------------------------ */

typedef struct {
    const uint8_t *codes;
    const uint16_t *scales;
    const uint16_t *X;
    int64_t M, rows, cols;
    const float *codebook;
    double *Y, *T;
    int64_t m0, m1;
    int bits;
} packed_job;

static void packed_rows(const packed_job *g) {
    int64_t rb = packed_row_bytes(g->cols, g->bits);
    for (int64_t m = g->m0; m < g->m1; ++m) {
        for (int64_t r = 0; r < g->rows; ++r) {
            const uint8_t *row = g->codes + r * rb;
            double s = orc_half_to_double(g->scales[r]);
            double acc = 0.0, abs_acc = 0.0;
            for (int64_t k = 0; k < g->cols; ++k) {
                double w = (double)g->codebook[packed_code(row, k, g->bits)];
                double x = orc_half_to_double(g->X[m * g->cols + k]);
                double p = s * w * x;
                acc += p;
                abs_acc += fabs(p);
            }
            g->Y[m * g->rows + r] = acc;
            g->T[m * g->rows + r] = abs_acc;
        }
    }
}

static void *packed_thread(void *arg) {
    packed_rows((const packed_job *)arg);
    return NULL;
}

/* Y and T are M x rows, row-major.  Threads split the M rows of X when M > 1,
 * otherwise the weight rows. */
static void packed_gemm_bits(const uint8_t *codes, const uint16_t *scales, const uint16_t *X,
                             int64_t M, int64_t rows, int64_t cols, const float *codebook,
                             double *Y, double *T, int nthreads, int bits) {
    if (nthreads < 1) nthreads = 1;
    if (M == 1) {
        /* split weight rows: each thread sees a slice of the matrix */
        if (nthreads > rows) nthreads = (int)(rows > 0 ? rows : 1);
        packed_job *jobs = (packed_job *)calloc((size_t)nthreads, sizeof(packed_job));
        pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
        int64_t rb = packed_row_bytes(cols, bits);
        for (int t = 0; t < nthreads; ++t) {
            int64_t r0 = rows * t / nthreads, r1 = rows * (t + 1) / nthreads;
            packed_job g = {codes + r0 * rb, scales + r0, X, 1, r1 - r0, cols, codebook,
                            Y + r0, T + r0, 0, 1, bits};
            jobs[t] = g;
        }
        for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, packed_thread, &jobs[t]);
        packed_rows(&jobs[0]);
        for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
        free(jobs);
        free(th);
        return;
    }
    if (nthreads > M) nthreads = (int)(M > 0 ? M : 1);
    packed_job *jobs = (packed_job *)calloc((size_t)nthreads, sizeof(packed_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    for (int t = 0; t < nthreads; ++t) {
        packed_job g = {codes, scales, X, M, rows, cols, codebook, Y, T,
                        M * t / nthreads, M * (t + 1) / nthreads, bits};
        jobs[t] = g;
    }
    for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, packed_thread, &jobs[t]);
    packed_rows(&jobs[0]);
    for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
    free(jobs);
    free(th);
}

void orc_packed_gemm(const uint8_t *codes, const uint16_t *scales, const uint16_t *X,
                     int64_t M, int64_t rows, int64_t cols, const float *codebook,
                     double *Y, double *T, int nthreads) {
    packed_gemm_bits(codes, scales, X, M, rows, cols, codebook, Y, T, nthreads, 2);
}

/* 4-bit codes, 16-entry codebook */
void orc_packed4_gemm(const uint8_t *codes, const uint16_t *scales, const uint16_t *X,
                      int64_t M, int64_t rows, int64_t cols, const float *codebook,
                      double *Y, double *T, int nthreads) {
    packed_gemm_bits(codes, scales, X, M, rows, cols, codebook, Y, T, nthreads, 4);
}

/* Selected outputs only: Y[n] = Y(mm[n], rr[n]). */
static void packed_gemm_at_bits(const uint8_t *codes, const uint16_t *scales, const uint16_t *X,
                                int64_t cols, const float *codebook, int64_t n, const int64_t *mm,
                                const int64_t *rr, double *Y, double *T, int bits) {
    int64_t rb = packed_row_bytes(cols, bits);
    for (int64_t q = 0; q < n; ++q) {
        const uint8_t *row = codes + rr[q] * rb;
        double s = orc_half_to_double(scales[rr[q]]);
        double acc = 0.0, abs_acc = 0.0;
        for (int64_t k = 0; k < cols; ++k) {
            double p = s * (double)codebook[packed_code(row, k, bits)] *
                       orc_half_to_double(X[mm[q] * cols + k]);
            acc += p;
            abs_acc += fabs(p);
        }
        Y[q] = acc;
        T[q] = abs_acc;
    }
}

void orc_packed_gemm_at(const uint8_t *codes, const uint16_t *scales, const uint16_t *X,
                        int64_t cols, const float *codebook,
                        int64_t n, const int64_t *mm, const int64_t *rr, double *Y, double *T) {
    packed_gemm_at_bits(codes, scales, X, cols, codebook, n, mm, rr, Y, T, 2);
}

void orc_packed4_gemm_at(const uint8_t *codes, const uint16_t *scales, const uint16_t *X,
                         int64_t cols, const float *codebook,
                         int64_t n, const int64_t *mm, const int64_t *rr, double *Y, double *T) {
    packed_gemm_at_bits(codes, scales, X, cols, codebook, n, mm, rr, Y, T, 4);
}
