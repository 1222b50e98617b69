/*
 * CPU oracle for the dense GEMM  C = alpha * op(A) * op(B) + beta * C_in + bias.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark do.  It shares no code, header or table with the CUDA library.
 *
 * What it computes (the plain definition, written out):
 *   "Matrix Multiplication: The Operation Behind Modern AI", section
 *   "One formula for every matmul" and the opening definition: for an M x K
 *   matrix A and a K x N matrix B, C_ij = sum_k A_ik * B_kj, 2*M*N*K flops.
 *   The epilogue alpha*S + beta*C_in + bias (bias broadcast over rows and not
 *   scaled by alpha) is the BLAS-style reading of the library call
 *   gemm_run(..., alpha, beta, bias*).
 *
 * Arithmetic: every stored f16 / bf16 / f32 input is decoded EXACTLY to f64
 * by bit manipulation from the IEEE-754 binary16 and the bfloat16 definitions
 * (no GPU header, no library conversion).  Each product of two decoded half
 * values is exact in f64 (11+11 or 8+8 significand bits <= 53).  The sum over
 * k runs in ascending k with an f64 accumulator; the epilogue is evaluated in
 * f64 and the result is returned UNROUNDED (no cast to the output dtype).
 *
 * Loop order is i-k-j (row accumulator, contiguous inner loop), which is still
 * the plain definition.  Threads split the list of output rows; nothing else is
 * blocked, fused or reordered.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* dtype codes used by the oracle's own interface (E4M3 and E5M2 are inputs only) */
enum { OR_F16 = 0, OR_BF16 = 1, OR_F32 = 2, OR_E4M3 = 3, OR_E5M2 = 4 };
/* layout codes: A ROW = M x K with K contiguous, A COL = stored K x M (M contiguous);
 *               B ROW = K x N with N contiguous, B COL = stored N x K (K contiguous). */
enum { OR_ROW = 0, OR_COL = 1 };

/* IEEE-754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double oracle_f16_to_f64(uint16_t h) {
    const unsigned sign = (h >> 15) & 1u;
    const unsigned expo = (h >> 10) & 0x1fu;
    const unsigned frac = h & 0x3ffu;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24);                     /* subnormal: frac * 2^(1-15-10) */
    } else if (expo == 0x1f) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(frac | 0x400u), (int)expo - 25); /* (2^10 + frac) * 2^(e-15-10) */
    }
    return sign ? -v : v;
}

/* bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits (the top half of a binary32). */
double oracle_bf16_to_f64(uint16_t b) {
    const unsigned sign = (b >> 15) & 1u;
    const unsigned expo = (b >> 7) & 0xffu;
    const unsigned frac = b & 0x7fu;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -133);                    /* subnormal: frac * 2^(1-127-7) */
    } else if (expo == 0xff) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(frac | 0x80u), (int)expo - 134); /* (2^7 + frac) * 2^(e-127-7) */
    }
    return sign ? -v : v;
}

/* IEEE-754 binary32: 1 sign, 8 exponent (bias 127), 23 fraction bits. */
double oracle_f32_to_f64(uint32_t w) {
    const unsigned sign = (w >> 31) & 1u;
    const unsigned expo = (w >> 23) & 0xffu;
    const unsigned frac = w & 0x7fffffu;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -149);
    } else if (expo == 0xff) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(frac | 0x800000u), (int)expo - 150);
    }
    return sign ? -v : v;
}

/* 8-bit floats, from the OCP "8-bit floating point" definitions (the FP8 formats of the tensor
 * cores the matrix-multiplication page mentions):
 *   E4M3: 1 sign, 4 exponent (bias 7), 3 fraction bits; exponent field 0 is subnormal
 *         (frac * 2^-9); no infinities; S.1111.111 is NaN, so the largest value is 448.
 *   E5M2: 1 sign, 5 exponent (bias 15), 2 fraction bits; IEEE-754 style: exponent 0 is
 *         subnormal (frac * 2^-16), exponent 31 is infinity (frac 0) or NaN. */
double oracle_e4m3_to_f64(uint8_t b) {
    const unsigned sign = (b >> 7) & 1u;
    const unsigned expo = (b >> 3) & 0xfu;
    const unsigned frac = b & 0x7u;
    double v;
    if (expo == 0xf && frac == 0x7) return NAN;
    if (expo == 0) v = ldexp((double)frac, -9);                        /* frac * 2^(1-7-3) */
    else v = ldexp((double)(frac | 0x8u), (int)expo - 10);             /* (8 + frac) * 2^(e-7-3) */
    return sign ? -v : v;
}

double oracle_e5m2_to_f64(uint8_t b) {
    const unsigned sign = (b >> 7) & 1u;
    const unsigned expo = (b >> 2) & 0x1fu;
    const unsigned frac = b & 0x3u;
    double v;
    if (expo == 0) v = ldexp((double)frac, -16);                       /* frac * 2^(1-15-2) */
    else if (expo == 0x1f) v = frac ? NAN : INFINITY;
    else v = ldexp((double)(frac | 0x4u), (int)expo - 17);             /* (4 + frac) * 2^(e-15-2) */
    return sign ? -v : v;
}

static double load_elem(const void* base, int64_t idx, int dtype) {
    if (dtype == OR_F16) return oracle_f16_to_f64(((const uint16_t*)base)[idx]);
    if (dtype == OR_BF16) return oracle_bf16_to_f64(((const uint16_t*)base)[idx]);
    if (dtype == OR_E4M3) return oracle_e4m3_to_f64(((const uint8_t*)base)[idx]);
    if (dtype == OR_E5M2) return oracle_e5m2_to_f64(((const uint8_t*)base)[idx]);
    return oracle_f32_to_f64(((const uint32_t*)base)[idx]);
}

/* op(A)_ik and op(B)_kj as stored */
static int64_t a_index(int64_t i, int64_t k, int64_t lda, int layout) {
    return layout == OR_ROW ? i * lda + k : k * lda + i;
}
static int64_t b_index(int64_t k, int64_t j, int64_t ldb, int layout) {
    return layout == OR_ROW ? k * ldb + j : j * ldb + k;
}

typedef struct {
    int64_t M, N, K;
    const void* A; int64_t lda; int layoutA;
    const double* Bd;           /* op(B) decoded, K x N row-major */
    int dtype_in;
    double alpha, beta;
    const void* Cin; int64_t ldcin; int dtype_cin;
    const double* biasd;        /* decoded bias (N) or NULL */
    const int64_t* rows; int64_t nrows;
    const int64_t* cols; int64_t ncols;   /* NULL = all N columns */
    double* out; int64_t ldout;           /* out[r * ldout + c], r over rows list, c over cols list */
    int64_t r_begin, r_end;
} job_t;

static void* worker(void* p) {
    job_t* j = (job_t*)p;
    const int64_t nc = j->cols ? j->ncols : j->N;
    double* acc = (double*)malloc(sizeof(double) * (size_t)(nc > 0 ? nc : 1));
    double* arow = (double*)malloc(sizeof(double) * (size_t)(j->K > 0 ? j->K : 1));
    for (int64_t r = j->r_begin; r < j->r_end; ++r) {
        const int64_t i = j->rows[r];
        for (int64_t k = 0; k < j->K; ++k)
            arow[k] = load_elem(j->A, a_index(i, k, j->lda, j->layoutA), j->dtype_in);
        for (int64_t c = 0; c < nc; ++c) acc[c] = 0.0;
        /* S_ij = sum_k a_ik * b_kj, k ascending */
        for (int64_t k = 0; k < j->K; ++k) {
            const double a = arow[k];
            const double* brow = j->Bd + k * j->N;
            if (j->cols) {
                for (int64_t c = 0; c < nc; ++c) acc[c] += a * brow[j->cols[c]];
            } else {
                for (int64_t c = 0; c < nc; ++c) acc[c] += a * brow[c];
            }
        }
        /* epilogue: alpha * S + beta * C_in + bias; C_in is not read when beta == 0 */
        double* orow = j->out + r * j->ldout;
        for (int64_t c = 0; c < nc; ++c) {
            const int64_t col = j->cols ? j->cols[c] : c;
            double v = j->alpha * acc[c];
            if (j->beta != 0.0) v += j->beta * load_elem(j->Cin, i * j->ldcin + col, j->dtype_cin);
            if (j->biasd) v += j->biasd[col];
            orow[c] = v;
        }
    }
    free(acc);
    free(arow);
    return NULL;
}

int oracle_num_cpus(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/*
 * Reference result on a sub-grid of C.
 *   rows[nrows]   output rows to compute (NULL = all M rows, nrows ignored)
 *   cols[ncols]   output columns to compute (NULL = all N columns)
 *   out           f64, out[r * ldout + c] for r < nrows, c < ncols
 *   bias          NULL or N elements of dtype_bias
 *   Cin           read only when beta != 0; element (i, j) at Cin[i * ldcin + j]
 *   nthreads      <= 0 means every online CPU
 * Returns 0 on success, -1 on a bad argument or an allocation failure.
 */
int oracle_gemm(int64_t M, int64_t N, int64_t K,
                const void* A, int64_t lda, int layoutA,
                const void* B, int64_t ldb, int layoutB,
                int dtype_in,
                double alpha, double beta,
                const void* Cin, int64_t ldcin, int dtype_cin,
                const void* bias, int dtype_bias,
                const int64_t* rows, int64_t nrows,
                const int64_t* cols, int64_t ncols,
                double* out, int64_t ldout,
                int nthreads) {
    if (M < 0 || N < 0 || K < 0 || !out) return -1;
    if (K > 0 && (!A || !B)) return -1;
    if (beta != 0.0 && !Cin) return -1;
    int64_t* all_rows = NULL;
    if (!rows) {
        all_rows = (int64_t*)malloc(sizeof(int64_t) * (size_t)(M > 0 ? M : 1));
        if (!all_rows) return -1;
        for (int64_t i = 0; i < M; ++i) all_rows[i] = i;
        rows = all_rows;
        nrows = M;
    }
    if (nrows == 0) { free(all_rows); return 0; }
    /* decode op(B) once into a K x N f64 row-major array */
    double* Bd = (double*)malloc(sizeof(double) * (size_t)((K * N) > 0 ? K * N : 1));
    double* biasd = NULL;
    if (!Bd) { free(all_rows); return -1; }
    for (int64_t k = 0; k < K; ++k)
        for (int64_t j = 0; j < N; ++j)
            Bd[k * N + j] = load_elem(B, b_index(k, j, ldb, layoutB), dtype_in);
    if (bias) {
        biasd = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
        if (!biasd) { free(Bd); free(all_rows); return -1; }
        for (int64_t j = 0; j < N; ++j) biasd[j] = load_elem(bias, j, dtype_bias);
    }
    if (nthreads <= 0) nthreads = oracle_num_cpus();
    if (nthreads > nrows) nthreads = (int)nrows;
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    job_t* jobs = (job_t*)malloc(sizeof(job_t) * (size_t)nthreads);
    int rc = 0;
    if (!th || !jobs) rc = -1;
    int started = 0;
    for (int t = 0; rc == 0 && t < nthreads; ++t) {
        job_t* j = &jobs[t];
        j->M = M; j->N = N; j->K = K;
        j->A = A; j->lda = lda; j->layoutA = layoutA;
        j->Bd = Bd; j->dtype_in = dtype_in;
        j->alpha = alpha; j->beta = beta;
        j->Cin = Cin; j->ldcin = ldcin; j->dtype_cin = dtype_cin;
        j->biasd = biasd;
        j->rows = rows; j->nrows = nrows;
        j->cols = cols; j->ncols = ncols;
        j->out = out; j->ldout = ldout;
        j->r_begin = nrows * t / nthreads;
        j->r_end = nrows * (t + 1) / nthreads;
        if (pthread_create(&th[t], NULL, worker, j) != 0) { rc = -1; break; }
        ++started;
    }
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    free(th);
    free(jobs);
    free(Bd);
    free(biasd);
    free(all_rows);
    return rc;
}

/* Decode n stored elements of `dtype` to f64 (used by the tolerance check and the pins). */
int oracle_decode_array(const void* src, int dtype, int64_t n, double* dst) {
    if (n < 0 || (n > 0 && (!src || !dst))) return -1;
    for (int64_t i = 0; i < n; ++i) dst[i] = load_elem(src, i, dtype);
    return 0;
}

/* ==========================================================================
 * Q4_0-quantised weights.
 *
 * Source: "02 . 8m/8m(2) -- Tiled wmma f16 prefill GEMM (LANDED)", section 3.2
 * "Key code" (the Q4_0 dequantisation into an f16 scratch) and section 2.3 (the
 * weights are dequantised to f16, then one f16 tensor-core GEMM with f32
 * accumulation consumes them).  The block format as that page states it:
 *   - a row of the weight matrix (one output column n of C) holds K weights along
 *     K, in K/32 consecutive blocks of 18 bytes;
 *   - a block is a binary16 scale d (2 bytes, little-endian) followed by 16 bytes
 *     q[0..15];
 *   - weight i (0 <= i < 16) of the block is the low nibble of q[i], weight 16+i
 *     the high nibble of q[i];
 *   - its value is d * (nibble - 8), formed in f32 and converted to f16 with
 *     round-to-nearest-even.  The f32 product is exact (11 + 4 significand bits),
 *     so the stored f16 is the exact product rounded once to binary16.
 * The GEMM then reads those f16 values: C = alpha * A * W^T + beta * C_in + bias
 * with W the N x K dequantised matrix, i.e. B stored N x K (layout COL).
 * ========================================================================== */

/* Round-to-nearest-even of a non-negative value y that is exactly an integer plus
 * a fraction representable in f64. */
static double rne(double y) {
    const double f = floor(y);
    const double r = y - f;
    if (r > 0.5) return f + 1.0;
    if (r < 0.5) return f;
    return fmod(f, 2.0) == 0.0 ? f : f + 1.0;
}

/* f64 -> IEEE-754 binary16, round to nearest, ties to even, overflow to infinity
 * (written from the format definition: 1 sign, 5 exponent bits with bias 15, 10
 * fraction bits; subnormals are multiples of 2^-24). */
uint16_t oracle_f64_to_f16(double x) {
    if (isnan(x)) return 0x7e00u;
    const uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (isinf(a)) return sign | 0x7c00u;
    if (a == 0.0) return sign;
    int E;
    frexp(a, &E);                       /* a = m * 2^E, m in [0.5, 1): floor(log2 a) = E - 1 */
    int e = E - 1;
    if (e < -14) {                      /* subnormal range: units of 2^-24 */
        const double n = rne(ldexp(a, 24));
        return sign | (uint16_t)n;      /* n == 1024 is exactly the smallest normal's bits */
    }
    double n = rne(ldexp(a, 10 - e));   /* 1024 <= n <= 2048 */
    if (n == 2048.0) { n = 1024.0; ++e; }
    if (e > 15) return sign | 0x7c00u;
    return sign | (uint16_t)(((e + 15) << 10) | ((int)n - 1024));
}

/* Dequantise N rows of K weights (K a multiple of 32) from Q4_0 blocks at row pitch
 * ldbq bytes into binary16 bits, row n at out + n * ldo. */
int oracle_q4_0_to_f16(const uint8_t* bq, int64_t ldbq, int64_t N, int64_t K, uint16_t* out, int64_t ldo) {
    if (N < 0 || K < 0 || K % 32 != 0 || ldbq < K / 32 * 18 || ldo < K) return -1;
    if (N > 0 && K > 0 && (!bq || !out)) return -1;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t b = 0; b < K / 32; ++b) {
            const uint8_t* blk = bq + n * ldbq + b * 18;
            const double d = oracle_f16_to_f64((uint16_t)(blk[0] | (blk[1] << 8)));
            for (int i = 0; i < 16; ++i) {
                const int lo = blk[2 + i] & 0x0f, hi = blk[2 + i] >> 4;
                out[n * ldo + b * 32 + i] = oracle_f64_to_f16(d * (double)(lo - 8));
                out[n * ldo + b * 32 + 16 + i] = oracle_f64_to_f16(d * (double)(hi - 8));
            }
        }
    }
    return 0;
}
