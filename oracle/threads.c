/*
 * threads.c -- the oracle's loops spread over several host threads: the
 * multi-core CPU baseline.
 *
 * TEST AND BENCHMARK INFRASTRUCTURE, NOT PRODUCT CODE.  It is linked with
 * oracle.c into its own library and calls the single-thread definitions
 * there unchanged: the input is cut into one contiguous chunk per thread,
 * each thread runs the oracle's float64 Kahan (or int64) loop over its chunk,
 * and the chunk results are added in chunk order on the calling thread.
 *
 * The result is the same for any run with the same thread count.  For the
 * integer sum it equals the single-thread oracle exactly.  For the float sums
 * the chunk results are themselves compensated float64 sums, and adding at
 * most a few hundred of them in plain float64 adds an error of a few hundred
 * units in the last place of a double: far below any float32 tolerance, but
 * not bit-identical to the one-loop oracle, which stays the parity reference.
 *
 * Row sums split the rows, not the columns: every output row is computed by
 * exactly the single-thread loop, so they match the oracle bit for bit.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

double oracle_sum_f32(const float* x, int64_t n);
double oracle_sumsq_f32(const float* x, int64_t n);
double oracle_sum_bf16(const uint16_t* x, int64_t n);
double oracle_sumsq_bf16(const uint16_t* x, int64_t n);
int64_t oracle_sum_i32(const int32_t* x, int64_t n);
void oracle_rowsum_f32(const float* x, int64_t rows, int64_t cols, double* out);

/* Operation codes of oracle_threaded_reduce. */
enum { T_SUM_F32 = 0, T_SUMSQ_F32 = 1, T_SUM_BF16 = 2, T_SUMSQ_BF16 = 3, T_SUM_I32 = 4 };

enum { MAX_THREADS = 512 };

typedef struct {
    int op;
    const void* x;
    int64_t lo, hi;   /* elements [lo, hi) of the input, or rows for row sums */
    int64_t cols;     /* row sums only */
    double* rows_out; /* row sums only */
    double d;         /* float result of this chunk */
    int64_t i;        /* integer result of this chunk */
} chunk;

static void* run_chunk(void* arg) {
    chunk* c = (chunk*)arg;
    const int64_t len = c->hi - c->lo;
    switch (c->op) {
        case T_SUM_F32: c->d = oracle_sum_f32((const float*)c->x + c->lo, len); break;
        case T_SUMSQ_F32: c->d = oracle_sumsq_f32((const float*)c->x + c->lo, len); break;
        case T_SUM_BF16: c->d = oracle_sum_bf16((const uint16_t*)c->x + c->lo, len); break;
        case T_SUMSQ_BF16: c->d = oracle_sumsq_bf16((const uint16_t*)c->x + c->lo, len); break;
        case T_SUM_I32: c->i = oracle_sum_i32((const int32_t*)c->x + c->lo, len); break;
        default: /* row sums: rows [lo, hi) */
            oracle_rowsum_f32((const float*)c->x + c->lo * c->cols, len, c->cols, c->rows_out + c->lo);
            break;
    }
    return NULL;
}

/* Runs the chunks, the first on the calling thread; returns 0 on success,
 * -1 when a thread could not be started (the chunks already started are
 * joined first). */
static int run_all(chunk* cs, int k) {
    pthread_t tid[MAX_THREADS];
    int started = 0, rc = 0;
    for (int t = 1; t < k; ++t) {
        if (pthread_create(&tid[t], NULL, run_chunk, &cs[t]) != 0) {
            rc = -1;
            break;
        }
        started = t;
    }
    if (rc == 0) run_chunk(&cs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(tid[t], NULL);
    return rc;
}

/* Splits [0, n) into k contiguous chunks whose sizes differ by at most one. */
static int split(int op, const void* x, int64_t n, int threads, int64_t cols, double* rows_out,
                 chunk* cs) {
    int k = threads < 1 ? 1 : (threads > MAX_THREADS ? MAX_THREADS : threads);
    if (n < k) k = n > 0 ? (int)n : 1;
    const int64_t base = n / k, extra = n % k;
    int64_t lo = 0;
    for (int t = 0; t < k; ++t) {
        const int64_t len = base + (t < extra ? 1 : 0);
        cs[t] = (chunk){op, x, lo, lo + len, cols, rows_out, 0.0, 0};
        lo += len;
    }
    return k;
}

/* One scalar reduction (op = 0..4 above) of n elements on `threads` threads.
 * Float results go to *out_d, the int32 sum to *out_i.  Returns 0, or -1 for
 * an unknown op or a thread that could not be started. */
int oracle_threaded_reduce(int op, const void* x, int64_t n, int threads, double* out_d,
                           int64_t* out_i) {
    if (op < T_SUM_F32 || op > T_SUM_I32 || n < 0) return -1;
    chunk cs[MAX_THREADS];
    const int k = split(op, x, n, threads, 0, NULL, cs);
    if (run_all(cs, k) != 0) return -1;
    double d = 0.0;
    uint64_t i = 0; /* modulo 2^64, as the single-thread loop */
    for (int t = 0; t < k; ++t) {
        d += cs[t].d;
        i += (uint64_t)cs[t].i;
    }
    if (out_d) *out_d = d;
    if (out_i) *out_i = i <= (uint64_t)INT64_MAX ? (int64_t)i : -(int64_t)(~i) - 1;
    return 0;
}

/* Row sums of a row-major rows x cols float32 matrix on `threads` threads,
 * each thread taking a contiguous block of rows.  Returns 0 or -1. */
int oracle_threaded_rowsum_f32(const float* x, int64_t rows, int64_t cols, int threads, double* out) {
    if (rows < 0 || cols < 0) return -1;
    chunk cs[MAX_THREADS];
    const int k = split(-1, x, rows, threads, cols, out, cs);
    return run_all(cs, k);
}
