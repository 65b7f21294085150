/*
 * oracle.c -- the CPU oracle for the sum reductions.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, the smoke check
 * and the bench's CPU-baseline leg may load or call this file.  It shares no
 * code, header or constant with the CUDA library; neither includes the other.
 *
 * Every routine is the plain definition of its result written out as one
 * loop over the input in index order:
 *
 *   - the page "03_shared_memory_sync_reduction.py", demo 3 (parallel
 *     reduction), takes as the expected result of every kernel version the
 *     float64 sum of the float32 input, and checks each version against it;
 *   - floating-point sums here are float64 with Kahan compensation
 *     (y = x - c; t = s + y; c = (t - s) - y; s = t), so the oracle is far
 *     more accurate than any float32 GPU result it is compared with;
 *   - integer sums are int64 accumulation modulo 2^64, exact for any n < 2^32;
 *   - the row-segmented sum is the same loop run once per row.  On the page,
 *     versions 1-3 write one partial per block of B consecutive inputs and
 *     versions 4-5 one per 2B, so a block's output is a segment sum; a row
 *     of a row-major matrix is such a segment.
 *
 * Non-finite terms (Inf/NaN) are set aside from the compensated loop and
 * added plainly at the end, so infinities and NaNs propagate as in a plain
 * IEEE sum (the compensation term would otherwise turn a lone +Inf into NaN).
 *
 * Build: gcc -O2 -fPIC -shared -ffp-contract=off -fno-fast-math
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

typedef struct {
    double s;          /* running sum of the finite terms            */
    double c;          /* Kahan compensation: the lost low-order part */
    double nonfinite;  /* plain sum of the Inf/NaN terms             */
} kahan_acc;

static void kahan_init(kahan_acc* k) {
    k->s = 0.0;
    k->c = 0.0;
    k->nonfinite = 0.0;
}

static void kahan_add(kahan_acc* k, double v) {
    if (!isfinite(v)) {
        k->nonfinite += v;
        return;
    }
    double y = v - k->c;
    double t = k->s + y;
    k->c = (t - k->s) - y;
    k->s = t;
}

static double kahan_result(const kahan_acc* k) {
    if (!(k->nonfinite == 0.0)) return k->s + k->nonfinite; /* also taken for NaN */
    return k->s;
}

/* bfloat16 is the upper 16 bits of an IEEE binary32; widening is exact. */
static double bf16_bits_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ---- float32 input ---------------------------------------------------- */

double oracle_sum_f32(const float* x, int64_t n) {
    kahan_acc k;
    kahan_init(&k);
    for (int64_t i = 0; i < n; ++i) kahan_add(&k, (double)x[i]);
    return kahan_result(&k);
}

/* x_i^2 of a float32 value is exact in float64 (24-bit significand squared). */
double oracle_sumsq_f32(const float* x, int64_t n) {
    kahan_acc k;
    kahan_init(&k);
    for (int64_t i = 0; i < n; ++i) {
        double v = (double)x[i];
        kahan_add(&k, v * v);
    }
    return kahan_result(&k);
}

/* sum of |x_i|: the scale that the float tolerances are stated against. */
double oracle_abssum_f32(const float* x, int64_t n) {
    kahan_acc k;
    kahan_init(&k);
    for (int64_t i = 0; i < n; ++i) kahan_add(&k, fabs((double)x[i]));
    return kahan_result(&k);
}

/* ---- bfloat16 input (raw 16-bit patterns) ------------------------------ */

double oracle_sum_bf16(const uint16_t* x, int64_t n) {
    kahan_acc k;
    kahan_init(&k);
    for (int64_t i = 0; i < n; ++i) kahan_add(&k, bf16_bits_to_double(x[i]));
    return kahan_result(&k);
}

double oracle_sumsq_bf16(const uint16_t* x, int64_t n) {
    kahan_acc k;
    kahan_init(&k);
    for (int64_t i = 0; i < n; ++i) {
        double v = bf16_bits_to_double(x[i]);
        kahan_add(&k, v * v);
    }
    return kahan_result(&k);
}

double oracle_abssum_bf16(const uint16_t* x, int64_t n) {
    kahan_acc k;
    kahan_init(&k);
    for (int64_t i = 0; i < n; ++i) kahan_add(&k, fabs(bf16_bits_to_double(x[i])));
    return kahan_result(&k);
}

/* ---- int32 input, int64 result ----------------------------------------- */

/* The int64 sum of int32 values, defined as addition modulo 2^64 (the
 * two's-complement int64 the result is returned in).  Exact, and equal to the
 * mathematical sum, while |sum| < 2^63, which any n < 2^32 guarantees
 * (|x_i| <= 2^31).  The loop adds in uint64_t, whose wrap-around C defines,
 * so a sum past 2^63 wraps instead of being signed overflow. */
static int64_t from_twos_complement(uint64_t u) {
    if (u <= (uint64_t)INT64_MAX) return (int64_t)u;
    return -(int64_t)(~u) - 1; /* u - 2^64, without overflow */
}

int64_t oracle_sum_i32(const int32_t* x, int64_t n) {
    uint64_t s = 0;
    for (int64_t i = 0; i < n; ++i) s += (uint64_t)(int64_t)x[i];
    return from_twos_complement(s);
}

/* The sum of int64 values modulo 2^64: the combine of the int64 partials of
 * a sum split into chunks (each chunk's int32 sum is one partial; the whole
 * sum is the sum of the partials, integer addition being associative). */
int64_t oracle_sum_i64(const int64_t* x, int64_t n) {
    uint64_t s = 0;
    for (int64_t i = 0; i < n; ++i) s += (uint64_t)x[i];
    return from_twos_complement(s);
}

/* ---- row-segmented float32 sum (row-major, contiguous) ----------------- */

void oracle_rowsum_f32(const float* x, int64_t rows, int64_t cols, double* out) {
    for (int64_t r = 0; r < rows; ++r) {
        const float* row = x + r * cols;
        kahan_acc k;
        kahan_init(&k);
        for (int64_t j = 0; j < cols; ++j) kahan_add(&k, (double)row[j]);
        out[r] = kahan_result(&k);
    }
}

void oracle_rowabssum_f32(const float* x, int64_t rows, int64_t cols, double* out) {
    for (int64_t r = 0; r < rows; ++r) {
        const float* row = x + r * cols;
        kahan_acc k;
        kahan_init(&k);
        for (int64_t j = 0; j < cols; ++j) kahan_add(&k, fabs((double)row[j]));
        out[r] = kahan_result(&k);
    }
}

/* ---- maximum ------------------------------------------------------------ */

/* The page "lecture02/simt.py" models atomic_max as: old = A[i]; if v > old
 * then A[i] = v.  Folding every input through that rule from -Inf gives the
 * maximum; a NaN is never greater than anything, so it never replaces the
 * running value (NaNs are ignored; all-NaN or empty input gives -Inf). */
float oracle_max_f32(const float* x, int64_t n) {
    float m = -INFINITY;
    for (int64_t i = 0; i < n; ++i)
        if (x[i] > m) m = x[i];
    return m;
}

int32_t oracle_max_i32(const int32_t* x, int64_t n) {
    int32_t m = INT32_MIN;
    for (int64_t i = 0; i < n; ++i)
        if (x[i] > m) m = x[i];
    return m;
}
