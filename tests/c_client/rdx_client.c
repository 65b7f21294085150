/* A plain C11 client of librdx.so: device memory from the CUDA runtime, no
 * C++ and no PyTorch.  Calls every entry point of rdx.h at least once and
 * checks the results against closed forms and host sums (inputs are small
 * integers, so every float sum is exact; the sums of squares pass 2^24 and
 * are compared within 1e-6 relative). */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "rdx.h"

#define CHECK_CUDA(call)                                                         \
    do {                                                                         \
        cudaError_t e_ = (call);                                                 \
        if (e_ != cudaSuccess) {                                                 \
            fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));          \
            return 2;                                                            \
        }                                                                        \
    } while (0)

#define CHECK_RDX(call)                                                          \
    do {                                                                         \
        rdx_status s_ = (call);                                                  \
        if (s_ != RDX_OK) {                                                      \
            fprintf(stderr, "%s: %s %s\n", #call, rdx_status_string(s_),         \
                    rdx_last_cuda_error());                                      \
            return 3;                                                            \
        }                                                                        \
    } while (0)

int main(void) {
    const int64_t n = ((int64_t)1 << 22) + 3; /* 4 Mi + 3 elements */
    const int64_t rows = 1000, cols = 4099;   /* rows*cols < n */
    float* hf = (float*)malloc((size_t)n * sizeof(float));
    int32_t* hi = (int32_t*)malloc((size_t)n * sizeof(int32_t));
    if (!hf || !hi) return 4;
    for (int64_t i = 0; i < n; ++i) {
        hf[i] = (float)(i % 7);               /* 0..6 */
        hi[i] = (int32_t)((i % 2001) - 1000); /* -1000..1000 */
    }
    /* closed forms: n = 7q + r gives 21q + r(r-1)/2; the int series repeats every 2001 */
    const int64_t q = n / 7, r = n % 7;
    const double sum_f = 21.0 * (double)q + (double)(r * (r - 1) / 2);
    int64_t sum_i = 0;
    for (int64_t i = (n / 2001) * 2001; i < n; ++i) sum_i += (i % 2001) - 1000; /* whole periods sum to 0 */

    /* the same values as bfloat16 bit patterns (small integers: exact) */
    rdx_bf16* hb = (rdx_bf16*)malloc((size_t)n * sizeof(rdx_bf16));
    if (!hb) return 4;
    for (int64_t i = 0; i < n; ++i) {
        uint32_t u;
        memcpy(&u, &hf[i], sizeof u);
        hb[i] = (rdx_bf16)(u >> 16);
    }
    const int64_t rows3 = n / 3;                        /* narrow rows: 3 columns */
    const int64_t nparts = rdx_ladder_num_partials(5, n);

    float *df, *dout, *drows, *dmax, *drows3, *dparts, *dl5, *dbsum;
    int32_t *di, *dimax;
    int64_t* dsum_i;
    rdx_bf16* db;
    void* ws;
    cudaStream_t s;
    CHECK_CUDA(cudaStreamCreate(&s));
    CHECK_CUDA(cudaMalloc((void**)&df, (size_t)n * sizeof(float)));
    CHECK_CUDA(cudaMalloc((void**)&di, (size_t)n * sizeof(int32_t)));
    CHECK_CUDA(cudaMalloc((void**)&dout, 2 * sizeof(float)));
    CHECK_CUDA(cudaMalloc((void**)&dmax, sizeof(float)));
    CHECK_CUDA(cudaMalloc((void**)&dimax, sizeof(int32_t)));
    CHECK_CUDA(cudaMalloc((void**)&dsum_i, sizeof(int64_t)));
    CHECK_CUDA(cudaMalloc((void**)&drows, (size_t)rows * sizeof(float)));
    CHECK_CUDA(cudaMalloc((void**)&drows3, (size_t)rows3 * sizeof(float)));
    CHECK_CUDA(cudaMalloc((void**)&dparts, (size_t)nparts * sizeof(float)));
    CHECK_CUDA(cudaMalloc((void**)&dl5, sizeof(float)));
    CHECK_CUDA(cudaMalloc((void**)&dbsum, sizeof(float)));
    CHECK_CUDA(cudaMalloc((void**)&db, (size_t)n * sizeof(rdx_bf16)));
    CHECK_CUDA(cudaMemcpy(db, hb, (size_t)n * sizeof(rdx_bf16), cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMalloc(&ws, rdx_workspace_bytes()));
    CHECK_CUDA(cudaMemset(ws, 0, rdx_workspace_bytes()));
    CHECK_CUDA(cudaMemcpy(df, hf, (size_t)n * sizeof(float), cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(di, hi, (size_t)n * sizeof(int32_t), cudaMemcpyHostToDevice));

    CHECK_RDX(rdx_sum_f32(df, n, dout, s));
    CHECK_RDX(rdx_sum_i32_i64(di, n, dsum_i, s));
    CHECK_RDX(rdx_max_f32(df, n, dmax, s));
    CHECK_RDX(rdx_max_i32(di, n, dimax, s));
    CHECK_RDX(rdx_rowsum_f32(df, rows, cols, drows, s));
    CHECK_RDX(rdx_rowsum_f32(df, rows3, 3, drows3, s));
    CHECK_RDX(rdx_ladder_sum_f32(5, df, n, dparts, dl5, s));
    CHECK_RDX(rdx_sum_bf16_f32acc(db, n, dbsum, s));
    float got_f = 0.f, got_max = 0.f, pair[2] = {0.f, 0.f};
    int32_t got_imax = 0;
    int64_t got_i = 0;
    float got_l5 = 0.f, got_b = 0.f;
    float* got_rows = (float*)malloc((size_t)rows * sizeof(float));
    float* got_rows3 = (float*)malloc((size_t)rows3 * sizeof(float));
    if (!got_rows || !got_rows3) return 4;
    CHECK_CUDA(cudaMemcpyAsync(&got_f, dout, sizeof(float), cudaMemcpyDeviceToHost, s));
    CHECK_CUDA(cudaMemcpyAsync(&got_i, dsum_i, sizeof(int64_t), cudaMemcpyDeviceToHost, s));
    CHECK_CUDA(cudaMemcpyAsync(&got_max, dmax, sizeof(float), cudaMemcpyDeviceToHost, s));
    CHECK_CUDA(cudaMemcpyAsync(&got_imax, dimax, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
    CHECK_CUDA(cudaMemcpyAsync(got_rows, drows, (size_t)rows * sizeof(float), cudaMemcpyDeviceToHost, s));
    CHECK_CUDA(cudaMemcpyAsync(got_rows3, drows3, (size_t)rows3 * sizeof(float), cudaMemcpyDeviceToHost, s));
    CHECK_CUDA(cudaMemcpyAsync(&got_l5, dl5, sizeof(float), cudaMemcpyDeviceToHost, s));
    CHECK_CUDA(cudaMemcpyAsync(&got_b, dbsum, sizeof(float), cudaMemcpyDeviceToHost, s));
    CHECK_RDX(rdx_reduce_ws(RDX_OP_SUM_SUMSQ_F32, df, n, dout, ws, rdx_workspace_bytes(), s));
    CHECK_CUDA(cudaMemcpyAsync(pair, dout, 2 * sizeof(float), cudaMemcpyDeviceToHost, s));
    /* the same sums split over 3 ranks, each chunk on this GPU, then the rank-order combine */
    float *dpf, *dcf;
    int64_t *dpi, *dci;
    CHECK_CUDA(cudaMalloc((void**)&dpf, 3 * sizeof(float)));
    CHECK_CUDA(cudaMalloc((void**)&dcf, sizeof(float)));
    CHECK_CUDA(cudaMalloc((void**)&dpi, 3 * sizeof(int64_t)));
    CHECK_CUDA(cudaMalloc((void**)&dci, sizeof(int64_t)));
    for (int rank = 0; rank < 3; ++rank) {
        int64_t lo = -1, hi = -1;
        CHECK_RDX(rdx_shard_range(n, 3, rank, 4, &lo, &hi));
        CHECK_RDX(rdx_sum_f32(df + lo, hi - lo, dpf + rank, s));
        CHECK_RDX(rdx_sum_i32_i64(di + lo, hi - lo, dpi + rank, s));
    }
    CHECK_RDX(rdx_combine_f32(dpf, 3, dcf, s));
    CHECK_RDX(rdx_combine_i64(dpi, 3, dci, s));
    float got_split_f = 0.f;
    int64_t got_split_i = 0;
    CHECK_CUDA(cudaMemcpyAsync(&got_split_f, dcf, sizeof(float), cudaMemcpyDeviceToHost, s));
    CHECK_CUDA(cudaMemcpyAsync(&got_split_i, dci, sizeof(int64_t), cudaMemcpyDeviceToHost, s));
    CHECK_CUDA(cudaStreamSynchronize(s));

    int bad = 0;
    if ((double)got_f != sum_f) { fprintf(stderr, "sum_f32 %.1f != %.1f\n", got_f, sum_f); bad = 1; }
    if (got_i != sum_i) { fprintf(stderr, "sum_i32 %lld != %lld\n", (long long)got_i, (long long)sum_i); bad = 1; }
    if (got_max != 6.f || got_imax != 1000) { fprintf(stderr, "max %g %d\n", got_max, got_imax); bad = 1; }
    if ((double)pair[0] != sum_f) { fprintf(stderr, "ws pair sum %.1f\n", pair[0]); bad = 1; }
    if ((double)got_l5 != sum_f) { fprintf(stderr, "ladder v5 sum %.1f != %.1f\n", got_l5, sum_f); bad = 1; }
    if ((double)got_b != sum_f) { fprintf(stderr, "bf16 sum %.1f != %.1f\n", got_b, sum_f); bad = 1; }
    for (int64_t row = 0; row < rows3 && !bad; ++row) {
        const double e = (double)hf[3 * row] + (double)hf[3 * row + 1] + (double)hf[3 * row + 2];
        if ((double)got_rows3[row] != e) { fprintf(stderr, "3-column row %lld\n", (long long)row); bad = 1; }
    }
    for (int64_t row = 0; row < rows && !bad; ++row) {
        double e = 0.0;
        for (int64_t j = 0; j < cols; ++j) e += (double)hf[row * cols + j];
        if ((double)got_rows[row] != e) { fprintf(stderr, "row %lld: %.1f != %.1f\n", (long long)row, got_rows[row], e); bad = 1; }
    }
    if ((double)got_split_f != sum_f) { fprintf(stderr, "split sum %.1f != %.1f\n", got_split_f, sum_f); bad = 1; }
    if (got_split_i != sum_i) { fprintf(stderr, "split int sum %lld\n", (long long)got_split_i); bad = 1; }
    if (rdx_reduce_kernels(RDX_OP_SUM_F32, n) != 1 || rdx_reduce_kernels(RDX_OP_SUM_F32, (int64_t)1 << 28) != 2) {
        fprintf(stderr, "kernel counts\n");
        bad = 1;
    }

    /* every other compute entry point once: sums of squares, the one-pass
     * pairs, strided rows, a ladder version's partials, the pair combine, the
     * static-scratch sum, the bank probe and the checked-build counter */
    const double sumsq = 91.0 * (double)q + (double)((r - 1) * r * (2 * r - 1) / 6); /* 0^2 + ... + 6^2 = 91 */
    const int64_t cols_s = 4000, ld = 4099;  /* rows * ld < n */
    const int64_t nl1 = rdx_ladder_num_partials(1, n);
    float *dsq, *dsqb, *dp2, *dp2b, *dstr, *dl1, *dpp, *dcp, *dna;
    int64_t* dcycles;
    uint32_t* dsink;
    CHECK_CUDA(cudaMalloc((void**)&dsq, sizeof(float)));
    CHECK_CUDA(cudaMalloc((void**)&dsqb, sizeof(float)));
    CHECK_CUDA(cudaMalloc((void**)&dp2, 2 * sizeof(float)));
    CHECK_CUDA(cudaMalloc((void**)&dp2b, 2 * sizeof(float)));
    CHECK_CUDA(cudaMalloc((void**)&dstr, (size_t)rows * sizeof(float)));
    CHECK_CUDA(cudaMalloc((void**)&dl1, (size_t)nl1 * sizeof(float)));
    CHECK_CUDA(cudaMalloc((void**)&dpp, 3 * 2 * sizeof(float)));
    CHECK_CUDA(cudaMalloc((void**)&dcp, 2 * sizeof(float)));
    CHECK_CUDA(cudaMalloc((void**)&dna, sizeof(float)));
    CHECK_CUDA(cudaMalloc((void**)&dcycles, sizeof(int64_t)));
    CHECK_CUDA(cudaMalloc((void**)&dsink, 32 * sizeof(uint32_t)));
    CHECK_RDX(rdx_sumsq_f32(df, n, dsq, s));
    CHECK_RDX(rdx_sumsq_bf16_f32acc(db, n, dsqb, s));
    CHECK_RDX(rdx_sum_sumsq_f32(df, n, dp2, s));
    CHECK_RDX(rdx_sum_sumsq_bf16_f32acc(db, n, dp2b, s));
    CHECK_RDX(rdx_rowsum_strided_f32(df, rows, cols_s, ld, dstr, s));
    CHECK_RDX(rdx_ladder_partials_f32(1, df, n, dl1, s));
    for (int rank = 0; rank < 3; ++rank) {
        int64_t lo = -1, hi = -1;
        CHECK_RDX(rdx_shard_range(n, 3, rank, 4, &lo, &hi));
        CHECK_RDX(rdx_sum_sumsq_f32(df + lo, hi - lo, dpp + 2 * rank, s));
    }
    CHECK_RDX(rdx_combine_f32x2(dpp, 3, dcp, s));
    CHECK_RDX(rdx_sum_f32_noalloc(df, n, dna, s));
    CHECK_RDX(rdx_bank_probe(0, 16, dcycles, dsink, s));
    float got_sq = 0.f, got_sqb = 0.f, p2[2] = {0.f, 0.f}, p2b[2] = {0.f, 0.f}, cp[2] = {0.f, 0.f}, got_na = 0.f;
    int64_t cycles = 0;
    float* got_str = (float*)malloc((size_t)rows * sizeof(float));
    float* got_l1 = (float*)malloc((size_t)nl1 * sizeof(float));
    if (!got_str || !got_l1) return 4;
    CHECK_CUDA(cudaMemcpyAsync(&got_sq, dsq, sizeof(float), cudaMemcpyDeviceToHost, s));
    CHECK_CUDA(cudaMemcpyAsync(&got_sqb, dsqb, sizeof(float), cudaMemcpyDeviceToHost, s));
    CHECK_CUDA(cudaMemcpyAsync(p2, dp2, 2 * sizeof(float), cudaMemcpyDeviceToHost, s));
    CHECK_CUDA(cudaMemcpyAsync(p2b, dp2b, 2 * sizeof(float), cudaMemcpyDeviceToHost, s));
    CHECK_CUDA(cudaMemcpyAsync(got_str, dstr, (size_t)rows * sizeof(float), cudaMemcpyDeviceToHost, s));
    CHECK_CUDA(cudaMemcpyAsync(got_l1, dl1, (size_t)nl1 * sizeof(float), cudaMemcpyDeviceToHost, s));
    CHECK_CUDA(cudaMemcpyAsync(cp, dcp, 2 * sizeof(float), cudaMemcpyDeviceToHost, s));
    CHECK_CUDA(cudaMemcpyAsync(&got_na, dna, sizeof(float), cudaMemcpyDeviceToHost, s));
    CHECK_CUDA(cudaMemcpyAsync(&cycles, dcycles, sizeof(int64_t), cudaMemcpyDeviceToHost, s));
    CHECK_CUDA(cudaStreamSynchronize(s));
    /* the sums of squares pass 2^24, so float32 partial sums round: compare within 1e-6 relative */
    const double sq_tol = 1e-6 * sumsq;
    if (got_sq - sumsq > sq_tol || sumsq - got_sq > sq_tol) { fprintf(stderr, "sumsq_f32 %.1f\n", got_sq); bad = 1; }
    if (got_sqb - sumsq > sq_tol || sumsq - got_sqb > sq_tol) { fprintf(stderr, "sumsq_bf16 %.1f\n", got_sqb); bad = 1; }
    if ((double)p2[0] != sum_f || p2[1] - sumsq > sq_tol || sumsq - p2[1] > sq_tol) { fprintf(stderr, "pair f32\n"); bad = 1; }
    if ((double)p2b[0] != sum_f || p2b[1] - sumsq > sq_tol || sumsq - p2b[1] > sq_tol) { fprintf(stderr, "pair bf16\n"); bad = 1; }
    if ((double)cp[0] != sum_f || cp[1] - sumsq > sq_tol || sumsq - cp[1] > sq_tol) { fprintf(stderr, "split pair\n"); bad = 1; }
    for (int64_t row = 0; row < rows && !bad; ++row) {
        double e = 0.0;
        for (int64_t j = 0; j < cols_s; ++j) e += (double)hf[row * ld + j];
        if ((double)got_str[row] != e) { fprintf(stderr, "strided row %lld\n", (long long)row); bad = 1; }
    }
    for (int64_t b = 0; b < nl1 && !bad; ++b) {
        double e = 0.0;
        for (int64_t i = b * 256; i < n && i < (b + 1) * 256; ++i) e += (double)hf[i];
        if ((double)got_l1[b] != e) { fprintf(stderr, "ladder v1 partial %lld\n", (long long)b); bad = 1; }
    }
    if (memcmp(&got_na, &got_f, sizeof(float)) != 0) { fprintf(stderr, "static-scratch sum %.1f\n", got_na); bad = 1; }
    if (cycles <= 0 || rdx_bank_probe_loads_per_iter() < 1) { fprintf(stderr, "bank probe\n"); bad = 1; }
    if (rdx_rowsum_kernels(rows, cols) < 1 || rdx_combine_max_parts() != 4096) { fprintf(stderr, "queries\n"); bad = 1; }
    uint64_t violations = 1;
    CHECK_RDX(rdx_debug_violations(&violations, 0));
    if (rdx_debug_build() != 0 || violations != 0) { fprintf(stderr, "normal build\n"); bad = 1; }
    /* the bounded staging wait: no call so far gave up; the test hook's tile
     * cannot complete, so its wait gives up after a second and is counted */
    uint64_t timeouts = 1;
    float* dprobe;
    CHECK_CUDA(cudaMalloc((void**)&dprobe, 100 * sizeof(float)));
    CHECK_RDX(rdx_wait_timeouts(&timeouts, 1));
    if (timeouts != 0) { fprintf(stderr, "timeouts before the probe\n"); bad = 1; }
    CHECK_RDX(rdx_debug_stage_timeout(df, 100, 16, dprobe, s));
    CHECK_RDX(rdx_wait_timeouts(&timeouts, 1));
    if (timeouts != 1) { fprintf(stderr, "probe timeouts %llu\n", (unsigned long long)timeouts); bad = 1; }
    /* the stream made calls, so it holds a workspace; releasing it twice frees it once */
    if (rdx_release_stream(s) != 1 || rdx_release_stream(s) != 0) { fprintf(stderr, "release stream\n"); bad = 1; }

    /* argument errors come back as statuses, nothing is enqueued */
    if (rdx_sum_f32(df, -1, dout, s) != RDX_ERR_INVALID_ARG) bad = 1;
    if (rdx_sum_f32(df, n, (float*)(df + 8), s) != RDX_ERR_INVALID_ARG) bad = 1;
    rdx_shutdown();
    printf(bad ? "c client FAILED\n" : "c client ok\n");
    return bad;
}
