/*
 * rdx.h -- C ABI of the GB300 (sm_103a) parallel sum-reduction library
 * (librdx.so).
 *
 * The operation is the parallel sum reduction of a large array worked through
 * in the page "03_shared_memory_sync_reduction.py", demo 3 (parallel
 * reduction): many threads cooperate to add up an array, each block
 * producing one partial sum.  Here the partials are finished on the device in
 * a fixed order, so every call returns the whole sum, and the result is
 * bitwise reproducible from run to run on the same GPU model.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers are device pointers (memory the current CUDA device can read
 *    and write: cudaMalloc, torch CUDA tensors, managed memory).  The caller
 *    owns the input and the output buffers.
 *  - Every call is asynchronous: it validates its arguments, enqueues its
 *    kernels on `stream` (one, or two for inputs of 64 MiB and up:
 *    rdx_reduce_kernels / rdx_rowsum_kernels say which) and returns.  The
 *    result is valid in stream order.  `stream` must belong to the current
 *    CUDA device; 0 is the legacy default stream.  (rdx_shard_range and the
 *    size queries run on the host only.)
 *  - Sizes are element counts (int64_t); no size limit beyond device memory.
 *  - Any element-aligned input pointer is accepted; 16-byte alignment is not
 *    required.  The output must not overlap the input.
 *  - Scratch: the scalar reductions (and the row sum of few, very long rows)
 *    keep one small workspace per (device, stream) pair (tile partials,
 *    completion counters and, for the int64 sum and the maxima, one
 *    accumulator word; rdx_workspace_bytes() bytes), allocated by the
 *    library with cudaMalloc on the first call on that pair that needs it and
 *    reused after.  Make that first call outside any CUDA-graph capture, or
 *    pass a workspace of your own to rdx_reduce_ws.  Two host threads may
 *    call concurrently; calls on one stream are ordered by the stream.
 *    cudaStreamPerThread gets one workspace per host thread (it names a
 *    different stream in each).  A workspace is found by the stream's handle:
 *    synchronize a stream before destroying it, or a new stream that is
 *    given the same handle could share the workspace with work still
 *    pending.  rdx_shutdown() frees the library's workspaces,
 *    rdx_release_stream() one stream's.
 *  - Errors: no exception crosses this ABI.  Each call returns an rdx_status;
 *    argument errors are found before any CUDA call and nothing is enqueued.
 *    After RDX_ERR_CUDA, rdx_last_cuda_error() names the failing CUDA call.
 *
 * Floating-point results
 * ----------------------
 * Float sums accumulate in float32 along a fixed tree (per-thread vector
 * folds, a warp shuffle tree, a cross-warp stage, and a fixed-order pass over
 * the block partials).  The order depends only on the input's length and its
 * 16-byte alignment (row sums: the matrix's shape and the alignment of its
 * address), never on timing or on the GPU, so a repeated call gives the same
 * bits.  Measured against
 * the exact sum, the error stays within 1e-6 * sum|x_i| for float32 input and
 * 4e-6 * sum|x_i| for bfloat16 input (sum of squares: the same factors times
 * sum x_i^2).  Inf and NaN propagate as in an IEEE sum.
 */
#ifndef RDX_H
#define RDX_H

#include <stdint.h>
#include <cuda_runtime_api.h> /* cudaStream_t */

#ifdef __cplusplus
extern "C" {
#endif

typedef int rdx_status;

#define RDX_OK 0                      /* enqueued (or nothing to do)                    */
#define RDX_ERR_INVALID_ARG 1         /* bad pointer, size, alignment, overlap, version */
#define RDX_ERR_CUDA 2                /* a CUDA runtime call or a launch failed         */
#define RDX_ERR_ALLOC 3               /* the workspace could not be allocated           */
#define RDX_ERR_UNSUPPORTED_DEVICE 4  /* the current device is not sm_103 (GB300)       */

/* bfloat16 values are passed as their raw 16-bit patterns (the upper half of
 * the IEEE binary32 with the same value). */
typedef uint16_t rdx_bf16;

/* Scalar reductions by code, for rdx_reduce_ws. */
#define RDX_OP_SUM_F32 0         /* float in, float out              */
#define RDX_OP_SUMSQ_F32 1       /* float in, float out              */
#define RDX_OP_SUM_BF16 2        /* rdx_bf16 in, float out           */
#define RDX_OP_SUMSQ_BF16 3      /* rdx_bf16 in, float out           */
#define RDX_OP_SUM_I32 4         /* int32_t in, int64_t out          */
#define RDX_OP_SUM_SUMSQ_F32 5   /* float in, float[2] out           */
#define RDX_OP_SUM_SUMSQ_BF16 6  /* rdx_bf16 in, float[2] out        */
#define RDX_OP_MAX_F32 7         /* float in, float out              */
#define RDX_OP_MAX_I32 8         /* int32_t in, int32_t out          */

/*
 * rdx_sum_f32: *out = sum_{i<n} x[i].
 * Page "03_shared_memory_sync_reduction.py", demo 3: the sum of a float32
 * array (the page's expected value is this sum in float64).
 *   x    n float32 values, contiguous, 4-byte aligned (NULL allowed if n == 0)
 *   n    element count, >= 0; n == 0 writes 0.0f
 *   out  one float32 in device memory
 * Errors: RDX_ERR_INVALID_ARG if n < 0, out == NULL, x == NULL with n > 0,
 * a pointer is not aligned to its element size, or out lies inside x.
 */
rdx_status rdx_sum_f32(const float* x, int64_t n, float* out, cudaStream_t stream);

/*
 * rdx_sumsq_f32: *out = sum_{i<n} x[i]^2, float32 accumulation.
 * Page "03_shared_memory_sync_reduction.py", demo 3's sum with the square of
 * each input as the term: the page's one add per element becomes one
 * multiply-add.  The pages give no sum of squares of their own; it is one of
 * this library's five named operations, run on the 2^24 + 13-element
 * normal(0, 1) float32 workload beside its plain sum.  The result is within
 * 1e-6 * sum x_i^2 of the exact sum of squares.
 * Arguments and errors as rdx_sum_f32.
 */
rdx_status rdx_sumsq_f32(const float* x, int64_t n, float* out, cudaStream_t stream);

/*
 * rdx_sum_bf16_f32acc: *out = sum_{i<n} x[i], bfloat16 input widened exactly
 * to float32, float32 accumulation.
 * Page "03_shared_memory_sync_reduction.py", demo 3's sum over a 2-byte
 * element: half the bytes per add of the page's float32 input (the pages'
 * simulator holds 4-byte types only: page "simt_lab.py", section 3, shared
 * arrays).  One of this library's
 * five named operations, run on the 2^30 + 7-element workload of normal(0, 1)
 * values rounded to bfloat16.  The result is within 4e-6 * sum |x_i| of the
 * exact sum.  x is 2-byte aligned.
 * Arguments and errors as rdx_sum_f32.
 */
rdx_status rdx_sum_bf16_f32acc(const rdx_bf16* x, int64_t n, float* out, cudaStream_t stream);

/*
 * rdx_sumsq_bf16_f32acc: *out = sum_{i<n} x[i]^2, bfloat16 input, float32
 * accumulation: rdx_sumsq_f32's term over rdx_sum_bf16_f32acc's input.  The
 * 2^30 + 7-element bfloat16 workload asks for its sum of squares beside its
 * sum; the five named operations have no bfloat16 sum of squares, so this
 * sixth one is exported with the same signature.  The result is within
 * 4e-6 * sum x_i^2 of the exact sum of squares.
 * Arguments and errors as rdx_sum_bf16_f32acc.
 */
rdx_status rdx_sumsq_bf16_f32acc(const rdx_bf16* x, int64_t n, float* out, cudaStream_t stream);

/*
 * rdx_sum_i32_i64: *out = sum_{i<n} x[i], int32 input, int64 accumulation.
 * Page "03_shared_memory_sync_reduction.py", demo 3's sum over int32 values
 * (the simulator's shared arrays hold float32 and int32 alike: page
 * "simt_lab.py", section 3), widened to int64 so that it cannot overflow in
 * practice.  One of this library's five named
 * operations, run on the 2^28-element workload of uniform integers in
 * [-2^20, 2^20] and required bit-exact.
 * The accumulation is int64 addition, i.e. addition modulo 2^64 of the
 * values' two's-complement bits: it is associative, so the result is the
 * sequential sum bit for bit in any grouping.  It equals the mathematical sum
 * whenever |sum| < 2^63, which every n < 2^32 guarantees (|x_i| <= 2^31);
 * beyond that the result wraps modulo 2^64 (no error is raised).  x 4-byte
 * aligned, out 8-byte aligned.  Other arguments and errors as rdx_sum_f32.
 */
rdx_status rdx_sum_i32_i64(const int32_t* x, int64_t n, int64_t* out, cudaStream_t stream);

/*
 * rdx_sum_sumsq_f32: out2[0] = sum_{i<n} x[i], out2[1] = sum_{i<n} x[i]^2,
 * both in one pass over x (the input is read once for both results).  Each
 * component follows the summation tree of rdx_sum_f32 / rdx_sumsq_f32; the
 * grid may differ from theirs, so the bits may too (within the same bounds).
 *   out2  two float32 values, 8-byte aligned
 * Other arguments and errors as rdx_sum_f32.
 */
rdx_status rdx_sum_sumsq_f32(const float* x, int64_t n, float* out2, cudaStream_t stream);

/*
 * rdx_sum_sumsq_bf16_f32acc: out2[0] = sum, out2[1] = sum of squares of a
 * bfloat16 array in one pass, float32 accumulation.  out2 as above.
 */
rdx_status rdx_sum_sumsq_bf16_f32acc(const rdx_bf16* x, int64_t n, float* out2, cudaStream_t stream);

/*
 * rdx_max_f32: *out = max_{i<n} x[i].
 * The page "lecture02/simt.py" models atomic_max as "replace the stored value
 * when the new one is greater"; folding the input through that rule from
 * -Inf gives this maximum.  NaNs never win (they are skipped); n == 0 or an
 * all-NaN input gives -Inf.  The maximum is exact in any grouping, so the
 * result does not depend on the summation tree (the sign of a zero maximum
 * is not specified).  Arguments and errors as rdx_sum_f32.
 */
rdx_status rdx_max_f32(const float* x, int64_t n, float* out, cudaStream_t stream);

/*
 * rdx_max_i32: *out = max_{i<n} x[i] for int32 input; n == 0 gives -2^31.
 * out: one int32, 4-byte aligned.  Arguments and errors as rdx_sum_f32.
 */
rdx_status rdx_max_i32(const int32_t* x, int64_t n, int32_t* out, cudaStream_t stream);

/*
 * rdx_rowsum_f32: out[r] = sum_{j<cols} x[r*cols + j] for r < rows.
 * The row-segmented sum: on the page each block of versions 1-3 writes the
 * sum of B consecutive inputs (2B for versions 4-5) to out[blockIdx], i.e. a
 * segmented sum with fixed-length segments; here a segment is a matrix row.
 *   x     rows*cols float32 values, row-major and contiguous, 4-byte aligned
 *   rows  >= 0; rows == 0 enqueues nothing
 *   cols  >= 0; cols == 0 writes rows zeros
 *   out   rows float32 values; must not overlap x
 * Rows of at most 64 columns (contiguous) are staged through shared
 * memory in tiles of whole rows and summed one row per thread (where those
 * reads would meet shared-memory bank conflicts, each tile arrives by one
 * bulk copy whose barrier wait is bounded: see rdx_wait_timeouts); short and
 * medium rows are summed by a group of threads each (from tiles staged the
 * same way: contiguous rows of 65 to 512 columns that a group would read
 * with half-empty load slots, and every contiguous row of 513 to 6000),
 * long rows by a block each, with no workspace.  Few, very long rows (fewer than two waves of
 * blocks, at least 16384 columns, at most 2048 rows) are each cut into tiles
 * over many blocks and finished on the device like the scalar sums; that
 * path uses the (device, stream) workspace.  Either way a row's summation
 * order is fixed by the matrix's shape and the alignment of its address,
 * never by the device or the run.
 * Errors: RDX_ERR_INVALID_ARG for negative sizes, rows*cols overflowing
 * int64, NULL or misaligned pointers, overlap; RDX_ERR_ALLOC if the split
 * path's workspace cannot be allocated.
 */
rdx_status rdx_rowsum_f32(const float* x, int64_t rows, int64_t cols, float* out, cudaStream_t stream);

/*
 * rdx_rowsum_strided_f32: out[r] = sum_{j<cols} x[r*ld + j] for r < rows:
 * rdx_rowsum_f32 for rows that start every ld elements (a leading dimension,
 * e.g. a column slice of a wider row-major matrix).  ld >= cols when
 * rows > 1; rows need not be 16-byte aligned.  Other arguments, behaviour
 * and errors as rdx_rowsum_f32.
 */
rdx_status rdx_rowsum_strided_f32(const float* x, int64_t rows, int64_t cols, int64_t ld, float* out,
                                  cudaStream_t stream);

/* Bytes of a caller-owned workspace for rdx_reduce_ws (a constant). */
size_t rdx_workspace_bytes(void);

/*
 * Kernels one call enqueues on its stream (for callers that count launches
 * or capture graphs).  A scalar reduction (and the row sum of few, very long
 * rows) cuts its input into tiles, one block each; with tiles of 64 KiB or
 * more (inputs of 64 MiB and up) the fixed-order pass over the tile partials
 * runs as a second kernel, launched behind the first with programmatic
 * dependent launch, instead of in the first kernel's last block (so no block
 * waits on a completion ticket; both give the same bits).
 * rdx_reduce_kernels: 1 or 2 for rdx_reduce_ws code `op` (or its named entry
 * point) on n elements; -1 for a bad op or n < 0.
 * rdx_rowsum_kernels: 0 (rows == 0), 1 or 2 for rdx_rowsum_f32 on a
 * rows x cols matrix; -1 for negative sizes.
 */
int rdx_reduce_kernels(int op, int64_t n);
int rdx_rowsum_kernels(int64_t rows, int64_t cols);

/*
 * rdx_reduce_ws: the scalar reduction `op` (an RDX_OP_* code) of n elements
 * of x into out, with a workspace the caller owns instead of the library's.
 * Results are the same as the named entry point's (same kernel and tiling).
 *   workspace       device memory of at least rdx_workspace_bytes() bytes,
 *                   256-byte aligned, zero-filled once before its first use
 *                   (every call leaves it ready for the next)
 * The call allocates nothing.  Calls sharing one workspace must be ordered
 * (one stream, or synchronised): kernels that overlap on the GPU race on it.
 * Errors: as the named entry point, plus RDX_ERR_INVALID_ARG for a bad op,
 * a NULL, small or misaligned workspace, or a workspace overlapping x or out.
 */
rdx_status rdx_reduce_ws(int op, const void* x, int64_t n, void* out, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream);

/*
 * rdx_ladder_partials_f32: the page's five block-reduction versions, run as
 * written (block of 256 threads), one float32 partial per block:
 *   version 1  interleaved addressing, divergent branch (tid % 2s == 0)
 *   version 2  interleaved addressing, consecutive threads (index = 2 s tid)
 *   version 3  sequential addressing
 *   version 4  first add during load (each block covers 512 inputs)
 *   version 5  version 4 + warp shuffle for the last 32 values
 * partials[b] = sum of the inputs block b covers (256 for versions 1-3, 512
 * for 4-5), combined in that version's tree order; inputs past n count as 0.
 *   partials  rdx_ladder_num_partials(version, n) float32 values
 * This is the teaching ladder kept for comparison; rdx_sum_f32 is the fast
 * path.  Errors: RDX_ERR_INVALID_ARG for a version outside 1..5, n < 0, NULL
 * or misaligned pointers, overlap.
 */
rdx_status rdx_ladder_partials_f32(int version, const float* x, int64_t n, float* partials,
                                   cudaStream_t stream);

/* Number of partials rdx_ladder_partials_f32 writes: ceil(n / 256) for
 * versions 1-3, ceil(n / 512) for 4-5; -1 for a bad version or n < 0. */
int64_t rdx_ladder_num_partials(int version, int64_t n);

/*
 * rdx_ladder_sum_f32: *out = the sum of the partials of the page's block
 * reduction `version`, finished on the device.  On the page (demo 3) the
 * host adds the per-block partials after the kernel; here the same kernel
 * also writes them to `partials` (bit for bit those of
 * rdx_ladder_partials_f32) and then, in the same launch, the block that
 * arrives last at the library's completion counter adds all of them in a
 * fixed order into *out (the finish of rdx_sum_f32; the order depends on n,
 * the version and the 16-byte alignment of `partials`).  Each version thus
 * becomes a complete sum that can be timed against rdx_sum_f32.
 *   partials  rdx_ladder_num_partials(version, n) float32 values (scratch
 *             the caller owns; holds the partials afterwards)
 *   out       one float32; n == 0 writes 0.0f
 * Uses the (device, stream) workspace's completion counter (allocated on the
 * stream's first call, as for rdx_sum_f32).  Errors: as
 * rdx_ladder_partials_f32, plus NULL, misaligned or overlapping `out`, and
 * RDX_ERR_ALLOC if the workspace cannot be allocated.
 */
rdx_status rdx_ladder_sum_f32(int version, const float* x, int64_t n, float* partials, float* out,
                              cudaStream_t stream);

/*
 * Reductions split over several GPUs.
 * Page "03_shared_memory_sync_reduction.py", demo 3: each block leaves one
 * partial and the partials are added in a second step outside the kernel
 * (demo 2 of the page: blocks exchange data only by ending the kernel).
 * Over P GPUs the same two stages appear one level up:
 *   1. rank r takes the chunk [lo, hi) that rdx_shard_range gives it and
 *      reduces it with the one-GPU entry point (rdx_sum_f32, ...), leaving
 *      one partial in device memory;
 *   2. the caller gathers the P partials into one device array in rank order
 *      (e.g. an NCCL all-gather; this library runs no collective);
 *   3. every rank adds them with rdx_combine_* in rank order.
 * P and the chunking fix every addition, so all ranks get the same bits on
 * every run.  Row sums split by rows (granule 1) and need no exchange: rank
 * r's rows are its slice of the output.
 */

/*
 * rdx_shard_range: the chunk [*lo, *hi) of rank `rank` among `parts` ranks
 * sharing n elements.  The elements are cut into whole granules of `granule`
 * elements; each rank gets floor(G / parts) or one more granule (lower ranks
 * take the extra ones), the chunks follow one another in rank order, and the
 * last rank also takes the n mod granule elements after the last whole
 * granule.  So the chunks tile [0, n), every chunk but the first starts at a
 * multiple of `granule`, and the split depends on (n, parts, granule) only.
 * Pass granule = 16 / sizeof(element) (4 for float32 or int32, 8 for
 * bfloat16) to keep each chunk's 16-byte alignment that of the whole array,
 * 1 to split rows.  Host only: no CUDA call, no device needed.
 *   n        elements (or rows), >= 0
 *   parts    ranks, >= 1;  rank in [0, parts)
 *   granule  >= 1
 *   lo, hi   two distinct host int64 slots for the result
 * Errors: RDX_ERR_INVALID_ARG for any argument outside those ranges.
 */
rdx_status rdx_shard_range(int64_t n, int parts, int rank, int64_t granule, int64_t* lo, int64_t* hi);

/* The most partials one rdx_combine_* call adds (4096). */
int rdx_combine_max_parts(void);

/*
 * rdx_combine_f32: *out = parts[0] + parts[1] + ... + parts[p-1], float32,
 * added one by one in index (rank) order: ((parts[0] + parts[1]) + parts[2])
 * + ...  One small kernel on `stream`; the result is valid in stream order.
 * Combining the float32 partials of P chunks adds at most P - 1 roundings of
 * 2^-24 times the running magnitude to the chunks' own error.
 *   parts  p float32 values in device memory, 4-byte aligned
 *   p      1 .. rdx_combine_max_parts()
 *   out    one float32 in device memory, outside parts
 * Errors: RDX_ERR_INVALID_ARG for a NULL or misaligned pointer, p out of
 * range, out inside parts; RDX_ERR_CUDA if the launch fails.
 */
rdx_status rdx_combine_f32(const float* parts, int p, float* out, cudaStream_t stream);

/*
 * rdx_combine_f32x2: the same for the [sum, sum of squares] pairs of
 * rdx_sum_sumsq_*: out2[c] = parts2[0][c] + parts2[1][c] + ... in rank
 * order, for c = 0, 1.  parts2 holds p pairs (2p float32 values) and out2 one
 * pair, both 8-byte aligned.  Other arguments and errors as rdx_combine_f32.
 */
rdx_status rdx_combine_f32x2(const float* parts2, int p, float* out2, cudaStream_t stream);

/*
 * rdx_combine_i64: *out = parts[0] + ... + parts[p-1] in int64 (modulo 2^64,
 * as rdx_sum_i32_i64), exact and independent of the order.  parts and out
 * are 8-byte aligned.  Other arguments and errors as rdx_combine_f32.
 */
rdx_status rdx_combine_i64(const int64_t* parts, int p, int64_t* out, cudaStream_t stream);

/*
 * rdx_sum_f32_noalloc: *out = sum_{i<n} x[i], like rdx_sum_f32, but the call
 * allocates no device memory.  (The paper, the pages this library follows,
 * has no counterpart: this entry point exists for callers of this library,
 * not for the method.)
 *
 * For callers that may not cudaMalloc while they run: code inside a framework
 * whose allocator owns all device memory (an allocation behind its back is
 * not accounted for and can fail once the framework has reserved the memory),
 * latency-critical code (cudaMalloc/cudaFree may synchronize the device and
 * cost far more than the sum), and programs whose memory budget is fixed at
 * start-up.
 *
 * Same kernel, grid and summation order as rdx_sum_f32, so the same result.
 * Scratch (block partials and a completion counter) lives in one static
 * device array of 32 KiB + 256 B that every GPU loading this library holds
 * until the process exits.  Limit: 8192 block partials, the most any call
 * of this library's tiling uses; a launch that would need more is refused
 * with RDX_ERR_INVALID_ARG and a message in rdx_last_cuda_error().
 * All calls share the array and it keeps the last call's contents; the
 * counter is cleared on `stream` before every launch.  Calls whose kernels
 * overlap on the GPU (unordered streams) race on the array: order them.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.
 * Arguments and other errors as rdx_sum_f32.
 */
rdx_status rdx_sum_f32_noalloc(const float* x, int64_t n, float* out, cudaStream_t stream);

/*
 * rdx_bank_probe: the shared-memory bank-conflict probe of the page
 * "03_shared_memory_sync_reduction.py", demo 1.  One warp reads one word of
 * a 32*33-word shared array at index fn(tid) mod 1056, for
 *   pattern 0..5  stride 1, 2, 4, 8, 16, 32 (tid * stride)
 *   pattern 6     stride 33        pattern 7  stride 3
 *   pattern 8     one word (broadcast)        pattern 9  tid / 2
 * iters * rdx_bank_probe_loads_per_iter() times, and writes the clock cycles
 * those loads took to *cycles (device memory, 8-byte aligned); sink (32 words
 * of device memory) receives the loaded data so no load is optimised away.
 * A conflict of w ways costs about w times the cycles of a conflict-free
 * access.  Errors: RDX_ERR_INVALID_ARG for a pattern outside 0..9, iters
 * outside 1..2^20, NULL, misaligned or overlapping outputs.
 */
rdx_status rdx_bank_probe(int pattern, int iters, int64_t* cycles, uint32_t* sink, cudaStream_t stream);

/* Loads one iteration of rdx_bank_probe issues. */
int rdx_bank_probe_loads_per_iter(void);

/*
 * Checked build.  A library compiled with -DRDX_DEBUG=1 tests every global
 * load and store of its kernels against the buffer it belongs to; an access
 * outside is skipped, never performed, and counted.  (This stands in for a
 * memory sanitizer: run the workloads through the checked build and require
 * a count of zero.)
 * rdx_debug_build: 1 for a checked build, 0 otherwise.
 * rdx_debug_violations: *count = out-of-range accesses caught since the last
 * reset (always 0 in a normal build); synchronizes the device first;
 * reset != 0 clears the count.  RDX_ERR_INVALID_ARG if count is NULL.
 */
int rdx_debug_build(void);
rdx_status rdx_debug_violations(uint64_t* count, int reset);

/*
 * Bounded waits.  The narrow-row kernel of rdx_rowsum_f32 (rows of fewer
 * than 64 columns whose shared-memory reads would share a bank) stages each
 * tile with one bulk copy and waits on a shared-memory barrier for its bytes.
 * A wait that has not completed after one second (the GPU's global timer)
 * gives up: the block counts one timeout, waits once more (bounded) for its
 * copy to land, and exits without writing its rows' sums.  No such wait has
 * ever been seen to give up on a healthy GPU; a nonzero count means that
 * some row sums of the calls since the last reset were not written.
 * rdx_wait_timeouts: *count = those timeouts on the current device since the
 * last reset; synchronizes the device first; reset != 0 clears the count.
 * Errors: RDX_ERR_INVALID_ARG if count is NULL; RDX_ERR_CUDA if the device
 * or the counter cannot be read.
 * rdx_debug_stage_timeout: test hook for that path.  Enqueues one tile of
 * `rows` rows of `cols` floats (0 < cols < 64, 0 < rows * cols <= 6144, x
 * 16-byte aligned and holding at least 4 floats) whose barrier is armed for
 * 16 bytes more than its copy brings, so that its wait gives up after one
 * second: the count rises by one and out is not written.  Errors:
 * RDX_ERR_INVALID_ARG for arguments outside those limits, NULL pointers or
 * overlap; RDX_ERR_CUDA if the launch fails.
 */
rdx_status rdx_wait_timeouts(uint64_t* count, int reset);
rdx_status rdx_debug_stage_timeout(const float* x, int64_t rows, int64_t cols, float* out, cudaStream_t stream);

/* Static text for a status code ("ok", "invalid argument", ...). */
const char* rdx_status_string(rdx_status status);

/* Text of the last CUDA error seen by an rdx call on this host thread
 * ("" if none).  Valid until the next rdx call on the same thread. */
const char* rdx_last_cuda_error(void);

/* Free every cached workspace.  Call only when no rdx work is in flight. */
void rdx_shutdown(void);

/*
 * rdx_release_stream: free the workspace the library keeps for (current
 * device, `stream`) (for cudaStreamPerThread: this host thread's), if it has
 * one; returns 1 if one was freed, 0 if there was none.  For callers that
 * create and destroy many streams: without it every stream handle that made
 * a call keeps its workspace (rdx_workspace_bytes()) until rdx_shutdown().
 * Call it after the stream's rdx work has completed (e.g. after
 * cudaStreamSynchronize) and before the stream is destroyed; a later call on
 * the stream allocates a new workspace.  cudaFree may synchronize the device.
 */
int rdx_release_stream(cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* RDX_H */
