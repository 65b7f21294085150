// launch.h -- host-side interface between the C-ABI shim (api.cu) and the
// kernel translation units.  Internal: not installed, not part of the ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace rdx {

// Launch `kernel` with programmatic stream serialization: it may start while
// the kernel ahead of it in the stream drains, and waits in pdl_wait() until
// that kernel's writes are visible (see device.cuh).
template <class... KArgs, class... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// The scalar reductions of the C ABI, numbered as the RDX_OP_* codes
// (SumSumSq*: sum and sum of squares in one pass).
enum class Op : int {
    SumF32 = 0,
    SumSqF32,
    SumBF16,
    SumSqBF16,
    SumI32,
    SumSumSqF32,
    SumSumSqBF16,
    MaxF32,
    MaxI32,
    kCount
};

// Properties of the current device (checked once per device).
struct DeviceCaps {
    int ordinal = -1;
    int sms = 0;  // streaming multiprocessors
    int cc_major = 0;
    int cc_minor = 0;
};

// ---- tiled reductions (reduce.cu) -----------------------------------------
// Most tiles (= block partials) one call of the tiled reductions uses, over
// all its rows: the size of every partials buffer (the library's workspace,
// a caller's workspace, the static scratch of the no-allocation sum).
#ifndef RDX_REDUCE_MAX_TILES
#define RDX_REDUCE_MAX_TILES 8192
#endif
constexpr int64_t kReduceMaxTiles = RDX_REDUCE_MAX_TILES;
// One call sums `rows` segments of `cols` elements, segment r starting at
// x + r * ld (the scalar reductions: rows = 1).  Each row is cut into `tiles`
// tiles of `tile` 16-byte vectors, one block each; the plan depends only on
// rows and cols.  rows * tiles <= reduce_max_partials() for rows <= that.
struct ReducePlan {
    int64_t tile = 0;
    int64_t tiles = 1;
    bool large = false;  // the deeper kernel variant (8 loads in flight, 4 blocks per SM)
    // the finish runs as a second kernel (one block per row) after the tiles'
    // grid instead of in its last block; only when tiles > 1
    bool separate_finish = false;
};
int reduce_block_threads();
int64_t reduce_max_partials();
int reduce_vec_elems(Op op);
size_t reduce_elem_bytes(Op op);
size_t reduce_acc_bytes(Op op);
ReducePlan reduce_plan(Op op, int64_t rows, int64_t cols);
// Whether `op` finishes through an accumulator word instead of partials (the
// int64 sum and the maxima, whose result does not depend on the order; rows
// must then be 1).
bool reduce_uses_words(Op op);
// partials: rows * plan.tiles slots (reduce_acc_bytes each; not touched by
// the word-finishing ops); counters: rows zeroed completion counters, left
// zeroed (not touched when plan.separate_finish); words: one zeroed 8-byte
// accumulator word, left zeroed (only the word-finishing ops touch it; it may
// be NULL for the others).  None of these is touched when plan.tiles == 1.
// out: rows results.  Enqueues one kernel, or two when plan.separate_finish.
cudaError_t reduce_launch(Op op, const void* x, int64_t rows, int64_t cols, int64_t ld, const ReducePlan& plan,
                          void* partials, unsigned* counters, unsigned long long* words, void* out,
                          cudaStream_t stream);

// ---- row-segmented sum (rowsum.cu) ----------------------------------------
// Rows of `cols` elements starting every `ld` elements; no workspace.
cudaError_t rowsum_launch(const float* x, int64_t rows, int64_t cols, int64_t ld, float* out, cudaStream_t stream);
// Whether a (rows, cols) matrix is better summed by the tiled reduce kernel
// (few, long rows: each row split over many blocks).
bool rowsum_use_split(int64_t rows, int64_t cols);
// Whether contiguous narrow rows go through shared memory (rowsum_narrow_kernel):
// depends on cols, ld and the 4/8/16-byte alignment of x.
bool rowsum_use_narrow(const float* x, int64_t cols, int64_t ld);
constexpr int64_t kMaxSplitRows = 2048;

// ---- the page's bank-conflict probe (banks.cu) -------------------------------
constexpr int kBankPatterns = 10;
int bank_probe_loads_per_iter();
// One warp; cycles[0] = clock cycles of iters * loads_per_iter loads; sink: 32 words.
cudaError_t bank_probe_launch(int pattern, int iters, long long* cycles, unsigned* sink, cudaStream_t stream);

// ---- reductions split over several GPUs (shard.cu) ---------------------------
// Chunk [*lo, *hi) of rank `rank` among `parts` (false for bad arguments).
bool shard_range(int64_t n, int64_t parts, int64_t rank, int64_t granule, int64_t* lo, int64_t* hi);
constexpr int kMaxCombineParts = 4096;  // partials one combine adds, at most
enum class CombineType : int { F32, F32x2, I64 };
// *out = parts[0] + parts[1] + ... + parts[p - 1], added in that order.
cudaError_t combine_launch(CombineType type, const void* parts, int p, void* out, cudaStream_t stream);

// ---- checked build (RDX_DEBUG=1): out-of-range accesses caught, per file ------
unsigned long long reduce_out_of_range(bool reset);
unsigned long long rowsum_out_of_range(bool reset);
// Staging waits of the narrow-row kernel that gave up on the current device
// (~0 if the count could not be read); reset clears it.
unsigned long long rowsum_stage_timeouts(bool reset);
// Test hook: one narrow-row tile (rows * cols <= 6144 floats, x 16-byte
// aligned) whose staging wait cannot complete, so that it gives up.
cudaError_t rowsum_stage_timeout_probe(const float* x, int64_t rows, int64_t cols, float* out, cudaStream_t stream);
unsigned long long ladder_out_of_range(bool reset);
unsigned long long shard_out_of_range(bool reset);

// ---- error text shared by every entry point (api.cu) ------------------------
// Replace the calling thread's rdx_last_cuda_error() text.
void set_last_error(const char* text);

// ---- the page's five block reductions (ladder.cu) --------------------------
constexpr int kLadderBlock = 256;
// partials: `blocks` floats.  With total != NULL the kernel also adds the
// partials on the device into *total, using *counter (zero before the launch,
// left zero after) as the completion counter.
cudaError_t ladder_launch(int version, const float* x, int64_t n, float* partials, int64_t blocks,
                          unsigned* counter, float* total, cudaStream_t stream);

}  // namespace rdx
