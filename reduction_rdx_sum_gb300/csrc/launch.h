// launch.h -- host-side interface between the C-ABI shim (api.cu) and the
// kernel translation units.  Internal: not installed, not part of the ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace rdx {

// The scalar reductions of the C ABI (the last two give sum and sum of squares
// in one pass).
enum class Op : int { SumF32 = 0, SumSqF32, SumBF16, SumSqBF16, SumI32, SumSumSqF32, SumSumSqBF16, kCount };

// Properties of the current device that the launch heuristics need.
struct DeviceCaps {
    int ordinal = -1;
    int sms = 0;  // streaming multiprocessors
    int cc_major = 0;
    int cc_minor = 0;
    int rowsum_cta_bps = 0;    // resident blocks per SM of the long-row kernel
    int rowsum_group_bps = 0;  // resident blocks per SM of the short-row kernel
};

// ---- scalar reductions (reduce.cu) ----------------------------------------
// How one call is cut: `head` elements before the first 16-byte boundary of x,
// then tiles of `tile` 16-byte vectors, one block each (`grid` blocks, at most
// reduce_max_partials()).  Depends only on n and x's alignment.
struct ReducePlan {
    int64_t head = 0;
    int64_t tile = 0;
    int64_t grid = 1;
};
int reduce_block_threads();
int reduce_unroll();
int64_t reduce_max_partials();
int reduce_vec_elems(Op op);
size_t reduce_elem_bytes(Op op);
size_t reduce_acc_bytes(Op op);
ReducePlan reduce_plan(Op op, const void* x, int64_t n);
// partials: plan.grid accumulator slots (reduce_acc_bytes each); counter: a
// zeroed completion counter.  Neither is touched when plan.grid == 1.
cudaError_t reduce_launch(Op op, const void* x, int64_t n, const ReducePlan& plan, void* partials,
                          unsigned* counter, void* out, cudaStream_t stream);

// ---- row-segmented sum (rowsum.cu) ----------------------------------------
cudaError_t rowsum_blocks_per_sm(int* cta_bps, int* group_bps);
cudaError_t rowsum_launch(const DeviceCaps& dev, const float* x, int64_t rows, int64_t cols, float* out,
                          cudaStream_t stream);

// ---- error text shared by every entry point (api.cu) ------------------------
// Replace the calling thread's rdx_last_cuda_error() text.
void set_last_error(const char* text);

// ---- the page's five block reductions (ladder.cu) --------------------------
constexpr int kLadderBlock = 256;
cudaError_t ladder_launch(int version, const float* x, int64_t n, float* partials, int64_t blocks,
                          cudaStream_t stream);

}  // namespace rdx
