// launch.h -- host-side interface between the C-ABI shim (api.cu) and the
// kernel translation units.  Internal: not installed, not part of the ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace rdx {

// The scalar reductions of the C ABI.
enum class Op : int { SumF32 = 0, SumSqF32, SumBF16, SumSqBF16, SumI32, kCount };

// Properties of the current device that the launch heuristics need.
struct DeviceCaps {
    int ordinal = -1;
    int sms = 0;             // streaming multiprocessors
    int cc_major = 0;
    int cc_minor = 0;
    int reduce_bps[int(Op::kCount)] = {};  // resident blocks per SM, per reduce kernel
    int rowsum_cta_bps = 0;
    int rowsum_warp_bps = 0;
};

// ---- scalar reductions (reduce.cu) ----------------------------------------
int reduce_block_threads();
int reduce_unroll();
int reduce_vec_elems(Op op);
size_t reduce_elem_bytes(Op op);
size_t reduce_acc_bytes(Op op);
cudaError_t reduce_blocks_per_sm(Op op, int* blocks);
// Grid for n elements starting at address x: whole waves of resident blocks,
// fewer when n is too small to give every thread one unrolled iteration.
// Depends on n, the alignment of x and the device only.
int reduce_grid(const DeviceCaps& dev, Op op, int64_t n, int64_t head);
// head = elements before the first 16-byte boundary of x (at most n).
int64_t reduce_head(Op op, const void* x, int64_t n);
// partials: grid accumulator slots; ticket: a zeroed completion counter.
cudaError_t reduce_launch(Op op, const void* x, int64_t n, int64_t head, void* partials,
                          unsigned* ticket, void* out, int grid, cudaStream_t stream);

// ---- row-segmented sum (rowsum.cu) ----------------------------------------
cudaError_t rowsum_blocks_per_sm(int* cta_bps, int* warp_bps);
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
