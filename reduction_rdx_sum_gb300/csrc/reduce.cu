// reduce.cu -- one-pass scalar sum reductions (float32, float32 squares,
// bfloat16 -> float32, int32 -> int64) with a deterministic on-device finish.
//
// The page "03_shared_memory_sync_reduction.py", demo 3, walks from a
// divergent shared-memory tree (version 1) to "first add during load" plus a
// warp-shuffle finish (version 5), and ends each kernel with one partial per
// block that the host adds up.  This kernel keeps version 5's shape and takes
// its two ideas further for a GPU with 152 SMs and HBM3e:
//   * add on load: each thread walks the array in grid-stride order with
//     kUnroll independent 16-byte loads in flight and folds each vector into
//     its own register accumulator (version 4's two elements per thread become
//     thousands);
//   * shuffle trees: a warp tree, then one shared-memory word per warp, then
//     a warp tree over those words (the shared-memory tree of versions 1-4 is
//     gone; one barrier per block);
//   * the per-block partials are finished on the device: the block that
//     arrives last at a completion counter (acquire-release atomic) adds all
//     partials in a fixed order and resets the counter.  Nothing waits on
//     anything, and no float atomics are used, so the result does not depend
//     on which block finishes first.
#include "device.cuh"
#include "launch.h"

#ifndef RDX_REDUCE_BLOCK
#define RDX_REDUCE_BLOCK 256
#endif
#ifndef RDX_REDUCE_UNROLL
#define RDX_REDUCE_UNROLL 8
#endif

namespace rdx {
namespace {

constexpr int kBlock = RDX_REDUCE_BLOCK;    // threads per block
constexpr int kUnroll = RDX_REDUCE_UNROLL;  // 16-byte loads in flight per thread
static_assert((kUnroll & (kUnroll - 1)) == 0, "kUnroll must be a power of two");

// Completion counter: acquire-release at GPU scope, so the partial this
// thread stored before is visible to the block that draws the last ticket,
// and that block sees every other block's partial.
__device__ __forceinline__ unsigned take_ticket(unsigned* counter) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
                 : "=r"(old)
                 : "l"(counter), "r"(1u)
                 : "memory");
    return old;
}

template <class P>
__global__ void __launch_bounds__(kBlock)
reduce_kernel(const typename P::In* __restrict__ x, int64_t n, int64_t head,
              typename P::Acc* __restrict__ partials, unsigned* __restrict__ counter,
              typename P::Acc* __restrict__ out) {
    using Acc = typename P::Acc;
    constexpr int V = P::kVec;
    __shared__ Acc smem[kBlock / kWarpSize];
    __shared__ unsigned last_block;

    const int64_t nthreads = int64_t(gridDim.x) * kBlock;
    const int64_t g = int64_t(blockIdx.x) * kBlock + threadIdx.x;
    const int64_t m = (n - head) / V;  // whole 16-byte vectors after the head
    const int64_t tail0 = head + m * V;
    const uint4* __restrict__ xv = reinterpret_cast<const uint4*>(x + head);

    Acc acc[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) acc[u] = Acc(0);

    // Fewer than V elements before the first 16-byte boundary and after the
    // last whole vector: the first threads take one each.
    if (g < head) acc[0] += P::term(x[g]);
    if (g < n - tail0) acc[kUnroll - 1] += P::term(x[tail0 + g]);

    int64_t i = g;
    for (; i + (kUnroll - 1) * nthreads < m; i += kUnroll * nthreads) {
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) v[u] = ld_stream16(xv + i + u * nthreads);
        batch_fence(v);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) acc[u] += P::fold(v[u]);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const int64_t j = i + u * nthreads;
        if (j < m) acc[u] += P::fold(ld_stream16(xv + j));
    }

    Acc a = block_sum<kBlock>(fold_array(acc), smem);

    if (gridDim.x == 1) {
        if (threadIdx.x == 0) *out = a;
        return;
    }
    if (threadIdx.x == 0) {
        partials[blockIdx.x] = a;
        last_block = take_ticket(counter) == gridDim.x - 1;
    }
    __syncthreads();
    if (!last_block) return;

    // The last block: every partial is in place.  Add them in block order
    // (thread t takes t, t + kBlock, ...; then the block tree).
    Acc b = Acc(0);
    for (int j = threadIdx.x; j < int(gridDim.x); j += kBlock) b += __ldcg(partials + j);
    b = block_sum<kBlock>(b, smem);
    if (threadIdx.x == 0) {
        *out = b;
        *counter = 0u;  // ready for the next call on this stream
    }
}

template <class P>
cudaError_t launch_typed(const void* x, int64_t n, int64_t head, void* partials, unsigned* counter, void* out,
                         int grid, cudaStream_t stream) {
    reduce_kernel<P><<<grid, kBlock, 0, stream>>>(static_cast<const typename P::In*>(x), n, head,
                                                   static_cast<typename P::Acc*>(partials), counter,
                                                   static_cast<typename P::Acc*>(out));
    return cudaGetLastError();
}

template <class P>
cudaError_t occupancy_typed(int* blocks) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, reduce_kernel<P>, kBlock, 0);
}

}  // namespace

int reduce_block_threads() { return kBlock; }
int reduce_unroll() { return kUnroll; }

int reduce_vec_elems(Op op) {
    switch (op) {
        case Op::SumBF16:
        case Op::SumSqBF16: return 8;
        default: return 4;
    }
}

size_t reduce_elem_bytes(Op op) { return 16 / size_t(reduce_vec_elems(op)); }

size_t reduce_acc_bytes(Op op) { return op == Op::SumI32 ? 8 : 4; }

cudaError_t reduce_blocks_per_sm(Op op, int* blocks) {
    switch (op) {
        case Op::SumF32: return occupancy_typed<SumF32>(blocks);
        case Op::SumSqF32: return occupancy_typed<SumSqF32>(blocks);
        case Op::SumBF16: return occupancy_typed<SumBF16>(blocks);
        case Op::SumSqBF16: return occupancy_typed<SumSqBF16>(blocks);
        case Op::SumI32: return occupancy_typed<SumI32>(blocks);
        default: return cudaErrorInvalidValue;
    }
}

int64_t reduce_head(Op op, const void* x, int64_t n) {
    const uintptr_t mis = reinterpret_cast<uintptr_t>(x) & 15u;
    const int64_t head = mis ? int64_t((16u - mis) / reduce_elem_bytes(op)) : 0;
    return head < n ? head : n;
}

int reduce_grid(const DeviceCaps& dev, Op op, int64_t n, int64_t head) {
    const int64_t m = (n - head) / reduce_vec_elems(op);
    const int64_t per_block = int64_t(kBlock) * kUnroll;  // vectors one block loads per iteration
    const int64_t want = (m + per_block - 1) / per_block;
    const int64_t cap = int64_t(dev.sms) * dev.reduce_bps[int(op)];
    int64_t g = want < cap ? want : cap;
    return int(g < 1 ? 1 : g);
}

cudaError_t reduce_launch(Op op, const void* x, int64_t n, int64_t head, void* partials, unsigned* counter,
                          void* out, int grid, cudaStream_t stream) {
    switch (op) {
        case Op::SumF32: return launch_typed<SumF32>(x, n, head, partials, counter, out, grid, stream);
        case Op::SumSqF32: return launch_typed<SumSqF32>(x, n, head, partials, counter, out, grid, stream);
        case Op::SumBF16: return launch_typed<SumBF16>(x, n, head, partials, counter, out, grid, stream);
        case Op::SumSqBF16: return launch_typed<SumSqBF16>(x, n, head, partials, counter, out, grid, stream);
        case Op::SumI32: return launch_typed<SumI32>(x, n, head, partials, counter, out, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace rdx
