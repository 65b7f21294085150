// ladder.cu -- the five block-level reductions of the page
// "03_shared_memory_sync_reduction.py", demo 3 (after Harris, "Optimizing
// Parallel Reduction in CUDA", 2007), as real CUDA kernels with the page's
// block of B = 256 threads and one float32 partial per block.
//
//   version 1  interleaved addressing: at step s the threads with
//              tid % 2s == 0 add sdata[tid + s] into sdata[tid]  (divergent)
//   version 2  interleaved addressing by consecutive threads:
//              index = 2 s tid, sdata[index] += sdata[index + s]  (bank
//              conflicts: stride 2s words)
//   version 3  sequential addressing: for s = B/2 .. 1 the first s threads
//              add sdata[tid + s] into sdata[tid]
//   version 4  version 3 with the first add during load: a block covers 2B
//              inputs, thread tid loads in[i] + in[i + B]
//   version 5  version 4, the shared-memory loop stopped at 64, then warp 0
//              adds sdata[tid] + sdata[tid + 32] and finishes with
//              __shfl_down_sync by 16, 8, 4, 2, 1
//
// They are kept as the comparison ladder for the fast kernel in reduce.cu.
// The page launches n / (B * per_thread) blocks and reads no index past the
// end; here the last block may be partial and inputs past n count as 0.
// The page adds the per-block partials on the host.  With kFinish the kernel
// also finishes on the device, as the fast kernel does: every block stores
// its partial and draws a ticket, and the block that draws the last one adds
// all partials in a fixed order and writes the total.
#include "device.cuh"
#include "launch.h"

namespace rdx {
namespace {

constexpr int B = kLadderBlock;

constexpr int kFinishLoads = 4;  // 16-byte loads of partials in flight per thread in the finish

template <int V, bool kFinish>
__global__ void __launch_bounds__(B) ladder_kernel(const float* __restrict__ in, int64_t n,
                                                   float* __restrict__ out, unsigned* __restrict__ counter,
                                                   float* __restrict__ total) {
    __shared__ float sdata[B];
    const int tid = threadIdx.x;
    const int64_t bx = blockIdx.x;

    const size_t span = size_t(n) * 4;
    if (V <= 3) {
        const int64_t i = bx * B + tid;
        sdata[tid] = i < n && guard(in + i, 4, in, span) ? in[i] : 0.f;
    } else {
        const int64_t i = bx * (2 * B) + tid;
        const float a = i < n && guard(in + i, 4, in, span) ? in[i] : 0.f;
        const float b = i + B < n && guard(in + i + B, 4, in, span) ? in[i + B] : 0.f;
        sdata[tid] = a + b;
    }
    const size_t out_span = size_t(gridDim.x) * 4;
    __syncthreads();

    if (V == 1) {
        for (int s = 1; s < B; s *= 2) {
            if (tid % (2 * s) == 0) sdata[tid] += sdata[tid + s];
            __syncthreads();
        }
    } else if (V == 2) {
        for (int s = 1; s < B; s *= 2) {
            const int index = 2 * s * tid;
            if (index < B) sdata[index] += sdata[index + s];
            __syncthreads();
        }
    } else if (V == 3 || V == 4) {
        for (int s = B / 2; s > 0; s >>= 1) {
            if (tid < s) sdata[tid] += sdata[tid + s];
            __syncthreads();
        }
    } else {
        for (int s = B / 2; s >= 64; s >>= 1) {
            if (tid < s) sdata[tid] += sdata[tid + s];
            __syncthreads();
        }
        if (tid < kWarpSize) {
            float val = sdata[tid] + sdata[tid + 32];
            for (int off = 16; off > 0; off >>= 1) val += __shfl_down_sync(kFullMask, val, off);
            if (tid == 0) sdata[0] = val;  // thread 0 stores the partial below, as in versions 1-4
        }
    }
    // thread 0 holds the block's partial in sdata[0] (its own write, or one
    // it saw before the last barrier)
    if (tid == 0 && guard(out + bx, 4, out, out_span)) out[bx] = sdata[0];
    if (!kFinish) return;

    // The device finish (last block done): thread 0 stored this block's
    // partial and now draws a ticket (acquire-release), so the block with
    // the last ticket sees every partial.  It adds them in a fixed order: the
    // few before the first 16-byte boundary and after the last whole 16-byte
    // vector one per thread; the vectors v = t, t + B, ... by thread t,
    // kFinishLoads loads in flight, into one float4 of four chains; then a
    // block tree.  Every block waits for its ticket before it exits: with
    // blocks this short (one or two inputs per thread), that round trip is a
    // large part of each block's life.
    __shared__ unsigned last_block;
    __shared__ float warp_sums[B / kWarpSize];
    if (tid == 0)
        last_block = guard(counter, 4, counter, 4) ? take_ticket(counter) == gridDim.x - 1 : 0u;
    __syncthreads();
    if (!last_block) return;
    const int64_t g = gridDim.x;
    int64_t head = int64_t(((16u - (unsigned(reinterpret_cast<uintptr_t>(out)) & 15u)) & 15u) >> 2);
    if (head > g) head = g;
    const int64_t m = (g - head) >> 2;  // whole float4 vectors
    const int64_t tail0 = head + 4 * m;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (tid < head && guard(out + tid, 4, out, out_span)) acc.x += load_cg(out + tid);
    if (tid < g - tail0 && guard(out + tail0 + tid, 4, out, out_span)) acc.y += load_cg(out + tail0 + tid);
    const float4* __restrict__ ov = reinterpret_cast<const float4*>(out + head);
    for (int64_t j = tid; j < m; j += kFinishLoads * B) {
        float4 p[kFinishLoads];
#pragma unroll
        for (int u = 0; u < kFinishLoads; ++u)
            p[u] = j + u * B < m && guard(ov + j + u * B, 16, out, out_span) ? __ldcg(ov + j + u * B)
                                                                            : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int u = 0; u < kFinishLoads; ++u) {
            acc.x += p[u].x; acc.y += p[u].y; acc.z += p[u].z; acc.w += p[u].w;
        }
    }
    const float sum = block_sum<B>((acc.x + acc.y) + (acc.z + acc.w), warp_sums, 0.f);
    if (tid == 0) {
        if (guard(total, 4, total, 4)) *total = sum;
        if (guard(counter, 4, counter, 4)) *counter = 0u;  // ready for the next call on this stream
    }
}

}  // namespace

RDX_DEFINE_VIOLATION_COUNTER(ladder_out_of_range)

cudaError_t ladder_launch(int version, const float* x, int64_t n, float* partials, int64_t blocks,
                          unsigned* counter, float* total, cudaStream_t stream) {
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
    const unsigned g = unsigned(blocks);
#define RDX_LADDER(V)                                                                   \
    (total ? ladder_kernel<V, true><<<g, B, 0, stream>>>(x, n, partials, counter, total) \
           : ladder_kernel<V, false><<<g, B, 0, stream>>>(x, n, partials, counter, total))
    switch (version) {
        case 1: RDX_LADDER(1); break;
        case 2: RDX_LADDER(2); break;
        case 3: RDX_LADDER(3); break;
        case 4: RDX_LADDER(4); break;
        case 5: RDX_LADDER(5); break;
        default: return cudaErrorInvalidValue;
    }
#undef RDX_LADDER
    return cudaGetLastError();
}

}  // namespace rdx
