// shard.cu -- the two pieces a reduction split over several GPUs needs
// beyond the one-GPU entry points: where each GPU's chunk of the input lies,
// and the fixed-order combine of the GPUs' partial results.
//
// The page "03_shared_memory_sync_reduction.py", demo 3, ends each kernel
// with one partial per block and adds the partials in a second step outside
// the kernel; demo 2 of the same page notes that blocks exchange data only
// by ending the kernel.  Split over P GPUs the same shape appears one level
// up: each GPU reduces its own contiguous chunk to one partial (the whole
// one-GPU path, finish included), the P partials are gathered (a collective
// the caller runs, e.g. an all-gather), and each GPU adds them here in rank
// order.  With P and the chunking fixed, the result is the same bits on
// every GPU and every run.
//
// Chunking (shard_range): the n elements are cut into whole granules of g
// elements (g = 16 / element size keeps every chunk 16-byte aligned relative
// to the array, so each GPU's vector body starts where the whole array's
// would; g = 1 splits a count of rows).  P chunks get floor(G / P) or that
// plus one granules, the larger ones first, and the last chunk also takes the
// n mod g elements past the last whole granule.  It depends on n, P and g
// only.
//
// Combine (combine_kernel): one block loads the P partials into shared
// memory with coalesced loads, then one thread adds them in rank order,
// ((p0 + p1) + p2) + ..., in the accumulator type of the reduction (float32,
// float32 pairs for sum + sum of squares, int64 modulo 2^64).
#include "device.cuh"
#include "launch.h"

namespace rdx {
namespace {

constexpr int kCombineThreads = 256;

template <class T>
struct CombineAdd {
    __device__ static T add(T a, T b) { return a + b; }
};
template <>
struct CombineAdd<long long> {  // two's-complement addition, modulo 2^64
    __device__ static long long add(long long a, long long b) {
        return static_cast<long long>(static_cast<unsigned long long>(a) + static_cast<unsigned long long>(b));
    }
};

template <class T>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const T* __restrict__ parts, int p,
                                                                  T* __restrict__ out) {
    __shared__ T staged[kMaxCombineParts];
    pdl_wait();
    pdl_release();
    const size_t span = size_t(p) * sizeof(T);
    for (int i = threadIdx.x; i < p; i += kCombineThreads)
        if (guard(parts + i, sizeof(T), parts, span)) staged[i] = load_cg(parts + i);
    __syncthreads();
    if (threadIdx.x == 0) {
        T acc = staged[0];
        for (int i = 1; i < p; ++i) acc = CombineAdd<T>::add(acc, staged[i]);
        if (guard(out, sizeof(T), out, sizeof(T))) *out = acc;
    }
}

}  // namespace

RDX_DEFINE_VIOLATION_COUNTER(shard_out_of_range)

bool shard_range(int64_t n, int64_t parts, int64_t rank, int64_t granule, int64_t* lo, int64_t* hi) {
    if (n < 0 || parts < 1 || rank < 0 || rank >= parts || granule < 1) return false;
    const int64_t g = n / granule;        // whole granules
    const int64_t q = g / parts, r = g % parts;
    const int64_t first = rank * q + (rank < r ? rank : r);
    const int64_t count = q + (rank < r ? 1 : 0);
    *lo = first * granule;
    *hi = rank == parts - 1 ? n : (first + count) * granule;
    return true;
}

cudaError_t combine_launch(CombineType type, const void* parts, int p, void* out, cudaStream_t stream) {
    if (p < 1 || p > kMaxCombineParts) return cudaErrorInvalidValue;
    switch (type) {
        case CombineType::F32:
            return launch_pdl(combine_kernel<float>, dim3(1), dim3(kCombineThreads), stream,
                              static_cast<const float*>(parts), p, static_cast<float*>(out));
        case CombineType::F32x2:
            return launch_pdl(combine_kernel<SumSq2>, dim3(1), dim3(kCombineThreads), stream,
                              static_cast<const SumSq2*>(parts), p, static_cast<SumSq2*>(out));
        case CombineType::I64:
            return launch_pdl(combine_kernel<long long>, dim3(1), dim3(kCombineThreads), stream,
                              static_cast<const long long*>(parts), p, static_cast<long long*>(out));
    }
    return cudaErrorInvalidValue;
}

}  // namespace rdx
