// banks.cu -- the shared-memory bank-conflict probe of the page
// "03_shared_memory_sync_reduction.py", demo 1: one warp reads one 4-byte
// word of a 32 x 33-word shared array at index fn(tid) for ten patterns
// (strides 1, 2, 4, 8, 16, 32, 33, 3, a broadcast, and pairs of threads on
// one word).  Each load is issued kProbeUnroll times per iteration; the
// kernel reports the clock cycles per load instruction, which grow with the
// number of wavefronts an access takes (ncu's shared-memory wavefront
// counters give the exact count).  It checks the conflict-free design of the
// reductions' cross-warp stage and the counters used to show it.
#include "device.cuh"
#include "launch.h"

namespace rdx {
namespace {

constexpr int kWords = 32 * 33;
constexpr int kProbeUnroll = 16;

__device__ __forceinline__ int probe_index(int pattern, int t) {
    switch (pattern) {
        case 0: return t;
        case 1: return 2 * t;
        case 2: return 4 * t;
        case 3: return 8 * t;
        case 4: return 16 * t;
        case 5: return 32 * t;
        case 6: return 33 * t;
        case 7: return 3 * t;
        case 8: return 0;
        default: return t / 2;
    }
}

__global__ void __launch_bounds__(32) bank_probe_kernel(int pattern, int iters, long long* __restrict__ cycles,
                                                        unsigned* __restrict__ sink) {
    __shared__ unsigned words[kWords];
    const int t = threadIdx.x;
    for (int i = t; i < kWords; i += 32) words[i] = unsigned(i) * 2654435761u;
    __syncwarp();
    const unsigned addr = unsigned(__cvta_generic_to_shared(&words[probe_index(pattern, t) % kWords]));
    unsigned acc = 0;
    // one untimed pass warms the instruction cache
    for (int pass = 0; pass < 2; ++pass) {
        const long long t0 = clock64();
        for (int it = 0; it < iters; ++it) {
#pragma unroll
            for (int k = 0; k < kProbeUnroll; ++k) {
                // .volatile: every load is performed (same address each time,
                // which the backend would otherwise load once)
                unsigned v;
                asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
                acc ^= v;
            }
        }
        const long long t1 = clock64();
        if (pass == 1 && t == 0) cycles[0] = t1 - t0;
    }
    sink[t] = acc;
}

}  // namespace

int bank_probe_loads_per_iter() { return kProbeUnroll; }

cudaError_t bank_probe_launch(int pattern, int iters, long long* cycles, unsigned* sink, cudaStream_t stream) {
    bank_probe_kernel<<<1, 32, 0, stream>>>(pattern, iters, cycles, sink);
    return cudaGetLastError();
}

}  // namespace rdx
