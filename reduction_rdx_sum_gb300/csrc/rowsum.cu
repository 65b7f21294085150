// rowsum.cu -- row-segmented float32 sum: out[r] = sum of row r of a
// row-major (rows, cols) matrix.
//
// On the page "03_shared_memory_sync_reduction.py", demo 3, every block writes
// the sum of its own contiguous segment to out[blockIdx]: a segmented sum.
// Here a segment is a row, and the work per row decides who sums it:
//   * short rows (cols <= kWarpRowMaxCols): a group of LPR lanes per row
//     (LPR = 1 .. 32, about four 16-byte vectors per lane), 32/LPR rows per
//     warp step; a warp finishes 32 consecutive rows and writes their sums as
//     one coalesced 128-byte store;
//   * long rows: one block per row, the same add-on-load loop and block tree
//     as the scalar reduction, a direct store of the row's sum.
// A row's summation order depends only on its address and length, never on
// the grid, so the result is bitwise reproducible.  No workspace is needed.
#include "device.cuh"
#include "launch.h"

namespace rdx {
namespace {

constexpr int kCtaBlock = 256;          // threads per row, long rows
constexpr int kCtaUnroll = 4;           // 16-byte loads in flight per thread, long rows
constexpr int kWarpBlock = 256;         // threads per block, short rows
constexpr int64_t kWarpRowMaxCols = 1024;

// Elements of a row before its first 16-byte boundary (rows of a matrix with
// cols % 4 != 0 start at varying alignments).
__device__ __forceinline__ int64_t row_head(const float* row, int64_t cols) {
    const int64_t h = int64_t(((16u - (unsigned(reinterpret_cast<uintptr_t>(row)) & 15u)) & 15u) >> 2);
    return h < cols ? h : cols;
}

// Sum of lane l's share of one row, the row split among LPR lanes.
template <int LPR>
__device__ __forceinline__ float row_share(const float* __restrict__ row, int64_t cols, int l) {
    const int64_t head = row_head(row, cols);
    const int64_t m = (cols - head) >> 2;
    const int64_t tail0 = head + 4 * m;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    // up to 3 scalars before the first and after the last whole vector; a
    // group may have fewer than 3 lanes, so stride by LPR
    for (int64_t k = l; k < head; k += LPR) acc[0] += __ldg(row + k);
    for (int64_t k = tail0 + l; k < cols; k += LPR) acc[1] += __ldg(row + k);
    const uint4* __restrict__ rv = reinterpret_cast<const uint4*>(row + head);
    int64_t j = l;
    for (; j + 3 * LPR < m; j += 4 * LPR) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = ld_stream16(rv + j + u * LPR);
        batch_fence(v);
#pragma unroll
        for (int u = 0; u < 4; ++u) acc[u] += SumF32::fold(v[u]);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        if (j + u * LPR < m) acc[u] += SumF32::fold(ld_stream16(rv + j + u * LPR));
    }
    return fold_array(acc);
}

// Short rows.  Warp w takes batches of 32 consecutive rows; within a batch,
// step s has group g (lanes g*LPR .. g*LPR+LPR-1) sum row s*NG + g, and lane
// i keeps the total of row i, so the 32 sums leave in one coalesced store.
template <int LPR>
__global__ void __launch_bounds__(kWarpBlock)
rowsum_warp_kernel(const float* __restrict__ x, int64_t rows, int64_t cols, float* __restrict__ out) {
    constexpr int NG = kWarpSize / LPR;  // rows in flight per warp step
    const int lane = threadIdx.x % kWarpSize;
    const int grp = lane / LPR;
    const int l = lane % LPR;
    const int64_t warp = (int64_t(blockIdx.x) * kWarpBlock + threadIdx.x) / kWarpSize;
    const int64_t nwarps = int64_t(gridDim.x) * (kWarpBlock / kWarpSize);
    const int64_t nbatch = (rows + kWarpSize - 1) / kWarpSize;
    for (int64_t b = warp; b < nbatch; b += nwarps) {
        const int64_t r0 = b * kWarpSize;
        float mine = 0.f;
#pragma unroll
        for (int step = 0; step < LPR; ++step) {
            const int64_t r = r0 + step * NG + grp;
            float s = 0.f;
            if (r < rows) s = row_share<LPR>(x + r * cols, cols, l);
            s = group_allreduce<LPR>(s);
            const float t = __shfl_sync(kFullMask, s, (lane % NG) * LPR);
            if (lane / NG == step) mine = t;
        }
        if (r0 + lane < rows) out[r0 + lane] = mine;
    }
}

// Long rows: one block per row (a block loops over rows r, r + gridDim.x, ...).
__global__ void __launch_bounds__(kCtaBlock)
rowsum_cta_kernel(const float* __restrict__ x, int64_t rows, int64_t cols, float* __restrict__ out) {
    __shared__ float smem[kCtaBlock / kWarpSize];
    const int t = threadIdx.x;
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const float* __restrict__ row = x + r * cols;
        const int64_t head = row_head(row, cols);
        const int64_t m = (cols - head) >> 2;
        const int64_t tail0 = head + 4 * m;
        float acc[kCtaUnroll];
#pragma unroll
        for (int u = 0; u < kCtaUnroll; ++u) acc[u] = 0.f;
        if (t < head) acc[0] += __ldg(row + t);
        if (t < cols - tail0) acc[kCtaUnroll - 1] += __ldg(row + tail0 + t);
        const uint4* __restrict__ rv = reinterpret_cast<const uint4*>(row + head);
        int64_t i = t;
        for (; i + (kCtaUnroll - 1) * kCtaBlock < m; i += kCtaUnroll * kCtaBlock) {
            uint4 v[kCtaUnroll];
#pragma unroll
            for (int u = 0; u < kCtaUnroll; ++u) v[u] = ld_stream16(rv + i + u * kCtaBlock);
            batch_fence(v);
#pragma unroll
            for (int u = 0; u < kCtaUnroll; ++u) acc[u] += SumF32::fold(v[u]);
        }
#pragma unroll
        for (int u = 0; u < kCtaUnroll; ++u) {
            if (i + u * kCtaBlock < m) acc[u] += SumF32::fold(ld_stream16(rv + i + u * kCtaBlock));
        }
        const float a = block_sum<kCtaBlock>(fold_array(acc), smem);
        if (t == 0) out[r] = a;
        __syncthreads();  // smem is reused by the next row
    }
}

// Lanes per row: about four 16-byte vectors per lane, a power of two <= 32.
int lanes_per_row(int64_t cols) {
    const int64_t vecs = cols / 4;
    int lpr = 1;
    while (lpr < 32 && int64_t(lpr) * 2 * 4 <= vecs) lpr *= 2;
    return lpr;
}

template <int LPR>
cudaError_t launch_warp(const float* x, int64_t rows, int64_t cols, float* out, cudaStream_t stream) {
    constexpr int64_t kWarpsPerBlock = kWarpBlock / kWarpSize;
    const int64_t nbatch = (rows + kWarpSize - 1) / kWarpSize;
    int64_t blocks = (nbatch + kWarpsPerBlock - 1) / kWarpsPerBlock;
    if (blocks > 0x7fffffff) blocks = 0x7fffffff;
    rowsum_warp_kernel<LPR><<<unsigned(blocks), kWarpBlock, 0, stream>>>(x, rows, cols, out);
    return cudaGetLastError();
}

}  // namespace

cudaError_t rowsum_blocks_per_sm(int* cta_bps, int* warp_bps) {
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(cta_bps, rowsum_cta_kernel, kCtaBlock, 0);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(warp_bps, rowsum_warp_kernel<16>, kWarpBlock, 0);
}

cudaError_t rowsum_launch(const DeviceCaps& dev, const float* x, int64_t rows, int64_t cols, float* out,
                          cudaStream_t stream) {
    (void)dev;
    if (rows <= 0) return cudaSuccess;
    if (cols <= kWarpRowMaxCols) {
        switch (lanes_per_row(cols)) {
            case 1: return launch_warp<1>(x, rows, cols, out, stream);
            case 2: return launch_warp<2>(x, rows, cols, out, stream);
            case 4: return launch_warp<4>(x, rows, cols, out, stream);
            case 8: return launch_warp<8>(x, rows, cols, out, stream);
            case 16: return launch_warp<16>(x, rows, cols, out, stream);
            default: return launch_warp<32>(x, rows, cols, out, stream);
        }
    }
    const int64_t blocks = rows < 0x7fffffff ? rows : 0x7fffffff;
    rowsum_cta_kernel<<<unsigned(blocks), kCtaBlock, 0, stream>>>(x, rows, cols, out);
    return cudaGetLastError();
}

}  // namespace rdx
