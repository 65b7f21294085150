// rowsum.cu -- row-segmented float32 sum: out[r] = sum of row r of a
// row-major (rows, cols) matrix.
//
// On the page "03_shared_memory_sync_reduction.py", demo 3, every block writes
// the sum of its own contiguous segment to out[blockIdx]: a segmented sum.
// Here a segment is a row, and the work per row decides who sums it:
//   * narrow rows (contiguous, cols < kNarrowMaxCols, i.e. at most 64; see
//     rowsum_use_narrow):
//     the matrix is read as one flat array, tile by tile, into shared
//     memory, and each thread sums whole rows from there;
//   * short rows (cols <= kFitRowMaxCols): a group of LPR lanes per row, each
//     lane holding at most four 16-byte vectors of the row, so a warp sums
//     32/LPR consecutive rows per step; the loads of kRowSteps steps are
//     issued together before any of them is reduced; where a power of two
//     of lanes would leave the slots half empty, groups of 5, 6, 9 or 10
//     lanes (see rowsum_fitg_lanes);
//   * staged rows (see rowsum_staged_lanes): short rows that would leave
//     those lanes' load slots half empty, and medium rows up to
//     kStagedMaxCols, are staged like narrow rows, 24 KiB of whole rows per
//     bulk copy, and summed from shared memory by a group of lanes per row;
//     rows with a leading dimension join them when the gap between rows is
//     small (the span is copied, gaps included), or from kRowsStagedMinCols
//     columns one bulk copy per row;
//   * other medium rows (cols <= kGroupRowMaxCols): a warp per row, looping
//     over the row four vectors per lane at a time;
//   * long rows: one block per row, the same add-on-load loop and block tree
//     as the scalar reduction (twice the loads in flight at half the
//     occupancy from kCtaDeepCols columns), a direct store of the row's sum.
// Rows may start every ld >= cols elements (a leading dimension).  Rows that
// are not 16-byte aligned have up to 3 floats before their first and after
// their last whole vector: the narrow kernel reads such rows from shared
// memory in a rotated order, the staged kernels load them one by one beside
// the bulk copy, and the others fetch them without holding the row's vector
// loads back (cp.async copies, or registers loaded ahead).  Every kernel is launched with programmatic dependent launch.  A
// row's summation order depends only on the shape and the alignment of x,
// never on the grid or the device, so the result is bitwise reproducible.  No
// workspace is needed.  (Few, very long rows go to the tiled kernel of
// reduce.cu instead; see rowsum_use_split.)
#include "device.cuh"
#include "launch.h"

namespace rdx {
namespace {

constexpr int kCtaBlock = 256;   // threads per row, long rows
constexpr int kCtaUnroll = 4;    // 16-byte loads in flight per thread, long rows
constexpr int kCtaUnrollDeep = 8;   // the same for rows of kCtaDeepCols or more, at 4 blocks per SM
constexpr int64_t kCtaDeepCols = 16384;  // measured: deeper is 1 % faster from here, slower below
constexpr int kGroupBlock = 256; // threads per block, short rows
#ifndef RDX_GROUP_ROW_MAX_COLS
#define RDX_GROUP_ROW_MAX_COLS 5120
#endif
constexpr int64_t kGroupRowMaxCols = RDX_GROUP_ROW_MAX_COLS;  // measured: a block per row is faster from about 6144
constexpr int64_t kFitRowMaxCols = 512;  // 4 vectors x 32 lanes x 4 floats
#ifndef RDX_ROW_STEPS
#define RDX_ROW_STEPS 1
#endif
constexpr int kRowSteps = RDX_ROW_STEPS;  // row steps whose loads are in flight together
constexpr int kNarrowBlock = 256;        // threads per block, narrow rows
constexpr int kNarrowTile = 4096;        // floats staged per block (16 KiB), narrow rows
constexpr int kNarrowBulkTile = 6144;    // the same with bulk-copy staging (24 KiB: 8 blocks per SM)
constexpr int64_t kStagedMaxCols = 6000;  // widest rows the staged kernel takes (a tile holds one row at least)
constexpr int64_t kStagedMaxGap = 8;      // rows with a leading dimension: staged as one span below this gap
constexpr int64_t kRowsStagedMinCols = 1500;  // wider gaps: one bulk copy per row from this width
static_assert(kStagedMaxCols <= kNarrowBulkTile, "a staged tile must hold a whole row");
constexpr int64_t kNarrowMaxCols = 65;   // narrow rows: fewer columns than this
// Rotated reads (see rowsum_narrow_kernel) pay one shared load per VEC-float
// group of a row; measured against the short-row kernel at every 4-byte base
// offset, they win up to a whole 64-column row read one float at a time
// (64 columns 4-12 bytes off 155.7 -> 148.5-151.6 us per GiB; 56 columns,
// bulk-staged, 157.7 -> 153.6).
constexpr int kRotatedMaxGroups = 64;

// Elements of a row before its first 16-byte boundary (rows of a matrix with
// cols % 4 != 0 start at varying alignments).
__device__ __forceinline__ int64_t row_head(const float* row, int64_t cols) {
    const int64_t h = int64_t(((16u - (unsigned(reinterpret_cast<uintptr_t>(row)) & 15u)) & 15u) >> 2);
    return h < cols ? h : cols;
}

// 4-byte asynchronous copy from global to shared memory (cp.async): the value
// passes through no register, so nothing waits for it until
// cp_async_wait_all(), which waits for every copy this thread issued.
__device__ __forceinline__ void cp_async4(float* smem_dst, const float* src) {
    const unsigned d = static_cast<unsigned>(__cvta_generic_to_shared(smem_dst));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Bulk-copy staging of the narrow kernel.  Thread 0 initialises a shared-
// memory barrier, arms it for the bytes to come (plus extra, 0 except in the
// timeout test) and starts one bulk copy (the copy engine of the SM, no
// thread registers) of `bytes` bytes from global src to shared dst; both
// addresses and the size are multiples of 16 bytes.  The barrier's phase 0
// completes when every byte has landed.
__device__ __forceinline__ unsigned smem_addr(const void* p) {
    return static_cast<unsigned>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void bulk_load(float* dst, const void* src, unsigned bytes, unsigned long long* bar,
                                          unsigned extra) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(bar)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes + extra)
                 : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}

// The same barrier driven by several threads: thread 0 initialises it for
// one arrival, every thread that starts a copy first adds its bytes to the
// barrier's expected count (mbar_expect_bytes), and thread 0 arrives only
// after a block-wide barrier has ordered every addition before it, so the
// phase cannot complete before the last copy's bytes have landed.
__device__ __forceinline__ void mbar_init_one(unsigned long long* bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(bar)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_bytes(unsigned long long* bar, unsigned bytes) {
    asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(unsigned long long* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void bulk_copy(float* dst, const void* src, unsigned bytes, unsigned long long* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}

// Staging waits that gave up, counted in every build and read (and cleared)
// by the host through rowsum_stage_timeouts().
__device__ unsigned long long g_stage_timeouts;
constexpr unsigned long long kStageWaitNs = 1000000000ull;  // one second of wall time

// Wait for phase 0 of the barrier, for at most kStageWaitNs by the GPU's
// global timer: true once it has completed, false if the wait gave up.
__device__ __forceinline__ bool mbar_wait_bounded(unsigned long long* bar) {
    const unsigned a = smem_addr(bar);
    unsigned long long t0 = 0;
    for (;;) {
        unsigned done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n selp.u32 %0, 1, 0, p;\n}"
            : "=r"(done)
            : "r"(a)
            : "memory");
        if (done) return true;
        unsigned long long now;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(now));
        if (t0 == 0) t0 = now;
        else if (now - t0 > kStageWaitNs) return false;
    }
}

// Sum of lane l's share of one row, the row split among LPR lanes: the up to
// 3 + 3 floats before the first and after the last whole vector, then the
// row's 16-byte vectors l, l + LPR, ..., four in flight at a time.
template <int LPR>
__device__ __forceinline__ float row_share(const float* __restrict__ row, int64_t cols, int l) {
    const int64_t head = row_head(row, cols);
    const int64_t m = (cols - head) >> 2;
    const int64_t tail0 = head + 4 * m;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    // up to 3 scalars before the first and after the last whole vector; a
    // group may have fewer than 3 lanes, so stride by LPR
    const size_t span = size_t(cols) * 4;
    for (int64_t k = l; k < head; k += LPR)
        if (guard(row + k, 4, row, span)) acc[0] += __ldg(row + k);
    for (int64_t k = tail0 + l; k < cols; k += LPR)
        if (guard(row + k, 4, row, span)) acc[1] += __ldg(row + k);
    const uint4* __restrict__ rv = reinterpret_cast<const uint4*>(row + head);
    int64_t j = l;
    for (; j + 3 * LPR < m; j += 4 * LPR) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            v[u] = guard(rv + j + u * LPR, 16, row, span) ? ld_stream16(rv + j + u * LPR) : SumF32::neutral();
        batch_fence(v);
#pragma unroll
        for (int u = 0; u < 4; ++u) acc[u] += SumF32::fold(v[u]);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        if (j + u * LPR < m && guard(rv + j + u * LPR, 16, row, span))
            acc[u] += SumF32::fold(ld_stream16(rv + j + u * LPR));
    }
    return fold_array(acc);
}

// Short rows.  Group g of warp w (lanes g*LPR .. g*LPR+LPR-1) sums row
// (w + k * nwarps) * NG + g for k = 0, 1, ...; lane 0 of the group stores it.
// The NG rows of one warp step are consecutive, so are their sums.
template <int LPR>
__global__ void __launch_bounds__(kGroupBlock)
rowsum_group_kernel(const float* __restrict__ x, int64_t rows, int64_t cols, int64_t ld,
                    float* __restrict__ out) {
    pdl_wait();     // the previous kernel in the stream has finished writing
    pdl_release();  // the next one may be scheduled into SMs this grid frees
    constexpr int NG = kWarpSize / LPR;  // rows in flight per warp step
    const int lane = threadIdx.x % kWarpSize;
    const int grp = lane / LPR;
    const int l = lane % LPR;
    const int64_t warp = (int64_t(blockIdx.x) * kGroupBlock + threadIdx.x) / kWarpSize;
    const int64_t nwarps = int64_t(gridDim.x) * (kGroupBlock / kWarpSize);
    const int64_t nsteps = (rows + NG - 1) / NG;
    for (int64_t k = warp; k < nsteps; k += nwarps) {
        const int64_t r = k * NG + grp;
        float s = 0.f;
        if (r < rows) s = row_share<LPR>(x + r * ld, cols, l);
        s = group_allreduce<LPR>(s);  // every lane takes part, in range or not
        if (l == 0 && r < rows && guard(out + r, 4, out, size_t(rows) * 4)) out[r] = s;
    }
}

// Short rows: every row has at most 4*LPR whole vectors, so one load round
// covers it.  A warp takes units of kRowSteps*NG consecutive rows; in a unit,
// step q has group g sum row q*NG + g.  All loads of the unit are issued
// before the first reduction.  Lane 0 of each group stores its row's sum.
// The up to 3 + 3 floats of a row that is not 16-byte aligned, before its
// first and after its last whole vector, are copied to shared memory with
// cp.async ahead of the vector loads (groups of more than two lanes): a
// load into a register that is added at once would hold the warp for a
// round trip before its vector loads.  They are added after the vectors, in
// the same order as before, so the result is the same bit for bit.  Groups
// of two or more lanes are held to 32 registers (8 blocks per SM); a lane per
// row needs 37 without spilling.
template <int LPR>
__global__ void __launch_bounds__(kGroupBlock, LPR > 1 ? 2048 / kGroupBlock : 1)
rowsum_fit_kernel(const float* __restrict__ x, int64_t rows, int64_t cols, int64_t ld,
                  float* __restrict__ out) {
    pdl_wait();     // the previous kernel in the stream has finished writing
    pdl_release();  // the next one may be scheduled into SMs this grid frees
    constexpr int NG = kWarpSize / LPR;
    constexpr int RU = NG * kRowSteps;  // rows per unit
    const int lane = threadIdx.x % kWarpSize;
    const int grp = lane / LPR;
    const int l = lane % LPR;
    const int64_t warp = (int64_t(blockIdx.x) * kGroupBlock + threadIdx.x) / kWarpSize;
    const int64_t nwarps = int64_t(gridDim.x) * (kGroupBlock / kWarpSize);
    const int64_t nunits = (rows + RU - 1) / RU;
    constexpr bool kAsyncEdges = LPR > 2;
    constexpr int kPer = (3 + LPR - 1) / LPR;  // edge floats per lane on each side of a row
    __shared__ float edge[kRowSteps][2 * kPer][kAsyncEdges ? kGroupBlock : 1];  // [step][head j, tail j][thread]
    for (int64_t k = warp; k < nunits; k += nwarps) {  // one pass unless the grid is capped
        uint4 v[kRowSteps * 4];
        int nh[kRowSteps], nt[kRowSteps];  // head and tail lengths of the step's row (0-3)
        float sc[kRowSteps];               // without kAsyncEdges: the edge floats' sum
#pragma unroll
        for (int q = 0; q < kRowSteps; ++q) {
            const int64_t r = k * RU + q * NG + grp;
            nh[q] = 0;
            nt[q] = 0;
            sc[q] = 0.f;
#pragma unroll
            for (int u = 0; u < 4; ++u) v[q * 4 + u] = make_uint4(0u, 0u, 0u, 0u);
            if (r < rows) {
                const float* __restrict__ row = x + r * ld;
                const int64_t head = row_head(row, cols);
                const int64_t m = (cols - head) >> 2;
                const int64_t tail0 = head + 4 * m;
                const size_t span = size_t(cols) * 4;
                if (kAsyncEdges) {
                    nh[q] = int(head);
                    nt[q] = int(cols - tail0);
                    for (int e = l; e < nh[q]; e += LPR)
                        if (guard(row + e, 4, row, span)) cp_async4(&edge[q][e / LPR][threadIdx.x], row + e);
                    for (int e = l; e < nt[q]; e += LPR)
                        if (guard(row + tail0 + e, 4, row, span))
                            cp_async4(&edge[q][kPer + e / LPR][threadIdx.x], row + tail0 + e);
                } else {
                    // one or two lanes per row: the copies cost more registers, or
                    // more time, than the round trip (measured), so the floats are
                    // added here
                    for (int64_t e = l; e < head; e += LPR)
                        if (guard(row + e, 4, row, span)) sc[q] += __ldg(row + e);
                    for (int64_t e = tail0 + l; e < cols; e += LPR)
                        if (guard(row + e, 4, row, span)) sc[q] += __ldg(row + e);
                }
                const uint4* __restrict__ rv = reinterpret_cast<const uint4*>(row + head);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if (l + u * LPR < m && guard(rv + l + u * LPR, 16, row, span))
                        v[q * 4 + u] = ld_stream16(rv + l + u * LPR);
                }
            }
        }
        batch_fence(v);
        if (kAsyncEdges) cp_async_wait_all();
#pragma unroll
        for (int q = 0; q < kRowSteps; ++q) {
            float acc[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) acc[u] = SumF32::fold(v[q * 4 + u]);
            if (kAsyncEdges) {
                // the head floats, then the tail floats, in index order
#pragma unroll
                for (int j = 0; j < kPer; ++j)
                    if (l + j * LPR < nh[q]) sc[q] += edge[q][j][threadIdx.x];
#pragma unroll
                for (int j = 0; j < kPer; ++j)
                    if (l + j * LPR < nt[q]) sc[q] += edge[q][kPer + j][threadIdx.x];
            }
            acc[0] += sc[q];
            float s = group_allreduce<LPR>(fold_array(acc));
            const int64_t r = k * RU + q * NG + grp;
            if (l == 0 && r < rows && guard(out + r, 4, out, size_t(rows) * 4)) out[r] = s;
        }
    }
}

// Long rows: one block per row (a block loops over rows r, r + gridDim.x, ...),
// U loads of 16 bytes in flight per thread.  Very long rows stream faster with
// U = 8 at 4 blocks per SM than with U = 4 at 8: the same bytes in flight over
// half as many concurrent streams.
template <int U, int kMinBlocks>
__global__ void __launch_bounds__(kCtaBlock, kMinBlocks)
rowsum_cta_kernel(const float* __restrict__ x, int64_t rows, int64_t cols, int64_t ld, float* __restrict__ out) {
    pdl_wait();     // the previous kernel in the stream has finished writing
    pdl_release();  // the next one may be scheduled into SMs this grid frees
    __shared__ float smem[kCtaBlock / kWarpSize];
    const int t = threadIdx.x;
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const float* __restrict__ row = x + r * ld;
        const int64_t head = row_head(row, cols);
        const int64_t m = (cols - head) >> 2;
        const int64_t tail0 = head + 4 * m;
        float acc[U];
#pragma unroll
        for (int u = 0; u < U; ++u) acc[u] = 0.f;
        const size_t span = size_t(cols) * 4;
        // the row's up to 3 + 3 edge floats: loaded now, added after the
        // vectors, so that no vector load waits for their round trip
        const float eh = t < head && guard(row + t, 4, row, span) ? __ldg(row + t) : 0.f;
        const float et = t < cols - tail0 && guard(row + tail0 + t, 4, row, span) ? __ldg(row + tail0 + t) : 0.f;
        const uint4* __restrict__ rv = reinterpret_cast<const uint4*>(row + head);
        int64_t i = t;
        for (; i + (U - 1) * kCtaBlock < m; i += U * kCtaBlock) {
            uint4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u)
                v[u] = guard(rv + i + u * kCtaBlock, 16, row, span) ? ld_stream16(rv + i + u * kCtaBlock)
                                                                    : SumF32::neutral();
            batch_fence(v);
#pragma unroll
            for (int u = 0; u < U; ++u) acc[u] += SumF32::fold(v[u]);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (i + u * kCtaBlock < m && guard(rv + i + u * kCtaBlock, 16, row, span))
                acc[u] += SumF32::fold(ld_stream16(rv + i + u * kCtaBlock));
        }
        if (t < head) acc[0] += eh;
        if (t < cols - tail0) acc[U - 1] += et;
        const float a = block_sum<kCtaBlock>(fold_array(acc), smem, 0.f);
        if (t == 0 && guard(out + r, 4, out, size_t(rows) * 4)) out[r] = a;
        __syncthreads();  // smem is reused by the next row
    }
}

// Stage rows [r0, r0 + nr) of the (rows, cols) matrix x whose rows start
// every ld floats, as the one span from the first float of row r0 to the
// last of row r0 + nr - 1 (at most kTile floats; the gaps between rows come
// along), in the block's shared array tile: span float i lands at
// tile[s + i], s = (4 - h) mod 4 with h
// the floats before the first 16-byte boundary, so that the 16-byte body
// lands on 16-byte boundaries.  BULK: thread 0 starts one bulk copy of the
// body, tracked by a shared-memory barrier (armed for extra_tx more bytes: 0
// except in the timeout test, where nothing then completes it); otherwise
// every thread loads its 16-byte vectors, all in flight together, and stores
// them.  The up to 3 + 3 floats outside the body are plain loads.  Returns
// with the tile complete and the block synchronised, or false if the bulk
// copy's bounded wait gave up: the timeout is counted, the copy is given a
// second bounded wait to land before the block's shared memory is released,
// and the block must then write nothing.
template <int kTile, bool BULK>
__device__ __forceinline__ bool stage_rows(const float* __restrict__ x, int64_t rows, int64_t cols, int64_t ld,
                                           int64_t r0, int nr, float* tile, int& s, unsigned extra_tx) {
    const int t = threadIdx.x;
    const int len = (nr - 1) * int(ld) + int(cols);  // floats of this tile's span, <= kTile
    const float* __restrict__ p0 = x + r0 * ld;
    const size_t span = (size_t(rows - 1) * size_t(ld) + size_t(cols)) * 4;
    int h = int(((16u - (unsigned(reinterpret_cast<uintptr_t>(p0)) & 15u)) & 15u) >> 2);
    if (h > len) h = len;
    const int m = (len - h) >> 2;                     // whole 16-byte vectors
    const int tail0 = h + 4 * m;
    s = -h & 3;
    const uint4* __restrict__ pv = reinterpret_cast<const uint4*>(p0 + h);
    if (BULK) {
        __shared__ __align__(8) unsigned long long bar;
        __shared__ int staged;
        if (t == 0) {
            staged = m > 0 && guard(pv, size_t(m) * 16, x, span);
            if (staged) bulk_load(tile + s + h, pv, unsigned(m) * 16u, &bar, extra_tx);
        }
        if (t < h && guard(p0 + t, 4, x, span)) tile[s + t] = __ldg(p0 + t);
        if (t < len - tail0 && guard(p0 + tail0 + t, 4, x, span)) tile[s + tail0 + t] = __ldg(p0 + tail0 + t);
        __syncthreads();  // the barrier is armed, the edge floats are stored
        if (staged && !mbar_wait_bounded(&bar)) {
            if (t == 0) atomicAdd(&g_stage_timeouts, 1ull);
            (void)mbar_wait_bounded(&bar);
            return false;
        }
    } else {
        constexpr int kLoads = kTile / 4 / kNarrowBlock;  // vectors per thread, all in flight
        uint4 v[kLoads];
#pragma unroll
        for (int u = 0; u < kLoads; ++u) {
            const int k = t + u * kNarrowBlock;
            v[u] = k < m && guard(pv + k, 16, x, span) ? ld_stream16(pv + k) : make_uint4(0u, 0u, 0u, 0u);
        }
        batch_fence(v);
#pragma unroll
        for (int u = 0; u < kLoads; ++u) {
            const int k = t + u * kNarrowBlock;
            if (k < m) *reinterpret_cast<uint4*>(tile + s + h + 4 * k) = v[u];
        }
        if (t < h && guard(p0 + t, 4, x, span)) tile[s + t] = __ldg(p0 + t);
        if (t < len - tail0 && guard(p0 + tail0 + t, 4, x, span)) tile[s + tail0 + t] = __ldg(p0 + tail0 + t);
        __syncthreads();
    }
    return true;
}

// Narrow rows of a contiguous matrix (ld == cols).  The matrix is read as
// one flat array cut into tiles of whole rows, at most kNarrowTile floats
// each, one tile per block.  The block stages its tile in shared memory
// (16-byte loads of the flat array, all in flight together; scalars for the
// few floats before the tile's first 16-byte boundary and after its last),
// then thread t sums rows t, t + kNarrowBlock, ... of the tile and stores
// them (consecutive threads, consecutive rows).
//
// Rows are read from shared memory VEC floats at a time (VEC = 1, 2 or 4,
// chosen by the launcher so that every row starts on a VEC-float boundary),
// so a row's sum is VEC chains of every VEC-th term, added at the end (two
// chains of alternate terms for VEC = 1).  Rows start every cols words:
// with VEC = 1 for odd cols, VEC = 2 for cols = 2 (mod 4) and VEC = 4 for
// cols = 4 (mod 8), a warp's reads meet no bank conflict.  Where rows that
// start cols words apart would share banks (cols with a large power of two,
// read 1 or 2 floats at a time: rows that are not 16-byte aligned), ROT
// rotates each lane's reads: lane l starts its row at VEC-float group
// l mod (cols / VEC) and wraps around, so the 32 lanes of a step read
// different columns.  The launcher (rowsum_narrow_read) takes this kernel
// only where the reads share a bank at most 2 ways (4 ways for 8 columns or
// fewer), and rotated reads only up to kRotatedMaxGroups loads per row.  The order depends only on cols, VEC, ROT and, with ROT, the row's
// lane (its index modulo 32).
//
// AD (rows not 16-byte aligned whose starts are 4 words apart modulo 8, or
// 8 words apart; see rowsum_narrow_read): each row is read as the 16-byte
// groups of shared memory that cover it, aligned down from its first word,
// with the words of the first and last group that belong to the neighbouring
// rows zeroed; four chains, one per word of a group.  Rows 4 (mod 8) words
// apart put consecutive lanes' groups in alternate halves of the banks, so
// these wide reads meet no conflict, and a row costs cols / 4 + 1 reads
// instead of cols.  The order depends on cols and the row's word offset in
// shared memory (its start modulo 4).
template <int VEC, bool ROT, bool AD, bool BULK>
__global__ void __launch_bounds__(kNarrowBlock)
rowsum_narrow_kernel(const float* __restrict__ x, int64_t rows, int64_t cols, int64_t rows_per_tile,
                     float* __restrict__ out, unsigned extra_tx) {
    pdl_wait();     // the previous kernel in the stream has finished writing
    pdl_release();  // the next one may be scheduled into SMs this grid frees
    constexpr int kTile = BULK ? kNarrowBulkTile : kNarrowTile;
    __shared__ __align__(16) float tile[kTile + 4];
    const int t = threadIdx.x;
    const int ci = int(cols);
    const int64_t r0 = int64_t(blockIdx.x) * rows_per_tile;
    const int nr = int(rows - r0 < rows_per_tile ? rows - r0 : rows_per_tile);
    int s;                                            // tile float i lives at tile[s + i]
    if (!stage_rows<kTile, BULK>(x, rows, cols, cols, r0, nr, tile, s, extra_tx)) return;

    for (int q = t; q < nr; q += kNarrowBlock) {
        const float* row = tile + s + q * ci;
        float sum;
        if (AD) {
            // words [o, o + ci) of the 16-byte groups starting at the row's
            // first word rounded down to a group; the last group ends at most
            // at word kTile + 4 of the tile (its staged data end at or before
            // word kTile + 3), and the words past the row, staged or not, are
            // zeroed
            const int start = s + q * ci;
            const int o = start & 3;
            const float4* g = reinterpret_cast<const float4*>(tile + (start - o));
            const int end = o + ci;
            const int ng = (end + 3) >> 2;
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int j = 0; j < ng; ++j) {
                float4 e = g[j];
                const int w0 = 4 * j;
                if (w0 + 0 < o || w0 + 0 >= end) e.x = 0.f;
                if (w0 + 1 < o || w0 + 1 >= end) e.y = 0.f;
                if (w0 + 2 < o || w0 + 2 >= end) e.z = 0.f;
                if (w0 + 3 < o || w0 + 3 >= end) e.w = 0.f;
                a.x += e.x; a.y += e.y; a.z += e.z; a.w += e.w;
            }
            sum = (a.x + a.y) + (a.z + a.w);
        } else if (ROT) {
            // VEC-float groups k0, k0 + 1, ..., wrapping at the row's end
            constexpr int kLanes = kWarpSize;
            const int w = ci / VEC;
            int k = (t % kLanes) % w;
            if (VEC == 2) {
                float2 a = make_float2(0.f, 0.f);
                for (int j = 0; j < w; ++j) {
                    const float2 e = *reinterpret_cast<const float2*>(row + 2 * k);
                    a.x += e.x; a.y += e.y;
                    k = k + 1 == w ? 0 : k + 1;
                }
                sum = a.x + a.y;
            } else {
                float a0 = 0.f, a1 = 0.f;
                int j = 0;
                for (; j + 1 < w; j += 2) {
                    a0 += row[k];
                    k = k + 1 == w ? 0 : k + 1;
                    a1 += row[k];
                    k = k + 1 == w ? 0 : k + 1;
                }
                if (j < w) a0 += row[k];
                sum = a0 + a1;
            }
        } else if (VEC == 4) {
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int j = 0; j < ci; j += 4) {
                const float4 e = *reinterpret_cast<const float4*>(row + j);
                a.x += e.x; a.y += e.y; a.z += e.z; a.w += e.w;
            }
            sum = (a.x + a.y) + (a.z + a.w);
        } else if (VEC == 2) {
            float2 a = make_float2(0.f, 0.f);
            for (int j = 0; j < ci; j += 2) {
                const float2 e = *reinterpret_cast<const float2*>(row + j);
                a.x += e.x; a.y += e.y;
            }
            sum = a.x + a.y;
        } else {
            float a0 = 0.f, a1 = 0.f;
            int j = 0;
            for (; j + 1 < ci; j += 2) {
                a0 += row[j];
                a1 += row[j + 1];
            }
            if (j < ci) a0 += row[j];
            sum = a0 + a1;
        }
        if (guard(out + r0 + q, 4, out, size_t(rows) * 4)) out[r0 + q] = sum;
    }
}

// Staged rows (see rowsum_staged_lanes: short rows that the short-row kernel
// would leave with half-empty load slots, and medium rows up to
// kStagedMaxCols, contiguous or with gaps under kStagedMaxGap floats between
// them): the span of a tile's rows, gaps included, is staged as in the
// narrow kernel by one bulk copy (at most 24 KiB, 8 blocks per SM, so the
// bytes in flight do not depend on the width), and row q is read at word
// q * ld of it by a group of LW lanes: lane l adds words l, l + LW, ... of
// the row in two alternating chains, the group's shuffle tree adds the
// lanes, and its first lane stores the sum.  A group reads consecutive
// words; the 32 / LW groups of a warp read rows ld words apart, which the
// launcher keeps to at most 2 ways of bank sharing.  The order depends on
// cols and LW only.
template <int LW>
__global__ void __launch_bounds__(kNarrowBlock)
rowsum_staged_kernel(const float* __restrict__ x, int64_t rows, int64_t cols, int64_t ld, int64_t rows_per_tile,
                     float* __restrict__ out) {
    pdl_wait();     // the previous kernel in the stream has finished writing
    pdl_release();  // the next one may be scheduled into SMs this grid frees
    __shared__ __align__(16) float tile[kNarrowBulkTile + 4];
    const int ci = int(cols);
    const int64_t r0 = int64_t(blockIdx.x) * rows_per_tile;
    const int nr = int(rows - r0 < rows_per_tile ? rows - r0 : rows_per_tile);
    int s;
    if (!stage_rows<kNarrowBulkTile, true>(x, rows, cols, ld, r0, nr, tile, s, 0u)) return;
    constexpr int kGroups = kWarpSize / LW;           // rows per warp step
    const int warp = threadIdx.x / kWarpSize, lane = threadIdx.x % kWarpSize;
    const int g = lane / LW, l = lane % LW;
    // the loop bound is the same for every lane of a warp, so the shuffle
    // tree always has the whole warp
    for (int qb = warp * kGroups; qb < nr; qb += (kNarrowBlock / kWarpSize) * kGroups) {
        const int q = qb + g;
        float a0 = 0.f, a1 = 0.f;
        if (q < nr) {
            const float* row = tile + s + q * int(ld);
            int j = l;
            for (; j + LW < ci; j += 2 * LW) {
                a0 += row[j];
                a1 += row[j + LW];
            }
            if (j < ci) a0 += row[j];
        }
        const float v = group_allreduce<LW>(a0 + a1);
        if (l == 0 && q < nr && guard(out + r0 + q, 4, out, size_t(rows) * 4)) out[r0 + q] = v;
    }
}

// Rows with a leading dimension whose gap to the next row is kStagedMaxGap
// floats or more (copying their span would read sectors without row data),
// from kRowsStagedMinCols columns: the rows of a tile are staged one bulk
// copy per row, each row's 16-byte body into a slot of W words (a multiple
// of 4 with 4 spare words in front), its up to 3 + 3 edge floats by plain
// loads, so
// that row q's words occupy [q W + 4 - h, q W + 4 - h + cols) with h the
// row's floats before its first 16-byte boundary.  W is padded so that the
// kGroups rows a warp reads at once start LW words apart modulo 32: the
// groups read disjoint banks.  Rows are then summed as in
// rowsum_staged_kernel (groups of LW lanes, two alternating chains per lane,
// the group's shuffle tree), so a row's sum has the same bits either way.
template <int LW>
__global__ void __launch_bounds__(kNarrowBlock)
rowsum_rows_staged_kernel(const float* __restrict__ x, int64_t rows, int64_t cols, int64_t ld, int64_t slot,
                          int64_t rows_per_tile, float* __restrict__ out) {
    pdl_wait();     // the previous kernel in the stream has finished writing
    pdl_release();  // the next one may be scheduled into SMs this grid frees
    __shared__ __align__(16) float tile[kNarrowBulkTile];
    __shared__ __align__(8) unsigned long long bar;
    const int t = threadIdx.x;
    const int ci = int(cols), w = int(slot);
    const int64_t r0 = int64_t(blockIdx.x) * rows_per_tile;
    const int nr = int(rows - r0 < rows_per_tile ? rows - r0 : rows_per_tile);
    const size_t span = (size_t(rows - 1) * size_t(ld) + size_t(cols)) * 4;
    if (t == 0) mbar_init_one(&bar);
    __syncthreads();  // the barrier is initialised
    for (int q = t; q < nr; q += kNarrowBlock) {
        const float* __restrict__ row = x + (r0 + q) * ld;
        const int h = int(row_head(row, cols));
        const int m = (ci - h) >> 2;
        const int tail0 = h + 4 * m;
        float* dst = tile + q * w + 4;
        if (m > 0 && guard(row + h, size_t(m) * 16, x, span)) {
            mbar_expect_bytes(&bar, unsigned(m) * 16u);
            bulk_copy(dst, row + h, unsigned(m) * 16u, &bar);
        }
        for (int e = 0; e < h; ++e)
            if (guard(row + e, 4, x, span)) dst[e - h] = __ldg(row + e);
        for (int e = tail0; e < ci; ++e)
            if (guard(row + e, 4, x, span)) dst[e - h] = __ldg(row + e);
    }
    __syncthreads();  // every expected byte count is in, the edge floats are stored
    if (t == 0) mbar_arrive(&bar);
    if (!mbar_wait_bounded(&bar)) {
        if (t == 0) atomicAdd(&g_stage_timeouts, 1ull);
        (void)mbar_wait_bounded(&bar);
        return;
    }
    constexpr int kGroups = kWarpSize / LW;
    const int warp = t / kWarpSize, lane = t % kWarpSize;
    const int g = lane / LW, l = lane % LW;
    for (int qb = warp * kGroups; qb < nr; qb += (kNarrowBlock / kWarpSize) * kGroups) {
        const int q = qb + g;
        float a0 = 0.f, a1 = 0.f;
        if (q < nr) {
            const float* row = tile + q * w + 4 - int(row_head(x + (r0 + q) * ld, cols));
            int j = l;
            for (; j + LW < ci; j += 2 * LW) {
                a0 += row[j];
                a1 += row[j + LW];
            }
            if (j < ci) a0 += row[j];
        }
        const float v = group_allreduce<LW>(a0 + a1);
        if (l == 0 && q < nr && guard(out + r0 + q, 4, out, size_t(rows) * 4)) out[r0 + q] = v;
    }
}

// Short rows whose power-of-two lane groups would run half empty and that the
// staged kernels do not take (rows with wide gaps between them): groups of G
// lanes (G = ceil(vecs / 4), not a power of two), 32 / G rows per warp step,
// the lanes past the last whole group idle; otherwise as rowsum_fit_kernel
// (at most four 16-byte vectors per lane in one load round, the edge floats
// copied with cp.async ahead of the vector loads and added after them).  The
// group's lanes are added by a shuffle-down tree in which lane l takes lane
// l + off only while l + off < G, so lane 0 of each group ends with the sum
// of its G lanes, in an order fixed by G.
template <int G>
__global__ void __launch_bounds__(kGroupBlock, 2048 / kGroupBlock)
rowsum_fitg_kernel(const float* __restrict__ x, int64_t rows, int64_t cols, int64_t ld,
                   float* __restrict__ out) {
    pdl_wait();     // the previous kernel in the stream has finished writing
    pdl_release();  // the next one may be scheduled into SMs this grid frees
    constexpr int NG = kWarpSize / G;
    const int lane = threadIdx.x % kWarpSize;
    const int grp = lane / G;
    const int l = lane % G;
    // one unit of NG rows per warp: the launcher sizes the grid to cover them
    const int64_t k = (int64_t(blockIdx.x) * kGroupBlock + threadIdx.x) / kWarpSize;
    __shared__ float edge[2][kGroupBlock];  // [head, tail][thread]
    {
        uint4 v[4];
        int nh = 0, nt = 0;
        float sc = 0.f;
        const int64_t r = k * NG + grp;
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = make_uint4(0u, 0u, 0u, 0u);
        if (grp < NG && r < rows) {
            const float* __restrict__ row = x + r * ld;
            const int64_t head = row_head(row, cols);
            const int64_t m = (cols - head) >> 2;
            const int64_t tail0 = head + 4 * m;
            const size_t span = size_t(cols) * 4;
            nh = int(head);
            nt = int(cols - tail0);
            for (int e = l; e < nh; e += G)
                if (guard(row + e, 4, row, span)) cp_async4(&edge[0][threadIdx.x], row + e);
            for (int e = l; e < nt; e += G)
                if (guard(row + tail0 + e, 4, row, span)) cp_async4(&edge[1][threadIdx.x], row + tail0 + e);
            const uint4* __restrict__ rv = reinterpret_cast<const uint4*>(row + head);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (l + u * G < m && guard(rv + l + u * G, 16, row, span)) v[u] = ld_stream16(rv + l + u * G);
            }
        }
        batch_fence(v);
        cp_async_wait_all();
        float acc[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) acc[u] = SumF32::fold(v[u]);
        if (l < nh) sc += edge[0][threadIdx.x];  // the head float, then the tail float
        if (l < nt) sc += edge[1][threadIdx.x];
        acc[0] += sc;
        float s = fold_array(acc);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float o = __shfl_down_sync(kFullMask, s, off);
            if (l + off < G) s += o;
        }
        if (l == 0 && grp < NG && r < rows && guard(out + r, 4, out, size_t(rows) * 4)) out[r] = s;
    }
}

// Lanes per row: the fewest (a power of two, at most 32) that leave each lane
// at most four 16-byte vectors of the row.
int lanes_per_row(int64_t cols) {
    const int64_t vecs = cols / 4;
    int lpr = 1;
    while (lpr < 32 && int64_t(lpr) * 4 < vecs) lpr *= 2;
    return lpr;
}

// Lanes per row of the staged kernel for the contiguous (rows, cols) matrix
// at x, or 0 where the short-row kernel keeps the rows.  That kernel gives a
// row the fewest lanes, a power of two, that leave each lane at most four
// 16-byte vectors, so a row just past a power of two fills about half of
// its lanes' load slots (68 columns: 17 vectors in 8 lanes x 4), keeps half
// the bytes in flight and reads well below the bandwidth (measured, 1 GiB:
// 68 columns 4 bytes off 202.8 us, 132 columns 210.9, 260 columns 200.7,
// against 145-150 us for rows that fill their slots).  The staged kernel
// holds 147-155 us at the widths it takes, so it takes the rows whose slots
// the short-row kernel would fill less than 60 % (16-byte aligned rows,
// which that kernel reads faster at equal fill) or 75 % (rows not all
// aligned; 80 % from 257 columns, where the staged kernel's groups of 32
// lanes still win at 78-80 %); measured over 65-512 columns at 0 and 4
// bytes off.  Groups of 8 lanes below 96 columns, 16 below 256, 32 above
// (the fastest in the same sweep); a warp's groups of 8 read 4 rows at once,
// cols words apart, and where they would share a bank more than 2 ways
// (93-95 columns) the short-row kernel keeps the rows.  Contiguous rows of
// 513 to kStagedMaxCols columns take it with groups of 32 lanes at every
// width and alignment: measured faster or equal against the warp-per-row
// and block-per-row kernels over 513-6144 columns at 0, 4 and 8 bytes off
// (1 GiB: 516 columns 4-8 bytes off 159.8-161.8 -> 149.5 us, 600 columns
// 157.7 -> 149.5, 1500 columns 155.7 -> 147.5, 5200 columns 156.7 -> 147.5;
// 1024 columns aligned and 6144 columns 4 bytes off one timer tick slower,
// 6000 columns equal).
static int staged_group_bank_ways(int64_t cols, int lw) {
    int count[kWarpSize] = {};
    for (int g = 0; g < kWarpSize / lw; ++g)
        for (int l = 0; l < lw; ++l) ++count[(g * cols + l) % kWarpSize];
    int worst = 0;
    for (int b = 0; b < kWarpSize; ++b) worst = worst > count[b] ? worst : count[b];
    return worst;
}

static int rowsum_staged_lanes(const float* x, int64_t cols, int64_t ld) {
    if (ld - cols >= kStagedMaxGap || cols < kNarrowMaxCols || cols > kStagedMaxCols) return 0;
    if (cols > kFitRowMaxCols) return 32;
    const int lpr = lanes_per_row(cols);
    const int64_t vecs = cols / 4, slots = 4 * int64_t(lpr);
    const bool aligned = cols % 4 == 0 && ld % 4 == 0 && reinterpret_cast<uintptr_t>(x) % 16 == 0;
    const bool sparse = aligned ? 10 * vecs < 6 * slots : lpr == 32 ? 10 * vecs < 8 * slots : 4 * vecs < 3 * slots;
    if (!sparse) return 0;
    const int lw = cols < 96 ? 8 : cols < 256 ? 16 : 32;
    if (lw == 8 && staged_group_bank_ways(ld, 8) > 2) return 0;
    return lw;
}

// Row slot of rowsum_rows_staged_kernel for rows of cols floats read by
// groups of lw lanes: at least cols + 4 words, a multiple of 4, and for
// groups of 8 or 16 an odd multiple of lw modulo 32, so that the 32 / lw
// rows a warp reads at once start in different banks.
static int64_t rows_staged_slot(int64_t cols, int lw) {
    int64_t w = (cols + 4 + 3) / 4 * 4;
    if (lw < kWarpSize)
        while ((w / lw) % 2 == 0 || w % lw != 0) w += 4;
    return w;
}

// Lanes per row of rowsum_rows_staged_kernel, or 0 where other kernels take
// the rows: rows with gaps of kStagedMaxGap floats or more between them, of
// kRowsStagedMinCols to kStagedMaxCols columns (measured with gaps of 16
// floats, 1 GiB spans: 1500-5000 columns 152-156 -> 147-150 us; below 1500
// columns the per-row copies cost more than they save, 600 columns 154 ->
// 170 us, 68 columns 197 -> 265).
static int rowsum_rows_staged_lanes(const float*, int64_t cols, int64_t ld) {
    return ld - cols >= kStagedMaxGap && cols >= kRowsStagedMinCols && cols <= kStagedMaxCols ? 32 : 0;
}

// Lanes per row of rowsum_fitg_kernel, or 0 where the power-of-two groups
// of rowsum_fit_kernel stay: rows that no staged kernel takes (see the
// launcher) and whose power-of-two groups would fill their warp's load slots
// at least a tenth less than groups of ceil(vecs / 4) lanes do (68-99 and
// 132-163 columns, groups of 5, 6, 9 or 10 lanes: 68 columns 53 % against
// 80 %, 160 columns 62 % against 94 %).
static int rowsum_fitg_lanes(int64_t cols) {
    if (cols < kNarrowMaxCols || cols > kFitRowMaxCols) return 0;
    const int64_t vecs = cols / 4;
    const int lpr = lanes_per_row(cols);
    const int g = int((vecs + 3) / 4);
    if (g != 5 && g != 6 && g != 9 && g != 10) return 0;  // the sizes the rule below can pick
    // slots used per warp, over 128: vecs * (32 / lpr) for power-of-two
    // groups, vecs * (32 / g) for groups of g; compare in integers
    const int64_t pow2 = vecs * (kWarpSize / lpr), any = vecs * (kWarpSize / g);
    return 10 * (any - pow2) >= 128 ? g : 0;
}

template <int LPR>
cudaError_t launch_fit(const float* x, int64_t rows, int64_t cols, int64_t ld, float* out, cudaStream_t stream) {
    constexpr int64_t kRU = (kWarpSize / LPR) * kRowSteps;
    constexpr int64_t kWarpsPerBlock = kGroupBlock / kWarpSize;
    const int64_t nunits = (rows + kRU - 1) / kRU;
    // one unit per warp: many short blocks that the hardware hands to SMs as
    // they free up (measured faster than a capped grid looping over units)
    int64_t blocks = (nunits + kWarpsPerBlock - 1) / kWarpsPerBlock;
    if (blocks > 0x7fffffff) blocks = 0x7fffffff;
    return launch_pdl(rowsum_fit_kernel<LPR>, dim3(unsigned(blocks)), dim3(kGroupBlock), stream, x, rows, cols, ld, out);
}

template <int LPR>
cudaError_t launch_group(const float* x, int64_t rows, int64_t cols, int64_t ld, float* out, cudaStream_t stream) {
    constexpr int64_t kNG = kWarpSize / LPR;
    constexpr int64_t kWarpsPerBlock = kGroupBlock / kWarpSize;
    const int64_t nsteps = (rows + kNG - 1) / kNG;
    int64_t blocks = (nsteps + kWarpsPerBlock - 1) / kWarpsPerBlock;
    // one step per warp, as in launch_fit
    if (blocks > 0x7fffffff) blocks = 0x7fffffff;
    return launch_pdl(rowsum_group_kernel<LPR>, dim3(unsigned(blocks)), dim3(kGroupBlock), stream, x, rows, cols, ld,
                      out);
}

}  // namespace

RDX_DEFINE_VIOLATION_COUNTER(rowsum_out_of_range)

unsigned long long rowsum_stage_timeouts(bool reset) {
    unsigned long long v = 0;
    if (cudaMemcpyFromSymbol(&v, g_stage_timeouts, sizeof v) != cudaSuccess) return ~0ull;
    if (reset) {
        const unsigned long long z = 0;
        if (cudaMemcpyToSymbol(g_stage_timeouts, &z, sizeof z) != cudaSuccess) return ~0ull;
    }
    return v;
}

cudaError_t rowsum_stage_timeout_probe(const float* x, int64_t rows, int64_t cols, float* out, cudaStream_t stream) {
    if (cols <= 0 || cols >= kNarrowMaxCols || rows <= 0 || rows > kNarrowBulkTile || rows * cols > kNarrowBulkTile)
        return cudaErrorInvalidValue;
    // one tile; its barrier is armed for 16 bytes more than the copy brings
    return launch_pdl(rowsum_narrow_kernel<1, false, false, true>, dim3(1), dim3(kNarrowBlock), stream, x, rows, cols,
                      rows, out, 16u);
}

bool rowsum_use_split(int64_t rows, int64_t cols) {
    // At most kMaxSplitRows rows (fewer than two waves of one block per row
    // on a 152-SM GPU), each long enough for at least four tiles.  The rule
    // uses no device property, so a call sums in the same order on any GPU.
    return rows <= kMaxSplitRows && cols >= 16384;
}

// Worst shared-memory bank sharing of the narrow kernel's row reads.  The 32
// lanes of a warp sum rows that start cols words apart, VEC words at a time;
// in step j lane l reads VEC-word group j of its row, or (rotated) group
// (j + l) mod (cols / VEC).  The figure is the most words one bank serves in
// any step, over VEC (a VEC-word read takes VEC banks per lane), rounded up.
static int narrow_bank_ways(int cols, int vec, bool rotated) {
    const int w = cols / vec;
    int worst = 0;
    for (int j = 0; j < w; ++j) {
        int count[kWarpSize] = {};
        for (int lane = 0; lane < kWarpSize; ++lane) {
            const int k = rotated ? (j + lane) % w : j;
            for (int e = 0; e < vec; ++e) ++count[(lane * cols + k * vec + e) % kWarpSize];
        }
        for (int b = 0; b < kWarpSize; ++b) worst = worst > (count[b] + vec - 1) / vec ? worst : (count[b] + vec - 1) / vec;
    }
    return worst;
}

// The same figure for the aligned-down reads (AD): lane l's row starts at
// word s0 + l * cols of the tile (s0 = the tile's staging offset, the same
// for every row when cols % 4 == 0), and in step j the lane reads 16-byte
// group j counted from the one holding that word, while its row has one.
static int narrow_ad_ways(int cols, int s0) {
    int worst = 0;
    for (int j = 0; j <= (3 + cols + 3) / 4; ++j) {
        int count[kWarpSize] = {};
        for (int lane = 0; lane < kWarpSize; ++lane) {
            const int start = s0 + lane * cols, o = start & 3;
            if (j >= (o + cols + 3) / 4) continue;
            const int g = (start - o) / 4 + j;
            for (int e = 0; e < 4; ++e) ++count[(4 * g + e) % kWarpSize];
        }
        for (int b = 0; b < kWarpSize; ++b) worst = worst > (count[b] + 3) / 4 ? worst : (count[b] + 3) / 4;
    }
    return worst;
}

// narrow_bank_ways and narrow_ad_ways for every narrow width, read width and
// staging offset, worked out once.
struct NarrowWays {
    unsigned char ways[kNarrowMaxCols][3][2] = {};  // [cols][vec 1, 2, 4 -> 0, 1, 2][rotated]
    unsigned char ad[kNarrowMaxCols][4] = {};       // [cols][s0], cols % 4 == 0
    NarrowWays() {
        for (int c = 1; c < kNarrowMaxCols; ++c) {
            for (int vi = 0; vi < 3; ++vi) {
                const int vec = 1 << vi;
                if (c % vec) continue;
                for (int r = 0; r < 2; ++r) ways[c][vi][r] = static_cast<unsigned char>(narrow_bank_ways(c, vec, r != 0));
            }
            if (c % 4 == 0)
                for (int s0 = 0; s0 < 4; ++s0) ad[c][s0] = static_cast<unsigned char>(narrow_ad_ways(c, s0));
        }
    }
};
static const NarrowWays& narrow_ways() {
    static const NarrowWays table;
    return table;
}

// Shared-memory read width of the narrow kernel.  Rows start every cols
// words after the tile's staging offset s = (4 - h) % 4, h the floats before
// the tile's first 16-byte boundary.  Every tile starts a whole number of
// rows (cols floats each) after x, so h, s and every row start are even (or
// multiples of 4) exactly when cols and x's alignment allow it.
static int narrow_vec(const float* x, int64_t cols) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(x);
    if (cols % 4 == 0 && a % 16 == 0) return 4;
    if (cols % 2 == 0 && a % 8 == 0) return 2;
    return 1;
}

// How the narrow kernel reads the rows of a (rows, cols) matrix at x, if it
// takes them at all.
enum class NarrowRead { kNo, kPlain, kRotated, kAlignedDown };

static NarrowRead rowsum_narrow_read(const float* x, int64_t cols, int64_t ld) {
    if (ld != cols || cols <= 0 || cols >= kNarrowMaxCols) return NarrowRead::kNo;
    const int vec = narrow_vec(x, cols);
    // 16-byte aligned rows of 16, 24, ... columns: the short-row kernel reads
    // them as whole vectors and is faster
    if (vec == 4 && cols % 8 == 0 && cols > 8) return NarrowRead::kNo;
    const NarrowWays& table = narrow_ways();
    const int vi = vec == 1 ? 0 : vec == 2 ? 1 : 2;
    // measured: at most 2-way always gains; up to 4-way only for 8 columns or fewer
    const int limit = cols <= 8 ? 4 : 2;
    // measured over 48-64 columns at every base offset (1 GiB each): for
    // 60 columns off 16-byte alignment the short-row kernel is faster (155.7
    // against 159.7 us); rows of width 2 (mod 4) from 50 columns up read one
    // float at a time take the narrow kernel, bulk-staged (50 columns 4 bytes
    // off 159.7 -> 154.7 us, 54 columns 157.7 -> 153.6, 58 columns 155.7 ->
    // 153.6, 62 columns a tie)
    if (vec < 4 && cols == 60) return NarrowRead::kNo;
    NarrowRead read = NarrowRead::kNo;
    if (table.ways[cols][vi][0] <= limit) read = NarrowRead::kPlain;
    else if (cols / vec <= kRotatedMaxGroups && table.ways[cols][vi][1] <= limit) read = NarrowRead::kRotated;
    // rows not 16-byte aligned, 8 or 4 (mod 8) words apart from 12 up: 16-byte
    // reads aligned down around each row (measured, 1 GiB: 8 columns 4 bytes
    // off 210.9 -> 204.8 us, 12 columns 176.1 -> 170.0, 28 columns 12 bytes
    // off 168.0 -> 157.7, 52 columns 8 bytes off 163.8 -> 157.7; slower at
    // other widths, where the wide reads meet bank conflicts)
    if (read != NarrowRead::kNo && vec < 4 && (cols == 8 || (cols % 8 == 4 && cols >= 12)))
        read = NarrowRead::kAlignedDown;
    return read;
}

// How many ways the chosen reads share a shared-memory bank (1 = no
// conflict).  Where they share 2 or more, the kernel stages its tiles with
// one bulk copy instead of per-thread loads (measured over every narrow
// width at every 4-byte base offset, 1 GiB each: 4 columns 4 bytes off
// 231 -> 186 us, 8 columns 4-12 bytes off 205 -> 170, even widths 4 or 12
// bytes off 4-14 us faster, 2-way rotated reads 1-14 us; where the reads do
// not conflict, per-thread loads are 2-10 us faster and stay).
static int narrow_read_ways(const float* x, int64_t cols, NarrowRead nr) {
    const NarrowWays& table = narrow_ways();
    const int vec = narrow_vec(x, cols);
    const int vi = vec == 1 ? 0 : vec == 2 ? 1 : 2;
    switch (nr) {
        case NarrowRead::kPlain: return table.ways[cols][vi][0];
        case NarrowRead::kRotated: return table.ways[cols][vi][1];
        case NarrowRead::kAlignedDown:
            return table.ad[cols][(reinterpret_cast<uintptr_t>(x) / 4) % 4];
        default: return 0;
    }
}

bool rowsum_use_narrow(const float* x, int64_t cols, int64_t ld) {
    return rowsum_narrow_read(x, cols, ld) != NarrowRead::kNo;
}

cudaError_t rowsum_launch(const float* x, int64_t rows, int64_t cols, int64_t ld, float* out, cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    const NarrowRead nr = rowsum_narrow_read(x, cols, ld);
    if (nr != NarrowRead::kNo) {
        const bool bulk = narrow_read_ways(x, cols, nr) >= 2;
        const int64_t rpt = (bulk ? kNarrowBulkTile : kNarrowTile) / cols;  // whole rows per tile
        const int64_t blocks = (rows + rpt - 1) / rpt;
        if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
        const dim3 grid{unsigned(blocks)}, block{unsigned(kNarrowBlock)};
        const bool rot = nr == NarrowRead::kRotated;
        const int vec = narrow_vec(x, cols);
        if (bulk) {
            if (nr == NarrowRead::kAlignedDown)
                return launch_pdl(rowsum_narrow_kernel<1, false, true, true>, grid, block, stream, x, rows, cols, rpt,
                                  out, 0u);
            if (vec == 4)
                return launch_pdl(rowsum_narrow_kernel<4, false, false, true>, grid, block, stream, x, rows, cols, rpt,
                                  out, 0u);
            if (vec == 2)
                return rot ? launch_pdl(rowsum_narrow_kernel<2, true, false, true>, grid, block, stream, x, rows, cols,
                                        rpt, out, 0u)
                           : launch_pdl(rowsum_narrow_kernel<2, false, false, true>, grid, block, stream, x, rows, cols,
                                        rpt, out, 0u);
            return rot ? launch_pdl(rowsum_narrow_kernel<1, true, false, true>, grid, block, stream, x, rows, cols, rpt,
                                    out, 0u)
                       : launch_pdl(rowsum_narrow_kernel<1, false, false, true>, grid, block, stream, x, rows, cols, rpt,
                                    out, 0u);
        }
        if (nr == NarrowRead::kAlignedDown)
            return launch_pdl(rowsum_narrow_kernel<1, false, true, false>, grid, block, stream, x, rows, cols, rpt, out,
                              0u);
        switch (vec) {
            case 4:
                return launch_pdl(rowsum_narrow_kernel<4, false, false, false>, grid, block, stream, x, rows, cols, rpt,
                                  out, 0u);
            case 2:
                return rot ? launch_pdl(rowsum_narrow_kernel<2, true, false, false>, grid, block, stream, x, rows, cols,
                                        rpt, out, 0u)
                           : launch_pdl(rowsum_narrow_kernel<2, false, false, false>, grid, block, stream, x, rows, cols,
                                        rpt, out, 0u);
            default:
                return rot ? launch_pdl(rowsum_narrow_kernel<1, true, false, false>, grid, block, stream, x, rows, cols,
                                        rpt, out, 0u)
                           : launch_pdl(rowsum_narrow_kernel<1, false, false, false>, grid, block, stream, x, rows, cols,
                                        rpt, out, 0u);
        }
    }
    if (const int lw = rowsum_rows_staged_lanes(x, cols, ld)) {
        const int64_t w = rows_staged_slot(cols, lw);
        const int64_t rpt = kNarrowBulkTile / w;  // whole rows per tile
        const int64_t blocks = (rows + rpt - 1) / rpt;
        if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
        const dim3 grid{unsigned(blocks)}, block{unsigned(kNarrowBlock)};
        if (lw == 8)
            return launch_pdl(rowsum_rows_staged_kernel<8>, grid, block, stream, x, rows, cols, ld, w, rpt, out);
        if (lw == 16)
            return launch_pdl(rowsum_rows_staged_kernel<16>, grid, block, stream, x, rows, cols, ld, w, rpt, out);
        return launch_pdl(rowsum_rows_staged_kernel<32>, grid, block, stream, x, rows, cols, ld, w, rpt, out);
    }
    if (const int lw = rowsum_staged_lanes(x, cols, ld)) {
        const int64_t rpt = (kNarrowBulkTile - cols) / ld + 1;  // whole rows per tile (their span fits)
        const int64_t blocks = (rows + rpt - 1) / rpt;
        if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
        const dim3 grid{unsigned(blocks)}, block{unsigned(kNarrowBlock)};
        if (lw == 8) return launch_pdl(rowsum_staged_kernel<8>, grid, block, stream, x, rows, cols, ld, rpt, out);
        if (lw == 16) return launch_pdl(rowsum_staged_kernel<16>, grid, block, stream, x, rows, cols, ld, rpt, out);
        return launch_pdl(rowsum_staged_kernel<32>, grid, block, stream, x, rows, cols, ld, rpt, out);
    }
    if (const int g = rowsum_fitg_lanes(cols)) {
        const int64_t ng = kWarpSize / g;
        const int64_t nsteps = (rows + ng - 1) / ng;
        constexpr int64_t kWarpsPerBlock = kGroupBlock / kWarpSize;
        const int64_t blocks = (nsteps + kWarpsPerBlock - 1) / kWarpsPerBlock;  // one unit per warp
        if (blocks > 0x7fffffff) return cudaErrorInvalidValue;  // would take more than 5 * 10^10 rows
        const dim3 grid{unsigned(blocks)}, block{unsigned(kGroupBlock)};
        switch (g) {
            case 5: return launch_pdl(rowsum_fitg_kernel<5>, grid, block, stream, x, rows, cols, ld, out);
            case 6: return launch_pdl(rowsum_fitg_kernel<6>, grid, block, stream, x, rows, cols, ld, out);
            case 9: return launch_pdl(rowsum_fitg_kernel<9>, grid, block, stream, x, rows, cols, ld, out);
            default: return launch_pdl(rowsum_fitg_kernel<10>, grid, block, stream, x, rows, cols, ld, out);
        }
    }
    if (cols <= kFitRowMaxCols) {
        switch (lanes_per_row(cols)) {
            case 1: return launch_fit<1>(x, rows, cols, ld, out, stream);
            case 2: return launch_fit<2>(x, rows, cols, ld, out, stream);
            case 4: return launch_fit<4>(x, rows, cols, ld, out, stream);
            case 8: return launch_fit<8>(x, rows, cols, ld, out, stream);
            case 16: return launch_fit<16>(x, rows, cols, ld, out, stream);
            default: return launch_fit<32>(x, rows, cols, ld, out, stream);
        }
    }
    if (cols <= kGroupRowMaxCols) return launch_group<32>(x, rows, cols, ld, out, stream);
    const int64_t blocks = rows < 0x7fffffff ? rows : 0x7fffffff;
    if (cols >= kCtaDeepCols)
        return launch_pdl(rowsum_cta_kernel<kCtaUnrollDeep, 4>, dim3(unsigned(blocks)), dim3(kCtaBlock), stream, x, rows,
                          cols, ld, out);
    return launch_pdl(rowsum_cta_kernel<kCtaUnroll, 8>, dim3(unsigned(blocks)), dim3(kCtaBlock), stream, x, rows, cols, ld,
                      out);
}

}  // namespace rdx
