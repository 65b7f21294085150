// reduce.cu -- one-pass scalar sum reductions (float32, float32 squares,
// bfloat16 -> float32, int32 -> int64, and sum + sum of squares together)
// with a deterministic on-device finish.
//
// The page "03_shared_memory_sync_reduction.py", demo 3, walks from a
// divergent shared-memory tree (version 1) to "first add during load" plus a
// warp-shuffle finish (version 5), and ends each kernel with one partial per
// block that the host adds up.  This kernel keeps version 5's shape and takes
// its ideas further for a GPU with 152 SMs and HBM3e:
//   * tiles: the 16-byte-aligned body of the input is cut into equal
//     contiguous tiles, one block per tile (8192 tiles of 128 KiB for a 1 GiB
//     input, about 1024 tiles of up to 64 KiB for 16-512 MiB inputs, tiles of
//     at least 16 KiB); the hardware hands tiles to SMs as they free up, so a
//     slow SM does not hold back the end of the kernel;
//   * add on load: inside its tile each thread keeps kUnroll independent
//     16-byte loads in flight (kUnrollLarge, at half the occupancy, for
//     inputs of many waves) and folds each vector into its own register
//     accumulator (version 4's two elements per thread become dozens);
//   * shuffle trees: a warp tree, then one shared-memory word per warp, then
//     a warp tree over those words (one barrier per block);
//   * the tile partials are finished on the device: the block that arrives
//     last at a completion counter (acquire-release atomic) adds all partials
//     in a fixed order and resets the counter.  Nothing waits on anything,
//     and no float atomics are used.  The reductions whose result has the
//     same bits in any order (the int64 sum and both maxima) fold each block
//     total into one accumulator word with an integer atomic instead, and
//     the last block only reads that word back.  With tiles of 64 KiB and
//     more the same pass (or the word's read) runs in finish_kernel, a
//     second kernel launched behind the tiles, and no tile block waits for a
//     ticket: the same bits, less tail where the tiles run many waves.
// Launched with programmatic dependent launch, a call queued behind another
// kernel is scheduled while that kernel drains and starts reading once its
// writes are visible.
// The same kernel sums the rows of a matrix with few, long rows: gridDim.y
// rows, each cut into tiles with its own completion counter and partials;
// the scalar reductions are the one-row case.
// The tiling depends only on the row length and the row's 16-byte alignment,
// so the summation order, and the result, are the same on every run and
// every GPU.
#include "device.cuh"
#include "launch.h"

#ifndef RDX_REDUCE_BLOCK
#define RDX_REDUCE_BLOCK 256
#endif
#ifndef RDX_REDUCE_MIN_TILE
#define RDX_REDUCE_MIN_TILE 1024
#endif
#ifndef RDX_SEPARATE_FINISH_MIN_TILE
#define RDX_SEPARATE_FINISH_MIN_TILE 4096
#endif

namespace rdx {
namespace {

constexpr int kBlock = RDX_REDUCE_BLOCK;                  // threads per block
constexpr int kUnroll = 4;                                // 16-byte loads in flight per thread
constexpr int kUnrollLarge = 8;                           // the same, inputs of kLargeTiles tiles or more
constexpr int64_t kMaxTiles = kReduceMaxTiles;            // tiles (= partials) aimed at per call
constexpr int64_t kMinTile = RDX_REDUCE_MIN_TILE;         // 16-byte vectors per tile, at least
constexpr int64_t kMidTiles = 1024;                       // tiles aimed at for mid-size inputs
constexpr int64_t kMidTileCap = 4096;                     // largest tile of the mid-size rule (64 KiB)
constexpr int kFinishLoadBytes = 32;                      // partial bytes in flight per thread, last block
// Tiles of at least this many 16-byte vectors (64 KiB: inputs of 64 MiB and
// up) finish in a second kernel instead of the last block.  Measured, fp32,
// L2 flushed, means of 61: 64 MiB 17.6 -> 17.0 us, 256 MiB 44.6 -> 43.4 us,
// 1 GiB 149.1 -> 148.7 us; with shorter tiles the second launch costs more
// than the tickets it saves (16 MiB 9.9 -> 10.7 us).
constexpr int64_t kSeparateFinishMinTile = RDX_SEPARATE_FINISH_MIN_TILE;
// 8 resident blocks of 256 threads fill an SM (2048 threads): at most 32
// registers per thread, so every dtype streams with full occupancy.
constexpr int kMinBlocksPerSm = 2048 / kBlock;
// Large inputs (many waves of tiles) stream faster from fewer, deeper
// blocks: 4 blocks per SM with 8 loads in flight per thread keep the same
// bytes in flight over half as many concurrent streams (measured: 1.0-1.5 %
// less time at 1-2 GiB, and slower below 256 MiB, where tiles are short).
constexpr int kMinBlocksLarge = 4;
constexpr int64_t kLargeTiles = 4096;
static_assert((kUnroll & (kUnroll - 1)) == 0 && (kUnrollLarge & (kUnrollLarge - 1)) == 0,
              "load batches are powers of two");
static_assert(kMinTile % kBlock == 0, "tiles are whole multiples of the block");

// The fixed-order pass over one row's g partials rp[0 .. g): thread t adds
// partials t, t + kBlock, ... (kFinishUnroll independent chains, their loads
// in flight together), then the block tree.  The result is valid in thread 0.
// Loads go through L2 (other blocks, or another grid, wrote the partials).
template <class P>
__device__ __forceinline__ typename P::Acc finish_row(const typename P::Acc* __restrict__ rp, int g,
                                                      const void* part_lo, size_t part_span,
                                                      typename P::Acc* smem) {
    using Acc = typename P::Acc;
    constexpr int kFinishUnroll = kFinishLoadBytes / int(sizeof(Acc));
    Acc b[kFinishUnroll];
#pragma unroll
    for (int u = 0; u < kFinishUnroll; ++u) b[u] = P::identity();
    int j = threadIdx.x;
    for (; j + (kFinishUnroll - 1) * kBlock < g; j += kFinishUnroll * kBlock) {
        Acc p[kFinishUnroll];
#pragma unroll
        for (int u = 0; u < kFinishUnroll; ++u)
            p[u] = guard(rp + j + u * kBlock, sizeof(Acc), part_lo, part_span) ? load_cg(rp + j + u * kBlock)
                                                                             : P::identity();
#pragma unroll
        for (int u = 0; u < kFinishUnroll; ++u) b[u] += p[u];
    }
#pragma unroll
    for (int u = 0; u < kFinishUnroll; ++u) {
        if (j + u * kBlock < g && guard(rp + j + u * kBlock, sizeof(Acc), part_lo, part_span))
            b[u] += load_cg(rp + j + u * kBlock);
    }
    return block_sum<kBlock>(fold_array(b), smem, P::identity());
}

// kSeparate: the grid leaves the finish to finish_kernel, launched right
// after it on the same stream: every block only stores its partial (or folds
// its total into the accumulator word) and exits, with no ticket to wait for.
template <class P, int U, int kMinBlocks, bool kSeparate>
__global__ void __launch_bounds__(kBlock, kMinBlocks)
reduce_kernel(const typename P::In* __restrict__ x, int64_t cols, int64_t ld, int64_t tile,
              typename P::Acc* __restrict__ partials, unsigned* __restrict__ counters,
              unsigned long long* __restrict__ words, typename P::Acc* __restrict__ out) {
    using Acc = typename P::Acc;
    constexpr int V = P::kVec;
    __shared__ Acc smem[kBlock / kWarpSize];
    __shared__ unsigned last_block;
    pdl_wait();     // the previous kernel in the stream has finished writing
    pdl_release();  // the next one may be scheduled into SMs this grid frees

    // This block's row and tile.  head = elements before the row's first
    // 16-byte boundary, then m whole 16-byte vectors, then the tail.
    const int64_t row = blockIdx.y;
    const typename P::In* __restrict__ xr = x + row * ld;
    const uintptr_t mis = reinterpret_cast<uintptr_t>(xr) & 15u;
    int64_t head = mis ? int64_t((16u - mis) / sizeof(typename P::In)) : 0;
    if (head > cols) head = cols;
    const int64_t m = (cols - head) / V;
    const int64_t t0 = int64_t(blockIdx.x) * tile;
    const int64_t t1 = t0 + tile < m ? t0 + tile : m;
    const uint4* __restrict__ xv = reinterpret_cast<const uint4*>(xr + head);

    // accumulator of load slot u: its own for float sums, a shared one for
    // exact (integer) sums
    constexpr bool kShared = is_exact<P>::value;
    auto kAccOf = [](int u) { return kShared ? 0 : u; };
    Acc acc[U];
#pragma unroll
    for (int u = 0; u < U; ++u) acc[u] = P::identity();

    // Fewer than V elements before the first 16-byte boundary and after the
    // last whole vector: the first threads of the row's tile 0 take one each.
    const size_t span = size_t(cols) * sizeof(typename P::In);  // this row's bytes
    if (blockIdx.x == 0) {
        const int64_t tail0 = head + m * V;
        if (threadIdx.x < head && guard(xr + threadIdx.x, sizeof(typename P::In), xr, span))
            acc[0] += P::term(xr[threadIdx.x]);
        if (threadIdx.x < cols - tail0 && guard(xr + tail0 + threadIdx.x, sizeof(typename P::In), xr, span))
            acc[U - 1] += P::term(xr[tail0 + threadIdx.x]);
    }

    int64_t i = t0 + threadIdx.x;
    for (; i + (U - 1) * kBlock < t1; i += U * kBlock) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            v[u] = guard(xv + i + u * kBlock, 16, xr, span) ? ld_stream16(xv + i + u * kBlock) : P::neutral();
        batch_fence(v);
#pragma unroll
        for (int u = 0; u < U; ++u) acc[kAccOf(u)] += P::fold(v[u]);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int64_t j = i + u * kBlock;
        if (j < t1 && guard(xv + j, 16, xr, span)) acc[kAccOf(u)] += P::fold(ld_stream16(xv + j));
    }

    Acc a = block_sum<kBlock>(fold_array(acc), smem, P::identity());

    const size_t out_span = size_t(gridDim.y) * sizeof(Acc);
    if (gridDim.x == 1) {
        if (threadIdx.x == 0 && guard(out + row, sizeof(Acc), out, out_span)) out[row] = a;
        return;
    }
    unsigned* counter = counters + row;
    if constexpr (has_word_finish<P>::value) {
        // Order-independent reductions: the block total goes into the row's
        // accumulator word (a fire-and-forget atomic, released by the ticket
        // that follows it); the block with the last ticket takes the word.
        // One thread does it all: no partial is stored or read again.
        if (threadIdx.x == 0) {
            unsigned long long* word = words + row;
            const size_t word_span = size_t(gridDim.y) * sizeof(unsigned long long);
            if (guard(word, sizeof *word, words, word_span)) P::fold_word(word, a);
            if (kSeparate) return;
            if (guard(counter, sizeof(unsigned), counters, gridDim.y * sizeof(unsigned)) &&
                take_ticket(counter) == gridDim.x - 1) {
                const Acc total = guard(word, sizeof *word, words, word_span) ? P::take_word(word) : P::identity();
                if (guard(out + row, sizeof(Acc), out, out_span)) out[row] = total;
                *counter = 0u;  // ready for the next call on this stream (checked above)
            }
        }
        return;
    }
    Acc* __restrict__ rp = partials + row * int64_t(gridDim.x);
    const size_t part_span = size_t(gridDim.x) * gridDim.y * sizeof(Acc);
    if (kSeparate) {
        if (threadIdx.x == 0 && guard(rp + blockIdx.x, sizeof(Acc), partials, part_span)) rp[blockIdx.x] = a;
        return;
    }
    if (threadIdx.x == 0) {
        if (guard(rp + blockIdx.x, sizeof(Acc), partials, part_span)) rp[blockIdx.x] = a;
        last_block = guard(counter, sizeof(unsigned), counters, gridDim.y * sizeof(unsigned))
                         ? take_ticket(counter) == gridDim.x - 1
                         : 0u;
    }
    __syncthreads();
    if (!last_block) return;

    // The row's last block: every partial of the row is in place.
    const Acc total = finish_row<P>(rp, int(gridDim.x), partials, part_span, smem);
    if (threadIdx.x == 0) {
        if (guard(out + row, sizeof(Acc), out, out_span)) out[row] = total;
        *counter = 0u;  // ready for the next call on this stream (checked above)
    }
}

// The finish of a kSeparate grid: one block per row, launched behind it with
// programmatic dependent launch.  griddepcontrol.wait returns once that grid
// has completed and its writes are visible, so every partial (or the whole
// accumulator word) is in place.  The same fixed-order pass as the last
// block's above, so the result has the same bits either way.
template <class P>
__global__ void __launch_bounds__(kBlock)
finish_kernel(const typename P::Acc* __restrict__ partials, int64_t tiles, unsigned long long* __restrict__ words,
              typename P::Acc* __restrict__ out) {
    using Acc = typename P::Acc;
    __shared__ Acc smem[kBlock / kWarpSize];
    pdl_wait();
    pdl_release();
    const int64_t row = blockIdx.x;
    const size_t out_span = size_t(gridDim.x) * sizeof(Acc);
    if constexpr (has_word_finish<P>::value) {
        if (threadIdx.x == 0) {
            unsigned long long* word = words + row;
            const size_t word_span = size_t(gridDim.x) * sizeof(unsigned long long);
            const Acc total = guard(word, sizeof *word, words, word_span) ? P::take_word(word) : P::identity();
            if (guard(out + row, sizeof(Acc), out, out_span)) out[row] = total;
        }
        return;
    }
    const size_t part_span = size_t(tiles) * gridDim.x * sizeof(Acc);
    const Acc total = finish_row<P>(partials + row * tiles, int(tiles), partials, part_span, smem);
    if (threadIdx.x == 0 && guard(out + row, sizeof(Acc), out, out_span)) out[row] = total;
}

template <class P>
cudaError_t launch_typed(const void* x, int64_t rows, int64_t cols, int64_t ld, const ReducePlan& plan,
                         void* partials, unsigned* counters, unsigned long long* words, void* out,
                         cudaStream_t stream) {
    const dim3 grid(unsigned(plan.tiles), unsigned(rows));
    const auto* xt = static_cast<const typename P::In*>(x);
    auto* pt = static_cast<typename P::Acc*>(partials);
    auto* ot = static_cast<typename P::Acc*>(out);
    cudaError_t e;
    if (plan.separate_finish) {
        e = plan.large ? launch_pdl(reduce_kernel<P, kUnrollLarge, kMinBlocksLarge, true>, grid, dim3(kBlock), stream,
                                    xt, cols, ld, plan.tile, pt, counters, words, ot)
                       : launch_pdl(reduce_kernel<P, kUnroll, kMinBlocksPerSm, true>, grid, dim3(kBlock), stream, xt,
                                    cols, ld, plan.tile, pt, counters, words, ot);
        if (e != cudaSuccess) return e;
        return launch_pdl(finish_kernel<P>, dim3(unsigned(rows)), dim3(kBlock), stream,
                          static_cast<const typename P::Acc*>(pt), plan.tiles, words, ot);
    }
    if (plan.large)
        return launch_pdl(reduce_kernel<P, kUnrollLarge, kMinBlocksLarge, false>, grid, dim3(kBlock), stream, xt, cols,
                          ld, plan.tile, pt, counters, words, ot);
    return launch_pdl(reduce_kernel<P, kUnroll, kMinBlocksPerSm, false>, grid, dim3(kBlock), stream, xt, cols, ld,
                      plan.tile, pt, counters, words, ot);
}

}  // namespace

RDX_DEFINE_VIOLATION_COUNTER(reduce_out_of_range)

int reduce_block_threads() { return kBlock; }
// rows * tiles <= kMaxTiles for any rows <= kMaxTiles (see reduce_plan)
int64_t reduce_max_partials() { return kMaxTiles; }

int reduce_vec_elems(Op op) {
    switch (op) {
        case Op::SumBF16:
        case Op::SumSqBF16:
        case Op::SumSumSqBF16: return 8;
        default: return 4;  // float and int32 inputs
    }
}

size_t reduce_elem_bytes(Op op) { return 16 / size_t(reduce_vec_elems(op)); }

size_t reduce_acc_bytes(Op op) {
    return (op == Op::SumI32 || op == Op::SumSumSqF32 || op == Op::SumSumSqBF16) ? 8 : 4;
}

ReducePlan reduce_plan(Op op, int64_t rows, int64_t cols) {
    ReducePlan p;
    const int64_t mmax = cols / reduce_vec_elems(op);  // whole vectors of a row, at most
    const int64_t r = rows > 0 ? rows : 1;
    // large inputs: up to kMaxTiles tiles, many waves for the block scheduler
    const int64_t target = kMaxTiles / r;
    int64_t tile = (mmax + target - 1) / (target > 0 ? target : 1);
    // mid-size inputs: about kMidTiles tiles of at most kMidTileCap vectors
    // (fewer, longer blocks: less per-block overhead where the whole input
    // is only a few waves deep)
    const int64_t mid = (r * mmax + kMidTiles - 1) / kMidTiles;
    const int64_t mid_tile = mid < kMidTileCap ? mid : kMidTileCap;
    if (tile < mid_tile) tile = mid_tile;
    tile = (tile + kBlock - 1) / kBlock * kBlock;  // whole blocks of vectors
    if (tile < kMinTile) tile = kMinTile;
    p.tile = tile;
    p.tiles = mmax > 0 ? (mmax + tile - 1) / tile : 1;
    // many waves of tiles long enough for whole batches of the deeper kernel
    p.large = r * p.tiles >= kLargeTiles && tile >= kUnrollLarge * kBlock;
    // long tiles: the finish in a kernel of its own (blocks exit without a ticket)
    p.separate_finish = p.tiles > 1 && tile >= kSeparateFinishMinTile;
    return p;
}

bool reduce_uses_words(Op op) { return op == Op::SumI32 || op == Op::MaxI32 || op == Op::MaxF32; }

cudaError_t reduce_launch(Op op, const void* x, int64_t rows, int64_t cols, int64_t ld, const ReducePlan& plan,
                          void* partials, unsigned* counters, unsigned long long* words, void* out,
                          cudaStream_t stream) {
    // the word finish serves one row (the scalar reductions)
    if (reduce_uses_words(op) && plan.tiles > 1 && (rows != 1 || words == nullptr)) return cudaErrorInvalidValue;
#define RDX_LAUNCH(P) launch_typed<P>(x, rows, cols, ld, plan, partials, counters, words, out, stream)
    switch (op) {
        case Op::SumF32: return RDX_LAUNCH(SumF32);
        case Op::SumSqF32: return RDX_LAUNCH(SumSqF32);
        case Op::SumBF16: return RDX_LAUNCH(SumBF16);
        case Op::SumSqBF16: return RDX_LAUNCH(SumSqBF16);
        case Op::SumI32: return RDX_LAUNCH(SumI32);
        case Op::SumSumSqF32: return RDX_LAUNCH(SumSumSqF32);
        case Op::SumSumSqBF16: return RDX_LAUNCH(SumSumSqBF16);
        case Op::MaxF32: return RDX_LAUNCH(MaxF32);
        case Op::MaxI32: return RDX_LAUNCH(MaxI32);
        default: return cudaErrorInvalidValue;
    }
#undef RDX_LAUNCH
}

}  // namespace rdx
