// device.cuh -- device-side building blocks shared by the reduction kernels:
// streaming 16-byte loads, the per-dtype "fold" of one 16-byte vector, the
// warp shuffle tree and the two-level block tree.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace rdx {

constexpr unsigned kFullMask = 0xffffffffu;
constexpr int kWarpSize = 32;

// ---------------------------------------------------------------------------
// Checked build (RDX_DEBUG=1): every global load and store of the kernels
// first asks guard() whether [p, p + bytes) lies inside the buffer it belongs
// to, [lo, lo + span).  An access outside is counted and skipped (never
// performed), so the build can run any input without faulting; the host
// reads the count through rdx_debug_violations().  In a normal build guard()
// is the constant true and costs nothing.
// ---------------------------------------------------------------------------
#ifndef RDX_DEBUG
#define RDX_DEBUG 0
#endif
#if RDX_DEBUG
static __device__ unsigned long long g_out_of_range;  // one per translation unit
__device__ __forceinline__ bool guard(const void* p, size_t bytes, const void* lo, size_t span) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(lo);
    const bool ok = a >= b && a + bytes <= b + span;
    if (!ok) atomicAdd(&g_out_of_range, 1ull);
    return ok;
}
// Host side: this translation unit's count (optionally reset to 0).
#define RDX_DEFINE_VIOLATION_COUNTER(fn)                                           \
    unsigned long long fn(bool reset) {                                           \
        unsigned long long v = 0;                                                 \
        if (cudaMemcpyFromSymbol(&v, g_out_of_range, sizeof v) != cudaSuccess) v = ~0ull; \
        if (reset) {                                                              \
            const unsigned long long z = 0;                                       \
            cudaMemcpyToSymbol(g_out_of_range, &z, sizeof z);                     \
        }                                                                         \
        return v;                                                                 \
    }
#else
__device__ __forceinline__ constexpr bool guard(const void*, size_t, const void*, size_t) { return true; }
#define RDX_DEFINE_VIOLATION_COUNTER(fn) \
    unsigned long long fn(bool) { return 0; }
#endif

// One 16-byte load on the read-only path.  Every input byte is read once, so
// the line is not kept in L1 (L1::no_allocate); L2::256B asks the L2 to fetch
// the whole 256-byte span the warp is about to stream through.  The asm is
// volatile so that a batch of these loads keeps its program order.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization (launch_pdl) may be scheduled while the kernel ahead of it in
// the stream is still running.  pdl_wait() holds the thread until that kernel
// has completed and its memory writes are visible (for a kernel launched
// without the attribute it returns at once), so it comes before the first
// global memory access.  pdl_release() lets the next such kernel be scheduled
// onto the SMs this grid leaves free; it waits there in pdl_wait().
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_release() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Issue order fence for a batch of loads: every register of v passes through
// an empty volatile asm placed after the whole batch, so no arithmetic on the
// batch can be scheduled between its loads and all N loads are in flight
// together (the compiler would otherwise sink each load next to its use).
template <int N>
__device__ __forceinline__ void batch_fence(uint4 (&v)[N]) {
#pragma unroll
    for (int u = 0; u < N; ++u) asm volatile("" : "+r"(v[u].x), "+r"(v[u].y), "+r"(v[u].z), "+r"(v[u].w));
}

// ---------------------------------------------------------------------------
// Term policies.  Each describes one reduction: the input element type, the
// accumulator, how one element becomes a term, and how the 16-byte vector of
// V elements becomes one accumulator value (a fixed pairwise tree, so every
// run adds the same operands in the same order).  Float policies keep one
// accumulator per load in flight (shorter rounding chains); exact ones may
// declare kExact and share one.
// ---------------------------------------------------------------------------

template <class P, class = void>
struct is_exact {
    static constexpr bool value = false;
};
template <class P>
struct is_exact<P, decltype(void(P::kExact))> {
    static constexpr bool value = P::kExact;
};

// Reductions whose result has the same bits in any order (int64 addition,
// which is addition modulo 2^64, and the maxima) may finish
// through one 8-byte accumulator word per row instead of block partials:
// every block folds its total in with a fire-and-forget atomic, and the
// block that draws the last ticket takes the word (reading it and leaving it
// zero).  Such a policy declares kWordFinish and provides
//   fold_word(word, acc)  atomically fold a block total into the word;
//   take_word(word)       atomically read the word, reset it to zero, and
//                         return the result it holds (zero stands for the
//                         policy's identity).
template <class P, class = void>
struct has_word_finish {
    static constexpr bool value = false;
};
template <class P>
struct has_word_finish<P, decltype(void(P::kWordFinish))> {
    static constexpr bool value = P::kWordFinish;
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

struct SumF32 {
    using In = float;
    using Acc = float;
    static constexpr int kVec = 4;
    __device__ static uint4 neutral() { return make_uint4(0u, 0u, 0u, 0u); }  // folds to the identity
    __device__ static Acc identity() { return 0.f; }
    __device__ static Acc term(In v) { return v; }
    __device__ static Acc fold(uint4 v) {
        return (__uint_as_float(v.x) + __uint_as_float(v.y)) + (__uint_as_float(v.z) + __uint_as_float(v.w));
    }
};

struct SumSqF32 {
    using In = float;
    using Acc = float;
    static constexpr int kVec = 4;
    __device__ static uint4 neutral() { return make_uint4(0u, 0u, 0u, 0u); }  // folds to the identity
    __device__ static Acc identity() { return 0.f; }
    __device__ static Acc term(In v) { return v * v; }
    __device__ static Acc fold(uint4 v) {
        const float a = __uint_as_float(v.x), b = __uint_as_float(v.y);
        const float c = __uint_as_float(v.z), d = __uint_as_float(v.w);
        return __fmaf_rn(a, a, b * b) + __fmaf_rn(c, c, d * d);
    }
};

struct SumBF16 {
    using In = uint16_t;
    using Acc = float;
    static constexpr int kVec = 8;
    __device__ static uint4 neutral() { return make_uint4(0u, 0u, 0u, 0u); }  // folds to the identity
    __device__ static Acc identity() { return 0.f; }
    __device__ static Acc term(In v) { return __uint_as_float(uint32_t(v) << 16); }
    __device__ static float pair(uint32_t w) { return bf16_lo(w) + bf16_hi(w); }
    __device__ static Acc fold(uint4 v) { return (pair(v.x) + pair(v.y)) + (pair(v.z) + pair(v.w)); }
};

struct SumSqBF16 {
    using In = uint16_t;
    using Acc = float;
    static constexpr int kVec = 8;
    __device__ static uint4 neutral() { return make_uint4(0u, 0u, 0u, 0u); }  // folds to the identity
    __device__ static Acc identity() { return 0.f; }
    __device__ static Acc term(In v) {
        const float f = __uint_as_float(uint32_t(v) << 16);
        return f * f;
    }
    __device__ static float pair(uint32_t w) {
        const float lo = bf16_lo(w), hi = bf16_hi(w);
        return __fmaf_rn(lo, lo, hi * hi);
    }
    __device__ static Acc fold(uint4 v) { return (pair(v.x) + pair(v.y)) + (pair(v.z) + pair(v.w)); }
};

struct SumI32 {
    using In = int32_t;
    using Acc = long long;
    static constexpr int kVec = 4;
    // int64 addition is exact and associative: the grouping cannot change the
    // result, so one accumulator per thread is enough (and saves registers).
    static constexpr bool kExact = true;
    __device__ static uint4 neutral() { return make_uint4(0u, 0u, 0u, 0u); }  // folds to the identity
    __device__ static Acc identity() { return 0; }
    __device__ static Acc term(In v) { return Acc(v); }
    __device__ static Acc fold(uint4 v) {
        return (Acc(int32_t(v.x)) + Acc(int32_t(v.y))) + (Acc(int32_t(v.z)) + Acc(int32_t(v.w)));
    }
    // the word holds the running int64 sum (its two's-complement bits)
    static constexpr bool kWordFinish = true;
    __device__ static void fold_word(unsigned long long* w, Acc a) {
        atomicAdd(w, static_cast<unsigned long long>(a));  // result unused: a reduction (red), no round trip
    }
    __device__ static Acc take_word(unsigned long long* w) { return static_cast<Acc>(atomicExch(w, 0ull)); }
};

// Sum and sum of squares carried together (one pass over the input for both).
// Each component is added in exactly the order the single reductions use.
struct __align__(8) SumSq2 {
    float s;  // sum
    float q;  // sum of squares
    SumSq2() = default;
    __host__ __device__ explicit SumSq2(float v) : s(v), q(v) {}
    __host__ __device__ SumSq2(float s_, float q_) : s(s_), q(q_) {}
};
__device__ __forceinline__ SumSq2 operator+(SumSq2 a, SumSq2 b) { return SumSq2(a.s + b.s, a.q + b.q); }
__device__ __forceinline__ SumSq2& operator+=(SumSq2& a, SumSq2 b) {
    a.s += b.s;
    a.q += b.q;
    return a;
}

struct SumSumSqF32 {
    using In = float;
    using Acc = SumSq2;
    static constexpr int kVec = 4;
    __device__ static uint4 neutral() { return make_uint4(0u, 0u, 0u, 0u); }  // folds to the identity
    __device__ static Acc identity() { return Acc(0.f); }
    __device__ static Acc term(In v) { return Acc(SumF32::term(v), SumSqF32::term(v)); }
    __device__ static Acc fold(uint4 v) { return Acc(SumF32::fold(v), SumSqF32::fold(v)); }
};

struct SumSumSqBF16 {
    using In = uint16_t;
    using Acc = SumSq2;
    static constexpr int kVec = 8;
    __device__ static uint4 neutral() { return make_uint4(0u, 0u, 0u, 0u); }  // folds to the identity
    __device__ static Acc identity() { return Acc(0.f); }
    __device__ static Acc term(In v) { return Acc(SumBF16::term(v), SumSqBF16::term(v)); }
    __device__ static Acc fold(uint4 v) { return Acc(SumBF16::fold(v), SumSqBF16::fold(v)); }
};

// Maximum.  The page "lecture02/simt.py" models atomic_max as "replace the
// stored value if the new one is greater"; folded from -Inf that is the
// maximum, with NaNs never winning.  fmaxf returns the other operand when one
// is NaN, so the same rule holds here in any grouping: the result does not
// depend on the order (up to the sign of a zero maximum).  The accumulator's
// "+" is the maximum, so the sum trees serve unchanged.
struct MaxAccF {
    float v;
    MaxAccF() = default;
    __host__ __device__ explicit MaxAccF(float x) : v(x) {}
};
__device__ __forceinline__ MaxAccF operator+(MaxAccF a, MaxAccF b) { return MaxAccF(fmaxf(a.v, b.v)); }
__device__ __forceinline__ MaxAccF& operator+=(MaxAccF& a, MaxAccF b) {
    a.v = fmaxf(a.v, b.v);
    return a;
}

struct MaxAccI {
    int v;
    MaxAccI() = default;
    __host__ __device__ explicit MaxAccI(int x) : v(x) {}
};
__device__ __forceinline__ MaxAccI operator+(MaxAccI a, MaxAccI b) { return MaxAccI(max(a.v, b.v)); }
__device__ __forceinline__ MaxAccI& operator+=(MaxAccI& a, MaxAccI b) {
    a.v = max(a.v, b.v);
    return a;
}

struct MaxF32 {
    using In = float;
    using Acc = MaxAccF;
    static constexpr int kVec = 4;
    static constexpr bool kExact = true;  // max is exact in any grouping
    __device__ static uint4 neutral() { return make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u); }
    __device__ static Acc identity() { return Acc(-__int_as_float(0x7f800000)); }  // -Inf
    __device__ static Acc term(In v) { return Acc(v); }
    __device__ static Acc fold(uint4 v) {
        return Acc(fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
                         fmaxf(__uint_as_float(v.z), __uint_as_float(v.w))));
    }
    // The word holds the running maximum as an unsigned key that orders as
    // the floats do: non-negative values with the sign bit set, negative ones
    // with every bit flipped (-Inf becomes 0x007fffff, -0 sorts just below
    // +0).  A block total is never NaN (the fold starts from -Inf and fmaxf
    // drops NaNs), and key 0, which no folded value gives, stands for -Inf.
    static constexpr bool kWordFinish = true;
    __device__ static unsigned key(float f) {
        const unsigned u = __float_as_uint(f);
        return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    }
    __device__ static void fold_word(unsigned long long* w, Acc a) {
        atomicMax(w, static_cast<unsigned long long>(key(a.v)));
    }
    __device__ static Acc take_word(unsigned long long* w) {
        const unsigned k = static_cast<unsigned>(atomicExch(w, 0ull));
        if (k == 0u) return identity();
        return Acc(__uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k));
    }
};

struct MaxI32 {
    using In = int32_t;
    using Acc = MaxAccI;
    static constexpr int kVec = 4;
    static constexpr bool kExact = true;
    __device__ static uint4 neutral() { return make_uint4(0x80000000u, 0x80000000u, 0x80000000u, 0x80000000u); }
    __device__ static Acc identity() { return Acc(int(0x80000000u)); }  // -2^31
    __device__ static Acc term(In v) { return Acc(v); }
    __device__ static Acc fold(uint4 v) {
        return Acc(max(max(int(v.x), int(v.y)), max(int(v.z), int(v.w))));
    }
    // The word holds the running maximum as an unsigned key: the value with
    // its sign bit flipped, which orders as the signed value does and maps
    // the identity -2^31 to zero.
    static constexpr bool kWordFinish = true;
    __device__ static void fold_word(unsigned long long* w, Acc a) {
        atomicMax(w, static_cast<unsigned long long>(static_cast<unsigned>(a.v) ^ 0x80000000u));
    }
    __device__ static Acc take_word(unsigned long long* w) {
        return Acc(static_cast<int>(static_cast<unsigned>(atomicExch(w, 0ull)) ^ 0x80000000u));
    }
};

// ---------------------------------------------------------------------------
// Shuffle and coherent-load overloads for the accumulator types.
// ---------------------------------------------------------------------------

__device__ __forceinline__ float shfl_down(float v, int off) { return __shfl_down_sync(kFullMask, v, off); }
__device__ __forceinline__ long long shfl_down(long long v, int off) { return __shfl_down_sync(kFullMask, v, off); }
__device__ __forceinline__ SumSq2 shfl_down(SumSq2 v, int off) {
    return SumSq2(shfl_down(v.s, off), shfl_down(v.q, off));
}
__device__ __forceinline__ MaxAccF shfl_down(MaxAccF v, int off) { return MaxAccF(shfl_down(v.v, off)); }
__device__ __forceinline__ MaxAccI shfl_down(MaxAccI v, int off) {
    return MaxAccI(__shfl_down_sync(kFullMask, v.v, off));
}

// Completion counter of the last-block-done finish: acquire-release at GPU
// scope, so the partial this thread stored before is visible to the block
// that draws the last ticket, and that block sees every other block's partial.
__device__ __forceinline__ unsigned take_ticket(unsigned* counter) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
                 : "=r"(old)
                 : "l"(counter), "r"(1u)
                 : "memory");
    return old;
}

// Loads of values other blocks wrote in this kernel: through L2 (ld.global.cg),
// never a stale L1 line.
__device__ __forceinline__ float load_cg(const float* p) { return __ldcg(p); }
__device__ __forceinline__ long long load_cg(const long long* p) { return __ldcg(p); }
__device__ __forceinline__ SumSq2 load_cg(const SumSq2* p) {
    const float2 v = __ldcg(reinterpret_cast<const float2*>(p));
    return SumSq2(v.x, v.y);
}
__device__ __forceinline__ MaxAccF load_cg(const MaxAccF* p) {
    return MaxAccF(__ldcg(reinterpret_cast<const float*>(p)));
}
__device__ __forceinline__ MaxAccI load_cg(const MaxAccI* p) { return MaxAccI(__ldcg(reinterpret_cast<const int*>(p))); }

// ---------------------------------------------------------------------------
// Trees.
// ---------------------------------------------------------------------------

// Lane 0 ends with the sum of the 32 lanes' values: shuffle-down by 16, 8, 4,
// 2, 1 (lanes past the warp's end read their own value, which never reaches
// lane 0).
template <class T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
    for (int off = kWarpSize / 2; off > 0; off >>= 1) v += shfl_down(v, off);
    return v;
}

// The exact integer trees run on the warp's 32-bit reduce unit (redux.sync,
// one instruction per 32 lanes) instead of five shuffle steps; every lane
// ends with the result.
//
// int64 sum: each lane's value, read as 64 unsigned bits, is cut into its
// high word and two 16-bit low parts.  32 parts of 16 bits add up to less
// than 2^21, so those two sums are exact; the high words' sum wraps modulo
// 2^32, which loses nothing, because it is weighted by 2^32 and int64
// (two's-complement) addition is itself addition modulo 2^64.
__device__ __forceinline__ long long warp_sum(long long v) {
    const unsigned long long u = static_cast<unsigned long long>(v);
    const unsigned hi = __reduce_add_sync(kFullMask, unsigned(u >> 32));
    const unsigned mid = __reduce_add_sync(kFullMask, unsigned(u >> 16) & 0xffffu);
    const unsigned lo = __reduce_add_sync(kFullMask, unsigned(u) & 0xffffu);
    return static_cast<long long>((static_cast<unsigned long long>(hi) << 32) +
                                  (static_cast<unsigned long long>(mid) << 16) + lo);
}

// int32 maximum: the reduce unit's signed maximum.
__device__ __forceinline__ MaxAccI warp_sum(MaxAccI v) { return MaxAccI(__reduce_max_sync(kFullMask, v.v)); }

// Every lane of each aligned group of `width` lanes ends with the group's sum.
// In the xor butterfly both partners add the same two values, so all lanes of
// the group hold the identical result.
template <int width, class T>
__device__ __forceinline__ T group_allreduce(T v) {
#pragma unroll
    for (int off = width / 2; off > 0; off >>= 1) v += __shfl_xor_sync(kFullMask, v, off);
    return v;
}

// Fixed pairwise fold of a register array (N a power of two).
template <int N, class T>
__device__ __forceinline__ T fold_array(T (&a)[N]) {
#pragma unroll
    for (int w = N / 2; w > 0; w >>= 1) {
#pragma unroll
        for (int i = 0; i < w; ++i) a[i] = a[i] + a[i + w];
    }
    return a[0];
}

// Block tree: warp trees, then lane 0 of warp w parks its value in smem[w]
// and warp 0 reduces smem[0 .. kWarps) (consecutive words: one shared-memory
// wavefront, no bank conflict).  The result is valid in thread 0.  smem must
// not be in use by other threads when called; the call ends before any
// thread may write smem again only after a later __syncthreads().
template <int kBlock, class T>
__device__ __forceinline__ T block_sum(T v, T* smem, T identity) {
    constexpr int kWarps = kBlock / kWarpSize;
    static_assert(kWarps <= kWarpSize, "block too large for a one-warp second stage");
    v = warp_sum(v);
    const int lane = threadIdx.x % kWarpSize;
    const int warp = threadIdx.x / kWarpSize;
    if (lane == 0) smem[warp] = v;
    __syncthreads();
    T r = identity;
    if (warp == 0) {
        r = lane < kWarps ? smem[lane] : identity;
        r = warp_sum(r);
    }
    return r;
}

}  // namespace rdx
