// api.cu -- the extern "C" entry points declared in include/rdx.h: argument
// validation (before any CUDA call), device capability cache, per-(device,
// stream) workspace cache, choice of kernel and launch.
#include "rdx.h"

#include <climits>
#include <cstdlib>
#include <functional>
#include <map>
#include <mutex>
#include <string>
#include <thread>
#include <tuple>

#include "device.cuh"  // RDX_DEBUG
#include "launch.h"

namespace {

using rdx::DeviceCaps;
using rdx::Op;

thread_local std::string t_last_error;

rdx_status fail_cuda(const char* what, cudaError_t e) {
    t_last_error = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
    return RDX_ERR_CUDA;
}

std::mutex g_mu;
std::map<int, DeviceCaps> g_caps;                          // by device ordinal
// by (device, stream, host thread): cudaStreamPerThread names a different
// stream in every host thread, so its workspaces are kept per thread (the
// thread part of the key is 0 for every other stream)
std::map<std::tuple<int, uintptr_t, size_t>, void*> g_workspaces;

// Workspace layout: [completion counters: one per row, kMaxSplitRows of them]
// [accumulator word of the order-independent reductions (int64 sum, maxima),
//  padded to 256 bytes]
// [tile partials: reduce_max_partials() slots of 8 bytes].  The counters and
// the word must be zero before a launch; every launch leaves them zero.
constexpr size_t kCounterBytes = size_t(rdx::kMaxSplitRows) * sizeof(unsigned);
constexpr size_t kWordBytes = 256;
constexpr size_t kZeroBytes = kCounterBytes + kWordBytes;  // the part that starts zeroed
static_assert(kCounterBytes % 256 == 0 && kZeroBytes % 256 == 0, "word and partials start 256-byte aligned");

size_t workspace_bytes() { return kZeroBytes + size_t(rdx::reduce_max_partials()) * 8; }

struct WorkspaceParts {
    unsigned* counters = nullptr;
    unsigned long long* words = nullptr;
    void* partials = nullptr;
};
WorkspaceParts parts_of(void* ws) {
    WorkspaceParts p;
    if (ws != nullptr) {
        p.counters = static_cast<unsigned*>(ws);
        p.words = reinterpret_cast<unsigned long long*>(static_cast<char*>(ws) + kCounterBytes);
        p.partials = static_cast<char*>(ws) + kZeroBytes;
    }
    return p;
}

bool is_aligned(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return na != 0 && nb != 0 && a0 < b0 + nb && b0 < a0 + na;
}

// Capabilities of the current device, cached per ordinal.
rdx_status current_device(const DeviceCaps** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda("cudaGetDevice", e);
    std::lock_guard<std::mutex> lock(g_mu);
    auto it = g_caps.find(dev);
    if (it == g_caps.end()) {
        DeviceCaps c;
        c.ordinal = dev;
        if ((e = cudaDeviceGetAttribute(&c.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&c.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&c.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
            return fail_cuda("cudaDeviceGetAttribute", e);
        if (c.cc_major != 10 || c.cc_minor != 3) {
            t_last_error = "device " + std::to_string(dev) + " has compute capability " + std::to_string(c.cc_major) +
                           "." + std::to_string(c.cc_minor) + "; this library is built for sm_103a only";
            return RDX_ERR_UNSUPPORTED_DEVICE;
        }
        it = g_caps.emplace(dev, c).first;
    }
    *out = &it->second;  // map nodes are never erased: the pointer stays valid
    return RDX_OK;
}

// The (device, stream) workspace; allocated, its counters zeroed and its
// partial slots poisoned (in stream order) on first use.
rdx_status stream_workspace(const DeviceCaps& dev, cudaStream_t stream, void** out) {
    std::lock_guard<std::mutex> lock(g_mu);
    const size_t thread_key =
        stream == cudaStreamPerThread ? std::hash<std::thread::id>{}(std::this_thread::get_id()) | 1u : 0u;
    const auto key = std::make_tuple(dev.ordinal, reinterpret_cast<uintptr_t>(stream), thread_key);
    auto it = g_workspaces.find(key);
    if (it != g_workspaces.end()) {
        *out = it->second;
        return RDX_OK;
    }
    const char* inject = std::getenv("RDX_FAULT_ALLOC");
    if (inject != nullptr && inject[0] == '1') {
        t_last_error = "workspace allocation refused: RDX_FAULT_ALLOC=1";
        return RDX_ERR_ALLOC;
    }
    void* p = nullptr;
    cudaError_t e = cudaMalloc(&p, workspace_bytes());
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        t_last_error = std::string("cudaMalloc of the workspace: ") + cudaGetErrorString(e);
        return RDX_ERR_ALLOC;
    }
    e = cudaMemsetAsync(p, 0, kZeroBytes, stream);
    // Poison the partial slots (all-ones bytes: a NaN for float slots): a
    // partial read before it was written would show up in the result.
    if (e == cudaSuccess) e = cudaMemsetAsync(static_cast<char*>(p) + kZeroBytes, 0xFF,
                                              workspace_bytes() - kZeroBytes, stream);
    if (e != cudaSuccess) {
        cudaFree(p);
        return fail_cuda("cudaMemsetAsync of the workspace", e);
    }
    g_workspaces.emplace(key, p);
    *out = p;
    return RDX_OK;
}

bool valid_op(int op) { return op >= 0 && op < int(Op::kCount); }

// Checks shared by the scalar reductions.
rdx_status check_scalar(Op op, const void* x, int64_t n, const void* out) {
    const size_t es = rdx::reduce_elem_bytes(op), os = rdx::reduce_acc_bytes(op);
    if (n < 0 || out == nullptr || (n > 0 && x == nullptr)) return RDX_ERR_INVALID_ARG;
    if (n > INT64_MAX / 16) return RDX_ERR_INVALID_ARG;
    if (!is_aligned(x, es) || !is_aligned(out, os)) return RDX_ERR_INVALID_ARG;
    if (overlaps(x, size_t(n) * es, out, os)) return RDX_ERR_INVALID_ARG;
    return RDX_OK;
}

// One row of n elements; ws is the workspace (NULL when the plan has one tile).
rdx_status launch_scalar(Op op, const void* x, int64_t n, void* out, void* ws, cudaStream_t stream) {
    const rdx::ReducePlan plan = rdx::reduce_plan(op, 1, n);
    const WorkspaceParts w = parts_of(ws);
    const cudaError_t e = rdx::reduce_launch(op, x, 1, n, n, plan, w.partials, w.counters, w.words, out, stream);
    if (e != cudaSuccess) return fail_cuda("reduce kernel launch", e);
    return RDX_OK;
}

rdx_status reduce_entry(Op op, const void* x, int64_t n, void* out, cudaStream_t stream) {
    t_last_error.clear();
    rdx_status st = check_scalar(op, x, n, out);
    if (st != RDX_OK) return st;
    const DeviceCaps* dev = nullptr;
    if ((st = current_device(&dev)) != RDX_OK) return st;
    void* ws = nullptr;
    if (rdx::reduce_plan(op, 1, n).tiles > 1 && (st = stream_workspace(*dev, stream, &ws)) != RDX_OK) return st;
    return launch_scalar(op, x, n, out, ws, stream);
}

rdx_status rowsum_entry(const float* x, int64_t rows, int64_t cols, int64_t ld, float* out, cudaStream_t stream) {
    t_last_error.clear();
    if (rows < 0 || cols < 0 || ld < 0) return RDX_ERR_INVALID_ARG;
    if (rows > 1 && ld < cols) return RDX_ERR_INVALID_ARG;
    if (rows > INT64_MAX / 16 || cols > INT64_MAX / 16 || ld > INT64_MAX / 16) return RDX_ERR_INVALID_ARG;
    if (rows > 1 && rows - 1 > (INT64_MAX / 16 - cols) / (ld > 0 ? ld : 1)) return RDX_ERR_INVALID_ARG;
    if (rows > 0 && out == nullptr) return RDX_ERR_INVALID_ARG;
    if (rows > 0 && cols > 0 && x == nullptr) return RDX_ERR_INVALID_ARG;
    if (!is_aligned(x, 4) || !is_aligned(out, 4)) return RDX_ERR_INVALID_ARG;
    const size_t span = rows > 0 && cols > 0 ? (size_t(rows - 1) * size_t(ld) + size_t(cols)) * 4 : 0;
    if (overlaps(x, span, out, size_t(rows) * 4)) return RDX_ERR_INVALID_ARG;
    if (rows == 0) return RDX_OK;

    const DeviceCaps* dev = nullptr;
    rdx_status st = current_device(&dev);
    if (st != RDX_OK) return st;
    if (rdx::rowsum_use_split(rows, cols)) {
        // few long rows: each row over many blocks (tiles + a per-row finish)
        const rdx::ReducePlan plan = rdx::reduce_plan(Op::SumF32, rows, cols);
        void* ws = nullptr;
        if ((st = stream_workspace(*dev, stream, &ws)) != RDX_OK) return st;
        const WorkspaceParts w = parts_of(ws);
        const cudaError_t e =
            rdx::reduce_launch(Op::SumF32, x, rows, cols, ld, plan, w.partials, w.counters, nullptr, out, stream);
        if (e != cudaSuccess) return fail_cuda("split-row kernel launch", e);
        return RDX_OK;
    }
    const cudaError_t e = rdx::rowsum_launch(x, rows, cols, ld, out, stream);
    if (e != cudaSuccess) return fail_cuda("rowsum kernel launch", e);
    return RDX_OK;
}

}  // namespace

void rdx::set_last_error(const char* text) { t_last_error = text; }

extern "C" {

rdx_status rdx_sum_f32(const float* x, int64_t n, float* out, cudaStream_t stream) {
    return reduce_entry(Op::SumF32, x, n, out, stream);
}

rdx_status rdx_sumsq_f32(const float* x, int64_t n, float* out, cudaStream_t stream) {
    return reduce_entry(Op::SumSqF32, x, n, out, stream);
}

rdx_status rdx_sum_bf16_f32acc(const rdx_bf16* x, int64_t n, float* out, cudaStream_t stream) {
    return reduce_entry(Op::SumBF16, x, n, out, stream);
}

rdx_status rdx_sumsq_bf16_f32acc(const rdx_bf16* x, int64_t n, float* out, cudaStream_t stream) {
    return reduce_entry(Op::SumSqBF16, x, n, out, stream);
}

rdx_status rdx_sum_i32_i64(const int32_t* x, int64_t n, int64_t* out, cudaStream_t stream) {
    return reduce_entry(Op::SumI32, x, n, out, stream);
}

rdx_status rdx_sum_sumsq_f32(const float* x, int64_t n, float* out2, cudaStream_t stream) {
    return reduce_entry(Op::SumSumSqF32, x, n, out2, stream);
}

rdx_status rdx_sum_sumsq_bf16_f32acc(const rdx_bf16* x, int64_t n, float* out2, cudaStream_t stream) {
    return reduce_entry(Op::SumSumSqBF16, x, n, out2, stream);
}

rdx_status rdx_max_f32(const float* x, int64_t n, float* out, cudaStream_t stream) {
    return reduce_entry(Op::MaxF32, x, n, out, stream);
}

rdx_status rdx_max_i32(const int32_t* x, int64_t n, int32_t* out, cudaStream_t stream) {
    return reduce_entry(Op::MaxI32, x, n, out, stream);
}

size_t rdx_workspace_bytes(void) { return workspace_bytes(); }

int rdx_reduce_kernels(int op, int64_t n) {
    if (!valid_op(op) || n < 0) return -1;
    return rdx::reduce_plan(Op(op), 1, n).separate_finish ? 2 : 1;
}

int rdx_rowsum_kernels(int64_t rows, int64_t cols) {
    if (rows < 0 || cols < 0) return -1;
    if (rows == 0) return 0;
    if (!rdx::rowsum_use_split(rows, cols)) return 1;
    return rdx::reduce_plan(Op::SumF32, rows, cols).separate_finish ? 2 : 1;
}

rdx_status rdx_reduce_ws(int op, const void* x, int64_t n, void* out, void* workspace, size_t workspace_size,
                         cudaStream_t stream) {
    t_last_error.clear();
    if (!valid_op(op)) return RDX_ERR_INVALID_ARG;
    rdx_status st = check_scalar(Op(op), x, n, out);
    if (st != RDX_OK) return st;
    if (workspace == nullptr || workspace_size < workspace_bytes() || !is_aligned(workspace, 256))
        return RDX_ERR_INVALID_ARG;
    const size_t es = rdx::reduce_elem_bytes(Op(op)), os = rdx::reduce_acc_bytes(Op(op));
    if (overlaps(workspace, workspace_bytes(), x, size_t(n) * es) || overlaps(workspace, workspace_bytes(), out, os))
        return RDX_ERR_INVALID_ARG;
    const DeviceCaps* dev = nullptr;
    if ((st = current_device(&dev)) != RDX_OK) return st;
    return launch_scalar(Op(op), x, n, out, workspace, stream);
}

rdx_status rdx_rowsum_f32(const float* x, int64_t rows, int64_t cols, float* out, cudaStream_t stream) {
    return rowsum_entry(x, rows, cols, cols, out, stream);
}

rdx_status rdx_rowsum_strided_f32(const float* x, int64_t rows, int64_t cols, int64_t ld, float* out,
                                  cudaStream_t stream) {
    return rowsum_entry(x, rows, cols, ld, out, stream);
}

int64_t rdx_ladder_num_partials(int version, int64_t n) {
    if (version < 1 || version > 5 || n < 0) return -1;
    const int64_t seg = version <= 3 ? rdx::kLadderBlock : 2 * rdx::kLadderBlock;
    return n / seg + (n % seg != 0);
}

rdx_status rdx_ladder_partials_f32(int version, const float* x, int64_t n, float* partials,
                                   cudaStream_t stream) {
    t_last_error.clear();
    const int64_t blocks = rdx_ladder_num_partials(version, n);
    if (blocks < 0) return RDX_ERR_INVALID_ARG;
    if (blocks > 0x7fffffff) return RDX_ERR_INVALID_ARG;
    if (n > 0 && (x == nullptr || partials == nullptr)) return RDX_ERR_INVALID_ARG;
    if (!is_aligned(x, 4) || !is_aligned(partials, 4)) return RDX_ERR_INVALID_ARG;
    if (overlaps(x, size_t(n) * 4, partials, size_t(blocks) * 4)) return RDX_ERR_INVALID_ARG;
    if (blocks == 0) return RDX_OK;

    const DeviceCaps* dev = nullptr;
    const rdx_status st = current_device(&dev);
    if (st != RDX_OK) return st;
    const cudaError_t e = rdx::ladder_launch(version, x, n, partials, blocks, nullptr, nullptr, stream);
    if (e != cudaSuccess) return fail_cuda("ladder kernel launch", e);
    return RDX_OK;
}

rdx_status rdx_ladder_sum_f32(int version, const float* x, int64_t n, float* partials, float* out,
                              cudaStream_t stream) {
    t_last_error.clear();
    const int64_t blocks = rdx_ladder_num_partials(version, n);
    if (blocks < 0) return RDX_ERR_INVALID_ARG;
    if (blocks > 0x7fffffff) return RDX_ERR_INVALID_ARG;
    if (out == nullptr || (n > 0 && (x == nullptr || partials == nullptr))) return RDX_ERR_INVALID_ARG;
    if (!is_aligned(x, 4) || !is_aligned(partials, 4) || !is_aligned(out, 4)) return RDX_ERR_INVALID_ARG;
    const size_t xb = size_t(n) * 4, pb = size_t(blocks) * 4;
    if (overlaps(x, xb, partials, pb) || overlaps(x, xb, out, 4) || overlaps(partials, pb, out, 4))
        return RDX_ERR_INVALID_ARG;

    const DeviceCaps* dev = nullptr;
    rdx_status st = current_device(&dev);
    if (st != RDX_OK) return st;
    if (blocks == 0) {
        const cudaError_t e = cudaMemsetAsync(out, 0, sizeof(float), stream);
        return e == cudaSuccess ? RDX_OK : fail_cuda("cudaMemsetAsync of the result", e);
    }
    void* ws = nullptr;  // its first completion counter (stream order keeps users apart)
    if ((st = stream_workspace(*dev, stream, &ws)) != RDX_OK) return st;
    const cudaError_t e =
        rdx::ladder_launch(version, x, n, partials, blocks, static_cast<unsigned*>(ws), out, stream);
    if (e != cudaSuccess) return fail_cuda("ladder kernel launch", e);
    return RDX_OK;
}

rdx_status rdx_bank_probe(int pattern, int iters, int64_t* cycles, uint32_t* sink, cudaStream_t stream) {
    t_last_error.clear();
    if (pattern < 0 || pattern >= rdx::kBankPatterns || iters < 1 || iters > (1 << 20)) return RDX_ERR_INVALID_ARG;
    if (cycles == nullptr || sink == nullptr || !is_aligned(cycles, 8) || !is_aligned(sink, 4))
        return RDX_ERR_INVALID_ARG;
    if (overlaps(cycles, 8, sink, 32 * 4)) return RDX_ERR_INVALID_ARG;
    const DeviceCaps* dev = nullptr;
    const rdx_status st = current_device(&dev);
    if (st != RDX_OK) return st;
    const cudaError_t e = rdx::bank_probe_launch(pattern, iters, reinterpret_cast<long long*>(cycles),
                                                 reinterpret_cast<unsigned*>(sink), stream);
    if (e != cudaSuccess) return fail_cuda("bank probe launch", e);
    return RDX_OK;
}

int rdx_bank_probe_loads_per_iter(void) { return rdx::bank_probe_loads_per_iter(); }

rdx_status rdx_shard_range(int64_t n, int parts, int rank, int64_t granule, int64_t* lo, int64_t* hi) {
    t_last_error.clear();
    if (lo == nullptr || hi == nullptr || lo == hi) return RDX_ERR_INVALID_ARG;
    return rdx::shard_range(n, parts, rank, granule, lo, hi) ? RDX_OK : RDX_ERR_INVALID_ARG;
}

int rdx_combine_max_parts(void) { return rdx::kMaxCombineParts; }

}  // extern "C"

namespace {

rdx_status combine_entry(rdx::CombineType type, size_t bytes, const void* parts, int p, void* out,
                         cudaStream_t stream) {
    t_last_error.clear();
    if (parts == nullptr || out == nullptr || p < 1 || p > rdx::kMaxCombineParts) return RDX_ERR_INVALID_ARG;
    const size_t align = bytes == 4 ? 4 : 8;
    if (!is_aligned(parts, align) || !is_aligned(out, align)) return RDX_ERR_INVALID_ARG;
    if (overlaps(parts, size_t(p) * bytes, out, bytes)) return RDX_ERR_INVALID_ARG;
    const DeviceCaps* dev = nullptr;
    const rdx_status st = current_device(&dev);
    if (st != RDX_OK) return st;
    const cudaError_t e = rdx::combine_launch(type, parts, p, out, stream);
    if (e != cudaSuccess) return fail_cuda("combine kernel launch", e);
    return RDX_OK;
}

}  // namespace

extern "C" {

rdx_status rdx_combine_f32(const float* parts, int p, float* out, cudaStream_t stream) {
    return combine_entry(rdx::CombineType::F32, 4, parts, p, out, stream);
}

rdx_status rdx_combine_f32x2(const float* parts2, int p, float* out2, cudaStream_t stream) {
    return combine_entry(rdx::CombineType::F32x2, 8, parts2, p, out2, stream);
}

rdx_status rdx_combine_i64(const int64_t* parts, int p, int64_t* out, cudaStream_t stream) {
    return combine_entry(rdx::CombineType::I64, 8, parts, p, out, stream);
}

int rdx_debug_build(void) { return RDX_DEBUG ? 1 : 0; }

rdx_status rdx_debug_violations(uint64_t* count, int reset) {
    t_last_error.clear();
    if (count == nullptr) return RDX_ERR_INVALID_ARG;
    *count = 0;
    if (!RDX_DEBUG) return RDX_OK;
    const cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail_cuda("cudaDeviceSynchronize", e);
    const unsigned long long parts[4] = {rdx::reduce_out_of_range(reset != 0), rdx::rowsum_out_of_range(reset != 0),
                                         rdx::ladder_out_of_range(reset != 0), rdx::shard_out_of_range(reset != 0)};
    for (unsigned long long v : parts) {
        if (v == ~0ull) {
            t_last_error = "cudaMemcpyFromSymbol of a violation counter failed";
            return RDX_ERR_CUDA;
        }
        *count += v;
    }
    return RDX_OK;
}

rdx_status rdx_wait_timeouts(uint64_t* count, int reset) {
    t_last_error.clear();
    if (count == nullptr) return RDX_ERR_INVALID_ARG;
    *count = 0;
    const cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail_cuda("cudaDeviceSynchronize", e);
    const unsigned long long v = rdx::rowsum_stage_timeouts(reset != 0);
    if (v == ~0ull) {
        t_last_error = "cudaMemcpyFromSymbol of the staging-timeout counter failed";
        return RDX_ERR_CUDA;
    }
    *count = v;
    return RDX_OK;
}

rdx_status rdx_debug_stage_timeout(const float* x, int64_t rows, int64_t cols, float* out, cudaStream_t stream) {
    t_last_error.clear();
    if (x == nullptr || out == nullptr || cols <= 0 || cols >= 64 || rows <= 0 || rows > 6144 ||
        rows * cols > 6144 || rows * cols < 4 || !is_aligned(x, 16) || !is_aligned(out, 4))
        return RDX_ERR_INVALID_ARG;
    if (overlaps(x, size_t(rows * cols) * 4, out, size_t(rows) * 4)) return RDX_ERR_INVALID_ARG;
    const DeviceCaps* dev = nullptr;
    const rdx_status st = current_device(&dev);
    if (st != RDX_OK) return st;
    const cudaError_t e = rdx::rowsum_stage_timeout_probe(x, rows, cols, out, stream);
    if (e != cudaSuccess) return fail_cuda("staging-timeout probe launch", e);
    return RDX_OK;
}

const char* rdx_status_string(rdx_status status) {
    switch (status) {
        case RDX_OK: return "ok";
        case RDX_ERR_INVALID_ARG: return "invalid argument";
        case RDX_ERR_CUDA: return "CUDA error";
        case RDX_ERR_ALLOC: return "workspace allocation failed";
        case RDX_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs sm_103)";
        default: return "unknown status";
    }
}

const char* rdx_last_cuda_error(void) { return t_last_error.c_str(); }

void rdx_shutdown(void) {
    std::lock_guard<std::mutex> lock(g_mu);
    for (auto& kv : g_workspaces) cudaFree(kv.second);
    g_workspaces.clear();
}

int rdx_release_stream(cudaStream_t stream) {
    t_last_error.clear();
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    const size_t thread_key =
        stream == cudaStreamPerThread ? std::hash<std::thread::id>{}(std::this_thread::get_id()) | 1u : 0u;
    std::lock_guard<std::mutex> lock(g_mu);
    auto it = g_workspaces.find(std::make_tuple(dev, reinterpret_cast<uintptr_t>(stream), thread_key));
    if (it == g_workspaces.end()) return 0;
    cudaFree(it->second);
    g_workspaces.erase(it);
    return 1;
}

}  // extern "C"
