// api.cu -- the extern "C" entry points declared in include/rdx.h: argument
// validation (before any CUDA call), device capability cache, per-(device,
// stream) workspace cache, grid choice and launch.
#include "rdx.h"

#include <climits>
#include <cstdlib>
#include <map>
#include <mutex>
#include <string>
#include <utility>

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
std::map<std::pair<int, uintptr_t>, void*> g_workspaces;  // by (device, stream)

// Workspace layout: [completion counter, padded to 256 B][tile partials].
constexpr size_t kCounterBytes = 256;

size_t workspace_bytes() { return kCounterBytes + size_t(rdx::reduce_max_partials()) * 8; }

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
        if ((e = rdx::rowsum_blocks_per_sm(&c.rowsum_cta_bps, &c.rowsum_group_bps)) != cudaSuccess)
            return fail_cuda("cudaOccupancyMaxActiveBlocksPerMultiprocessor", e);
        it = g_caps.emplace(dev, c).first;
    }
    *out = &it->second;  // map nodes are never erased: the pointer stays valid
    return RDX_OK;
}

// The (device, stream) workspace; allocated and its counter zeroed (in
// stream order) on first use.
rdx_status stream_workspace(const DeviceCaps& dev, cudaStream_t stream, void** out) {
    std::lock_guard<std::mutex> lock(g_mu);
    const auto key = std::make_pair(dev.ordinal, reinterpret_cast<uintptr_t>(stream));
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
    e = cudaMemsetAsync(p, 0, kCounterBytes, stream);
    if (e != cudaSuccess) {
        cudaFree(p);
        return fail_cuda("cudaMemsetAsync of the completion counter", e);
    }
    g_workspaces.emplace(key, p);
    *out = p;
    return RDX_OK;
}

rdx_status reduce_entry(Op op, const void* x, int64_t n, void* out, cudaStream_t stream) {
    t_last_error.clear();
    const size_t es = rdx::reduce_elem_bytes(op), os = rdx::reduce_acc_bytes(op);
    if (n < 0 || out == nullptr || (n > 0 && x == nullptr)) return RDX_ERR_INVALID_ARG;
    if (n > INT64_MAX / 16) return RDX_ERR_INVALID_ARG;
    if (!is_aligned(x, es) || !is_aligned(out, os)) return RDX_ERR_INVALID_ARG;
    if (overlaps(x, size_t(n) * es, out, os)) return RDX_ERR_INVALID_ARG;

    const DeviceCaps* dev = nullptr;
    rdx_status st = current_device(&dev);
    if (st != RDX_OK) return st;

    const rdx::ReducePlan plan = rdx::reduce_plan(op, x, n);
    unsigned* counter = nullptr;
    void* partials = nullptr;
    if (plan.grid > 1) {
        void* ws = nullptr;
        if ((st = stream_workspace(*dev, stream, &ws)) != RDX_OK) return st;
        counter = static_cast<unsigned*>(ws);
        partials = static_cast<char*>(ws) + kCounterBytes;
    }
    const cudaError_t e = rdx::reduce_launch(op, x, n, plan, partials, counter, out, stream);
    if (e != cudaSuccess) return fail_cuda("reduce kernel launch", e);
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

rdx_status rdx_rowsum_f32(const float* x, int64_t rows, int64_t cols, float* out, cudaStream_t stream) {
    t_last_error.clear();
    if (rows < 0 || cols < 0) return RDX_ERR_INVALID_ARG;
    if (cols > 0 && rows > INT64_MAX / 16 / cols) return RDX_ERR_INVALID_ARG;
    if (rows > INT64_MAX / 16) return RDX_ERR_INVALID_ARG;
    if (rows > 0 && out == nullptr) return RDX_ERR_INVALID_ARG;
    if (rows > 0 && cols > 0 && x == nullptr) return RDX_ERR_INVALID_ARG;
    if (!is_aligned(x, 4) || !is_aligned(out, 4)) return RDX_ERR_INVALID_ARG;
    if (overlaps(x, size_t(rows) * size_t(cols) * 4, out, size_t(rows) * 4)) return RDX_ERR_INVALID_ARG;
    if (rows == 0) return RDX_OK;

    const DeviceCaps* dev = nullptr;
    const rdx_status st = current_device(&dev);
    if (st != RDX_OK) return st;
    const cudaError_t e = rdx::rowsum_launch(*dev, x, rows, cols, out, stream);
    if (e != cudaSuccess) return fail_cuda("rowsum kernel launch", e);
    return RDX_OK;
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
    const cudaError_t e = rdx::ladder_launch(version, x, n, partials, blocks, stream);
    if (e != cudaSuccess) return fail_cuda("ladder kernel launch", e);
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

}  // extern "C"
