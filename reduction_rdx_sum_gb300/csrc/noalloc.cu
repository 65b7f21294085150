// noalloc.cu -- rdx_sum_f32_noalloc: the float32 sum for callers that may not
// allocate device memory.
//
// rdx_sum_f32 keeps its block partials and completion counter in a workspace
// that the library cudaMallocs on the first call on each (device, stream).
// Some callers cannot let that happen:
//   * code embedded in a host framework or runtime that owns all device memory
//     through its own allocator: a cudaMalloc behind its back is not counted,
//     can fail once the framework has reserved the memory, and fragments it;
//   * latency-critical callers: cudaMalloc and cudaFree may synchronize the
//     device and take far longer than the reduction itself;
//   * callers whose memory budget is fixed at start-up and may not grow while
//     they run.
// This entry point runs the same kernel as rdx_sum_f32 (same grid, same
// summation order, so the same result) but takes its scratch from a
// fixed-size array in the library's static device memory instead.
//
// Scratch: kScratchBytes = 256-byte completion counter + kMaxPartials float32
// block partials (32 KiB + 256 B).  The array exists on every GPU that loads
// the library and stays there until the process exits.  All calls share it:
// the counter is cleared on the caller's stream before every launch, and two
// calls whose kernels run at the same time on the GPU (different streams, no
// ordering between them) race on it and give wrong results.
//
// Set-up: the first call on each device, with that device current, checks
// the device and looks up the device address of the array
// (cudaGetSymbolAddress).  Make that first call before any stream capture.
#include "rdx.h"

#include <climits>
#include <mutex>
#include <string>

#include "launch.h"

namespace {

// block partials the scratch holds: as many as any call of the tiled
// reductions uses, so the limit follows a build that changes the tiling
constexpr int64_t kMaxPartials = rdx::kReduceMaxTiles;
constexpr size_t kCounterBytes = 256;
constexpr size_t kScratchBytes = kCounterBytes + size_t(kMaxPartials) * sizeof(float);

// Device code could name this array directly; host code must use the address
// from cudaGetSymbolAddress (the host-side symbol is only a stand-in).
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

struct DeviceSetup {
    bool ready = false;
    void* scratch = nullptr;  // device address of g_noalloc_scratch on this device
    rdx::DeviceCaps caps;
};

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
DeviceSetup g_setup[kMaxDevices];

rdx_status fail(rdx_status status, const std::string& text) {
    rdx::set_last_error(text.c_str());
    return status;
}

rdx_status fail_cuda(const char* what, cudaError_t e) {
    return fail(RDX_ERR_CUDA, std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")");
}

// One-time set-up for the current device.
rdx_status setup_current_device(const DeviceSetup** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda("cudaGetDevice", e);
    if (dev < 0 || dev >= kMaxDevices) return fail(RDX_ERR_UNSUPPORTED_DEVICE, "device ordinal out of range");
    std::lock_guard<std::mutex> lock(g_setup_mu);
    DeviceSetup& s = g_setup[dev];
    if (!s.ready) {
        rdx::DeviceCaps c;
        c.ordinal = dev;
        if ((e = cudaDeviceGetAttribute(&c.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&c.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&c.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
            return fail_cuda("cudaDeviceGetAttribute", e);
        if (c.cc_major != 10 || c.cc_minor != 3)
            return fail(RDX_ERR_UNSUPPORTED_DEVICE, "this library is built for sm_103a only");
        void* p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_noalloc_scratch)) != cudaSuccess)
            return fail_cuda("cudaGetSymbolAddress of the static scratch", e);
        s.scratch = p;
        s.caps = c;
        s.ready = true;
    }
    *out = &s;
    return RDX_OK;
}

bool is_aligned(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return na != 0 && nb != 0 && a0 < b0 + nb && b0 < a0 + na;
}

}  // namespace

extern "C" rdx_status rdx_sum_f32_noalloc(const float* x, int64_t n, float* out, cudaStream_t stream) {
    rdx::set_last_error("");
    if (n < 0 || out == nullptr || (n > 0 && x == nullptr)) return RDX_ERR_INVALID_ARG;
    if (n > INT64_MAX / 16) return RDX_ERR_INVALID_ARG;
    if (!is_aligned(x, 4) || !is_aligned(out, 4)) return RDX_ERR_INVALID_ARG;
    if (overlaps(x, size_t(n) * 4, out, 4)) return RDX_ERR_INVALID_ARG;

    const DeviceSetup* s = nullptr;
    rdx_status st = setup_current_device(&s);
    if (st != RDX_OK) return st;

    const rdx::ReducePlan plan = rdx::reduce_plan(rdx::Op::SumF32, 1, n);
    if (plan.tiles > kMaxPartials)
        return fail(RDX_ERR_INVALID_ARG, "rdx_sum_f32_noalloc: this launch needs " + std::to_string(plan.tiles) +
                                             " block partials; the static scratch holds " +
                                             std::to_string(kMaxPartials));

    unsigned char* scratch = static_cast<unsigned char*>(s->scratch);
    cudaError_t e = cudaMemsetAsync(scratch, 0, kCounterBytes, stream);
    if (e != cudaSuccess) return fail_cuda("cudaMemsetAsync of the completion counter", e);
    e = rdx::reduce_launch(rdx::Op::SumF32, x, 1, n, n, plan, scratch + kCounterBytes,
                           reinterpret_cast<unsigned*>(scratch), nullptr, out, stream);
    if (e != cudaSuccess) return fail_cuda("reduce kernel launch", e);
    return RDX_OK;
}
