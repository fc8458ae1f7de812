// fa_noalloc.cu — fa_bwd_noalloc: the backward pass with its scratch memory built into
// the library, for callers that cannot allocate device memory themselves.
//
// fa_bwd needs a workspace (the fp32 dQ accumulator plus two per-row vectors) that its
// caller allocates.  Some callers have no way to do that:
//   * code running as a plugin or callback inside a host framework that owns all device
//     memory and hands the plugin only its input and output tensors, with no allocator;
//   * latency-critical loops that must not call cudaMalloc, which can synchronise the
//     whole device;
//   * processes that reserve a fixed device-memory budget at start-up and forbid
//     allocations afterwards.
// For them this entry point uses a file-scope device array of FA_NOALLOC_SCRATCH_BYTES
// (64 MiB) as the workspace.  The array belongs to the library's module: every GPU that
// loads the library holds it until the process exits.
//
// Set-up: the first call on each device, with that device current, looks up the
// array's device address with cudaGetSymbolAddress (the array's name in host code is
// only a host-side stand-in, not a device address) and caches it per device.  That
// first call should therefore come before any stream capture.  The stream must belong
// to the current device (checked; another device's stream is an argument error).
//
// Sharing: every call uses the same array, and the array keeps the previous call's
// contents.  The backward's pre-processing kernel rewrites every part of the workspace
// it later reads (it clears the dQ accumulator and writes both per-row vectors), so
// nothing needs clearing here.  Calls whose kernels overlap on the GPU (for example on
// two streams at once) race on the array.
//
// Nothing here calls cudaMalloc, cudaFree or any allocating routine.
#include <mutex>

#include "fa.h"
#include "fa_internal.h"

namespace {

constexpr size_t kScratchBytes = FA_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
struct ScratchSlot {
    bool ready = false;
    void *ptr = nullptr;
};
ScratchSlot g_scratch[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (looked up once per device).
int scratch_for_current_device(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return FA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchSlot &s = g_scratch[dev];
    if (!s.ready) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return FA_ERR_CUDA;
        if (major != 10 || minor != 3) return FA_ERR_UNSUPPORTED;
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_bwd_scratch);
        if (e != cudaSuccess || p == nullptr) return FA_ERR_CUDA;
        s.ptr = p;
        s.ready = true;
    }
    *out = s.ptr;
    return FA_OK;
}

}  // namespace

extern "C" int fa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o, const float *lse,
                              const void *dout, void *dq, void *dk, void *dv, int B, int H, int N, int d,
                              float scale, int causal, fa_stream_t stream) {
    if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
    const size_t need = fa_bwd_workspace_size(B, H, N, d);
    if (need == 0)  // invalid or unsupported shape: fa_bwd reports which, before using a workspace
        return fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, nullptr, 0, B, H, N, d, scale, causal, stream);
    if (need > kScratchBytes) return FA_ERR_WORKSPACE;
    // The array used is the current device's: a stream of another device would run the
    // kernels there against this device's address.
    int cur = 0, sdev = 0;
    if (cudaGetDevice(&cur) != cudaSuccess) return FA_ERR_CUDA;
    if (cudaStreamGetDevice(reinterpret_cast<cudaStream_t>(stream), &sdev) != cudaSuccess) return FA_ERR_CUDA;
    if (sdev != cur) return FA_ERR_INVALID_ARG;
    void *scratch = nullptr;
    const int st = scratch_for_current_device(&scratch);
    if (st != FA_OK) return st;
    return fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, scratch, kScratchBytes, B, H, N, d, scale, causal, stream);
}
