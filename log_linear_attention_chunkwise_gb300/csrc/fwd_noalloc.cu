// lla_fwd_noalloc: the forward without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they run
// the forward: code inside a custom allocator or memory-pool callback, a
// plugin that is handed only the input and output buffers, or a runtime
// that forbids cudaMalloc while it replays or records work.  For them this
// entry point takes its scratch from one fixed array that lives in the
// library's device image, instead of from a workspace argument.
//
// The array is kNoAllocScratchBytes (64 MiB) on every GPU that loads the
// library, held until the process exits.  The first call on a device looks
// up the array's device address (cudaGetSymbolAddress, with that device
// current) and caches it; make that first call before any stream capture.
// A look-up that fails is not cached: the call returns LLA_ERR_CUDA and the
// next call tries again.  The address belongs to the current device, so the
// stream must belong to it too (checked where the runtime can tell).
// All calls share the one array and it keeps the last call's contents, so
// calls that overlap on the GPU (different streams, no ordering between
// them) race and must not be issued.  The forward resets every piece of the
// scratch it relies on, so nothing needs to be cleared between calls.
#include <mutex>

#include "lla_common.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;
constexpr int kMaxDevices = 64;

// File-scope device scratch.  In host code `lla_noalloc_scratch` names a
// host-side shadow, not device memory: only the address returned by
// cudaGetSymbolAddress may be handed to a kernel.
__device__ __align__(256) unsigned char lla_noalloc_scratch[kNoAllocScratchBytes];

void *g_scratch_ptr[kMaxDevices];
std::mutex g_setup_mu;

// Device address of the scratch array on device `dev` (the current device);
// only a successful look-up is kept.
lla_status scratch_for_device(int dev, void **ptr)
{
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, lla_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();  // leave no sticky-looking error behind for the caller
            return LLA_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *ptr = g_scratch_ptr[dev];
    return LLA_OK;
}

}  // namespace

extern "C" {

size_t lla_fwd_noalloc_max_scratch_bytes(void) { return kNoAllocScratchBytes; }

lla_status lla_fwd_noalloc(const void *q, const void *k, const void *v, const float *g,
                           const float *lambda, void *out, int B, int H, int T, int dk, int dv,
                           int chunk, lla_dtype in_dt, lla_dtype out_dt, int32_t *device_error,
                           void *stream)
{
    // lla_fwd's own checks first, in its order, so that the status of a bad
    // call does not depend on which entry point it came through
    bool empty = false;
    lla_status st = lla::fwd_args_status(q, k, v, g, lambda, out, B, H, T, dk, dv, chunk, in_dt,
                                         out_dt, &empty);
    if (st != LLA_OK || empty) return st;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LLA_ERR_CUDA;
    int stream_dev = -1;
    if (cudaStreamGetDevice((cudaStream_t)stream, &stream_dev) == cudaSuccess) {
        if (stream_dev != dev) return LLA_ERR_INVALID_ARGUMENT;
    } else {
        cudaGetLastError();  // a runtime without the query: the documented duty stays the caller's
    }
    const size_t need = lla_fwd_workspace_bytes(B, H, T, dk, dv, chunk, in_dt);
    if (need > kNoAllocScratchBytes) return LLA_ERR_WORKSPACE_TOO_SMALL;
    void *scratch = nullptr;
    st = scratch_for_device(dev, &scratch);
    if (st != LLA_OK) return st;
    return lla_fwd(q, k, v, g, lambda, out, B, H, T, dk, dv, chunk, in_dt, out_dt, scratch,
                   kNoAllocScratchBytes, device_error, stream);
}

}  // extern "C"
