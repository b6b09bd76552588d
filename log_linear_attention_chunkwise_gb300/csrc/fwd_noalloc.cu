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
cudaError_t g_setup_err[kMaxDevices];
std::once_flag g_setup_once[kMaxDevices];

// Device address of the scratch array on the current device (set up once).
lla_status scratch_for_current_device(void **ptr)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LLA_ERR_CUDA;
    std::call_once(g_setup_once[dev], [dev]() {
        void *p = nullptr;
        g_setup_err[dev] = cudaGetSymbolAddress(&p, lla_noalloc_scratch);
        g_scratch_ptr[dev] = p;
    });
    if (g_setup_err[dev] != cudaSuccess || g_scratch_ptr[dev] == nullptr) return LLA_ERR_CUDA;
    *ptr = g_scratch_ptr[dev];
    return LLA_OK;
}

}  // namespace

extern "C" {

size_t lla_fwd_noalloc_max_scratch_bytes(void) { return kNoAllocScratchBytes; }

lla_status lla_fwd_noalloc(const void *q, const void *k, const void *v, const float *g,
                           const float *lambda, void *out, int B, int H, int T, int dk, int dv,
                           int chunk, lla_dtype in_dt, lla_dtype out_dt, void *stream)
{
    // shape and dtype errors come back from lla_fwd itself, before any launch
    const size_t need = lla_fwd_workspace_bytes(B, H, T, dk, dv, chunk, in_dt);
    if (need > kNoAllocScratchBytes) return LLA_ERR_WORKSPACE_TOO_SMALL;
    if (need == 0)  // empty or rejected: lla_fwd decides which, with no scratch
        return lla_fwd(q, k, v, g, lambda, out, B, H, T, dk, dv, chunk, in_dt, out_dt, nullptr, 0,
                       stream);
    void *scratch = nullptr;
    lla_status st = scratch_for_current_device(&scratch);
    if (st != LLA_OK) return st;
    return lla_fwd(q, k, v, g, lambda, out, B, H, T, dk, dv, chunk, in_dt, out_dt, scratch,
                   kNoAllocScratchBytes, stream);
}

}  // extern "C"
