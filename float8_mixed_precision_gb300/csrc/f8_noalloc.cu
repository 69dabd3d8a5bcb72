// f8_linear_fwd_noalloc: the Float8 linear forward pass for callers that
// cannot allocate device memory.
//
// f8_linear_fwd needs a caller-provided device workspace (the row-major
// E4M3 copies of X and W and the amax launches' partial maxima).  Some
// callers have no way to provide one: a plugin hosted by a framework that
// owns every device byte through its own pool and forbids side allocations,
// or a service whose device-memory budget is fixed when it starts.  This
// entry point takes that workspace from a file-scope device array instead,
// so the call itself allocates nothing.  It then runs f8_linear_fwd's own
// code (linear_fwd_impl) with that array as the workspace: the same checks,
// the same kernels and the same arguments.
//
// Costs and limits:
//  - the array is kF8NoallocScratchBytes (64 MiB) and lives in every device
//    that loads this library, until the process exits;
//  - every call shares it: two calls whose work overlaps on the GPU (on
//    different streams, or from different threads without ordering) race on
//    it and may both produce wrong results; calls on one stream are ordered
//    and safe.  Nothing in the array needs to start at zero: each call
//    overwrites the bytes it reads;
//  - the first call on each device looks up the array's device address
//    (cudaGetSymbolAddress) with that device current; make that first call
//    before any stream capture.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "f8.h"
#include "f8_internal.h"

namespace {

constexpr size_t kF8NoallocScratchBytes = F8_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kF8NoallocScratchBytes];

std::mutex g_scratch_mutex;
uint8_t *g_scratch_ptr[kMaxDevices];

// Device address of g_noalloc_scratch on the current device (looked up once
// per device; in host code the symbol itself is only a stand-in).
uint8_t *scratch_on_current_device(int dev)
{
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess)
            return nullptr;
        g_scratch_ptr[dev] = static_cast<uint8_t *>(p);
    }
    return g_scratch_ptr[dev];
}

} // namespace

extern "C" f8_status f8_linear_fwd_noalloc(const void *x, const void *w, int64_t M, int64_t N,
                                           int64_t K, void *y, const f8_linear_saved *saved,
                                           void *stream)
{
    f8_status st = f8::check_linear_shape(M, N, K);
    if (st != F8_OK)
        return st;
    st = f8::check_saved(saved);
    if (st != F8_OK)
        return st;
    if (x == nullptr || w == nullptr || y == nullptr)
        return F8_ERR_INVALID;
    if (f8::linear_fwd_ws_bytes(M, N, K) > kF8NoallocScratchBytes)
        return F8_ERR_SHAPE;  // the workspace does not fit the static array
    const f8::DeviceInfo *dev = f8::device_info();
    if (dev == nullptr || dev->ordinal >= kMaxDevices)
        return F8_ERR_CUDA;
    if (dev->cc_major != 10 || dev->cc_minor != 3)
        return F8_ERR_UNSUPPORTED;
    uint8_t *scratch = scratch_on_current_device(dev->ordinal);
    if (scratch == nullptr)
        return F8_ERR_CUDA;
    return f8::linear_fwd_impl(x, w, M, N, K, y, saved, scratch, kF8NoallocScratchBytes,
                               static_cast<cudaStream_t>(stream));
}
