// f8_linear_fwd_noalloc: the Float8 linear forward pass for callers that
// cannot allocate device memory.
//
// f8_linear_fwd needs a caller-provided device workspace for the row-major
// E4M3 copies of X and W.  Some callers have no way to provide one: a plugin
// hosted by a framework that owns every device byte through its own pool and
// forbids side allocations, or a service whose device-memory budget is fixed
// when it starts.  This entry point takes that workspace from a file-scope
// device array instead, so the call itself allocates nothing.  It launches
// the same kernels as f8_linear_fwd, with the same arguments.
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

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

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
    if (M <= 0 || N <= 0 || K <= 0 || x == nullptr || w == nullptr || y == nullptr ||
        saved == nullptr || saved->x_t == nullptr || saved->w_t == nullptr ||
        saved->amax_x == nullptr || saved->scale_x == nullptr || saved->amax_w == nullptr ||
        saved->scale_w == nullptr)
        return F8_ERR_INVALID;
    if (M % 16 || N % 16 || K % 16 || M > INT32_MAX / 2 || N > INT32_MAX / 2 || K > INT32_MAX / 2)
        return F8_ERR_SHAPE;
    const size_t xq_bytes = round256(static_cast<size_t>(M) * static_cast<size_t>(K));
    const size_t wq_bytes = round256(static_cast<size_t>(N) * static_cast<size_t>(K));
    if (xq_bytes > kF8NoallocScratchBytes || wq_bytes > kF8NoallocScratchBytes - xq_bytes)
        return F8_ERR_SHAPE;  // the two E4M3 copies do not fit the static scratch
    if (!aligned(x, 16) || !aligned(w, 16) || !aligned(y, 16) || !aligned(saved->x_t, 16) ||
        !aligned(saved->w_t, 16) || !aligned(saved->amax_x, 4) || !aligned(saved->scale_x, 4) ||
        !aligned(saved->amax_w, 4) || !aligned(saved->scale_w, 4))
        return F8_ERR_ALIGN;

    const f8::DeviceInfo *dev = f8::device_info();
    if (dev == nullptr || dev->ordinal >= kMaxDevices)
        return F8_ERR_CUDA;
    if (dev->cc_major != 10 || dev->cc_minor != 3)
        return F8_ERR_UNSUPPORTED;
    uint8_t *scratch = scratch_on_current_device(dev->ordinal);
    if (scratch == nullptr)
        return F8_ERR_CUDA;
    uint8_t *x_q = scratch;
    uint8_t *w_q = scratch + xq_bytes;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = f8::launch_amax(x, M * K, saved->amax_x, *dev, st);
    if (e == cudaSuccess)
        e = f8::launch_amax(w, N * K, saved->amax_w, *dev, st);
    if (e == cudaSuccess)
        e = f8::launch_cast_transpose(x, M, K, saved->amax_x, nullptr, 0, nullptr, saved->scale_x,
                                      x_q, saved->x_t, 0, *dev, st);
    if (e == cudaSuccess)
        e = f8::launch_cast_transpose(w, N, K, saved->amax_w, nullptr, 0, nullptr, saved->scale_w,
                                      w_q, saved->w_t, 0, *dev, st);
    if (e == cudaSuccess)
        e = f8::launch_gemm(x_q, w_q, M, N, K, saved->scale_x, saved->scale_w, y, *dev, st);
    if (e == cudaErrorNotSupported)
        return F8_ERR_UNSUPPORTED;
    return e == cudaSuccess ? F8_OK : F8_ERR_CUDA;
}
