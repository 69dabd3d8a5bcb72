// C-ABI of libf8: argument checks on the host, per-device state, the
// device status word, and the forward / backward composition of a Float8
// linear out of the amax, cast_transpose and GEMM launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "f8.h"
#include "f8_internal.h"
#include "f8_ptx.cuh"

// One status word per device (each device that loads the module gets its
// own instance); kernels OR error bits into it.
__device__ unsigned g_f8_status_word;

namespace f8 {
std::atomic<unsigned long long> g_kernel_launches{0};
} // namespace f8

namespace f8 {
namespace {

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;

std::mutex g_dev_mutex;
DeviceInfo g_dev[kMaxDevices];
bool g_dev_ready[kMaxDevices];
std::atomic<uint64_t> g_wait_limit_ns{kDefaultWaitLimitNs};

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

f8_status from_cuda(cudaError_t e)
{
    if (e == cudaSuccess)
        return F8_OK;
    if (e == cudaErrorNotSupported)
        return F8_ERR_UNSUPPORTED;
    return F8_ERR_CUDA;
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// The GEMM kernels number the output tiles of a launch (128 x 256 at the
// smallest) in 32-bit ints.
bool tiles_fit(int64_t M, int64_t N) { return ((M + 127) / 128) * ((N + 255) / 256) <= INT32_MAX / 2; }

// Workspace of the forward pass: q(X) [M,K], q(W) [N,K], then the amax
// partial maxima of X and of W.  Of the backward pass: q(dY) [M,N],
// q(dY)^T [N,M], amax and scale of dY, then the partial maxima of dY.
constexpr size_t kPartialsBytes = sizeof(unsigned) * kMaxAmaxPartials;
// X + W (bf16) up to which f8_linear_fwd quantises the two in shared launches
constexpr int64_t kPairMaxBytes = 112ll << 20;

struct FwdWs {
    uint8_t *x_q;
    uint8_t *w_q;
    unsigned *parts_x;
    unsigned *parts_w;
};
struct BwdWs {
    uint8_t *dy_q;
    uint8_t *dy_t;
    float *amax_dy;
    float *scale_dy;
    unsigned *parts_dy;
};

size_t fwd_ws_bytes(int64_t M, int64_t N, int64_t K)
{
    return round256(static_cast<size_t>(M) * K) + round256(static_cast<size_t>(N) * K) +
           2 * kPartialsBytes;
}

size_t bwd_ws_bytes(int64_t M, int64_t N)
{
    return 2 * round256(static_cast<size_t>(M) * N) + 256 + kPartialsBytes;
}

FwdWs fwd_ws(void *workspace, int64_t M, int64_t N, int64_t K)
{
    uint8_t *p = static_cast<uint8_t *>(workspace);
    FwdWs w;
    w.x_q = p;
    p += round256(static_cast<size_t>(M) * K);
    w.w_q = p;
    p += round256(static_cast<size_t>(N) * K);
    w.parts_x = reinterpret_cast<unsigned *>(p);
    w.parts_w = reinterpret_cast<unsigned *>(p + kPartialsBytes);
    return w;
}

BwdWs bwd_ws(void *workspace, int64_t M, int64_t N)
{
    uint8_t *p = static_cast<uint8_t *>(workspace);
    const size_t mn = round256(static_cast<size_t>(M) * N);
    BwdWs w;
    w.dy_q = p;
    w.dy_t = p + mn;
    w.amax_dy = reinterpret_cast<float *>(p + 2 * mn);
    w.scale_dy = reinterpret_cast<float *>(p + 2 * mn + 128);
    w.parts_dy = reinterpret_cast<unsigned *>(p + 2 * mn + 256);
    return w;
}

// Quantisation of n tensors in launch pairs: consecutive tensors go into
// one multi-tensor pair while their bf16 total stays within `budget` bytes
// (the amax pass's reads then still sit in L2 when the cast re-reads
// them); a tensor beyond it, or one the TMA cast cannot take, gets a pair
// of its own.  `parts` holds kMaxAmaxPartials partial maxima; the batches
// reuse it one after the other (each amax launch waits for the cast before
// it).
cudaError_t quantize_batches(const QuantDesc *d, int n, int fmt, unsigned *parts, int64_t budget,
                             const DeviceInfo &dev, cudaStream_t st)
{
    int i = 0;
    while (i < n) {
        int j = i;
        int64_t bytes = 0;
        while (j < n && quantize_multi_castable(&d[j], 1) &&
               (j == i || bytes + 2 * d[j].rows * d[j].cols <= budget) && j - i < kMaxQuantTensors) {
            bytes += 2 * d[j].rows * d[j].cols;
            ++j;
            if (bytes > budget)
                break;
        }
        cudaError_t e;
        if (j - i >= 2) {
            e = launch_quantize_multi(&d[i], j - i, fmt, parts, dev, st);
        } else {
            j = i + 1;
            int np = 0;
            e = launch_amax_partials(d[i].x, d[i].rows * d[i].cols, parts, &np, dev, st);
            if (e == cudaSuccess)
                e = launch_cast_transpose(d[i].x, d[i].rows, d[i].cols, nullptr, parts, np,
                                          d[i].amax_out, d[i].scale_out, d[i].q, d[i].q_t, fmt, dev,
                                          st, true);
        }
        if (e != cudaSuccess)
            return e;
        i = j;
    }
    return cudaSuccess;
}

// The backward GEMMs of a linear from q(dY) (format fdy) and the saved
// q(X)^T, q(W)^T; both in one launch when both are wanted:
//   dX [M,K] = q(dY) [M,N] . (q(W)^T [K,N])^T
//   dW [N,K] = q(dY)^T [N,M] . (q(X)^T [K,M])^T
cudaError_t launch_bwd_gemms(const BwdWs &bw, const f8_linear_saved *saved, int64_t M, int64_t N,
                             int64_t K, int fdy, void *dx, void *dw, const DeviceInfo &dev,
                             cudaStream_t st)
{
    const GemmDesc gdx{bw.dy_q, saved->w_t, M, K, N, bw.scale_dy, saved->scale_w, dx,
                       fdy, F8_E4M3};
    const GemmDesc gdw{bw.dy_t, saved->x_t, N, K, M, bw.scale_dy, saved->scale_x, dw,
                       fdy, F8_E4M3};
    if (dx != nullptr && dw != nullptr)
        return launch_gemm2(gdx, gdw, dev, st);
    const GemmDesc &g = dx != nullptr ? gdx : gdw;
    if (g.c == nullptr)
        return cudaSuccess;
    return launch_gemm(g.a, g.b, g.M, g.N, g.K, g.sa, g.sb, g.c, dev, st, g.fa, g.fb);
}

} // namespace

namespace {

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);

CtxGetCurrentFn ctx_get_current_fn()
{
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
    });
    return fn;
}

// A host thread that has made no context-bound CUDA call yet has no
// current context, and the driver calls the library makes itself (the
// tensor-map encoder) would fail in it.  Such a thread gets the current
// device's primary context, as the runtime's own first launch would bind
// it; a context the caller made current is left alone.
void ensure_context(int dev)
{
    const CtxGetCurrentFn fn = ctx_get_current_fn();
    CUcontext c = nullptr;
    if (fn != nullptr && fn(&c) == CUDA_SUCCESS && c == nullptr)
        cudaSetDevice(dev);
}

} // namespace

const DeviceInfo *device_info()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return nullptr;
    ensure_context(dev);
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (!g_dev_ready[dev]) {
        DeviceInfo info;
        info.ordinal = dev;
        if (cudaDeviceGetAttribute(&info.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&info.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&info.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return nullptr;
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_f8_status_word) != cudaSuccess)
            return nullptr;
        info.status = static_cast<unsigned *>(p);
        g_dev[dev] = info;
        g_dev_ready[dev] = true;
    }
    return &g_dev[dev];
}

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

f8_status check_linear_shape(int64_t M, int64_t N, int64_t K)
{
    if (M <= 0 || N <= 0 || K <= 0)
        return F8_ERR_INVALID;
    if (M % 16 || N % 16 || K % 16)
        return F8_ERR_SHAPE;
    if (M > INT32_MAX / 2 || N > INT32_MAX / 2 || K > INT32_MAX / 2)
        return F8_ERR_SHAPE;
    // Y [M,N], dX [M,K], dW [N,K]
    if (!tiles_fit(M, N) || !tiles_fit(M, K) || !tiles_fit(N, K))
        return F8_ERR_SHAPE;
    return F8_OK;
}

f8_status check_saved(const f8_linear_saved *s)
{
    if (s == nullptr || s->x_t == nullptr || s->w_t == nullptr || s->amax_x == nullptr ||
        s->scale_x == nullptr || s->amax_w == nullptr || s->scale_w == nullptr)
        return F8_ERR_INVALID;
    if (!aligned(s->x_t, 16) || !aligned(s->w_t, 16) || !aligned(s->amax_x, 4) ||
        !aligned(s->scale_x, 4) || !aligned(s->amax_w, 4) || !aligned(s->scale_w, 4))
        return F8_ERR_ALIGN;
    return F8_OK;
}

size_t linear_fwd_ws_bytes(int64_t M, int64_t N, int64_t K) { return fwd_ws_bytes(M, N, K); }

} // namespace f8

using namespace f8;

namespace {

// The kernels are built for sm_103a only; refuse anything else up front.
f8_status get_device(const DeviceInfo **out)
{
    const DeviceInfo *d = device_info();
    if (d == nullptr)
        return F8_ERR_CUDA;
    if (d->cc_major != 10 || d->cc_minor != 3)
        return F8_ERR_UNSUPPORTED;
    *out = d;
    return F8_OK;
}

f8_status check_cast_args(const void *x, int64_t rows, int64_t cols, const float *amax,
                          const float *scale_out, const uint8_t *q, const uint8_t *q_t)
{
    if (rows < 0 || cols < 0 || amax == nullptr)
        return F8_ERR_INVALID;
    if (rows > 0 && cols > 0 && x == nullptr)
        return F8_ERR_INVALID;
    if (!aligned(x, 16) || !aligned(q, 16) || !aligned(q_t, 16) || !aligned(amax, 4) ||
        !aligned(scale_out, 4))
        return F8_ERR_ALIGN;
    return F8_OK;
}


f8_status check_gemm_args(const uint8_t *a, const uint8_t *b, int64_t M, int64_t N, int64_t K,
                          const float *sa, const float *sb, const void *c)
{
    if (M < 0 || N < 0 || K < 0 || sa == nullptr || sb == nullptr)
        return F8_ERR_INVALID;
    if (M > INT32_MAX / 2 || N > INT32_MAX / 2 || K > INT32_MAX / 2)
        return F8_ERR_SHAPE;
    if (!tiles_fit(M, N))
        return F8_ERR_SHAPE;
    if (M > 0 && N > 0 && (c == nullptr || (K > 0 && (a == nullptr || b == nullptr))))
        return F8_ERR_INVALID;
    if (K % 16 != 0)
        return F8_ERR_SHAPE;
    if (!aligned(a, 16) || !aligned(b, 16) || !aligned(c, 16) || !aligned(sa, 4) || !aligned(sb, 4))
        return F8_ERR_ALIGN;
    return F8_OK;
}

#define F8_TRY(expr)                                                                               \
    do {                                                                                           \
        f8_status st_ = (expr);                                                                    \
        if (st_ != F8_OK)                                                                          \
            return st_;                                                                            \
    } while (0)

#define F8_TRY_CUDA(expr) F8_TRY(from_cuda(expr))

} // namespace

f8_status f8::linear_fwd_impl(const void *x, const void *w, int64_t M, int64_t N, int64_t K,
                              void *y, const f8_linear_saved *saved, void *workspace,
                              size_t workspace_bytes, cudaStream_t st)
{
    F8_TRY(check_linear_shape(M, N, K));
    F8_TRY(check_saved(saved));
    if (x == nullptr || w == nullptr || y == nullptr || workspace == nullptr)
        return F8_ERR_INVALID;
    if (workspace_bytes < fwd_ws_bytes(M, N, K))
        return F8_ERR_INVALID;
    if (!aligned(x, 16) || !aligned(w, 16) || !aligned(y, 16) || !aligned(workspace, 256))
        return F8_ERR_ALIGN;
    const DeviceInfo *dev;
    F8_TRY(get_device(&dev));
    const FwdWs fw = fwd_ws(workspace, M, N, K);
    // X and W together when they fit in L2 with room to spare (the cast
    // re-reads what the amax launch just read): two launches instead of
    // four; otherwise each cast follows its own amax
    const QuantDesc xw[2] = {{x, M, K, saved->amax_x, saved->scale_x, fw.x_q, saved->x_t},
                             {w, N, K, saved->amax_w, saved->scale_w, fw.w_q, saved->w_t}};
    F8_TRY_CUDA(quantize_batches(xw, 2, F8_E4M3, fw.parts_x,
                                 quant_pair_enabled() ? quant_batch_bytes(kPairMaxBytes) : 0, *dev,
                                 st));
    return from_cuda(launch_gemm(fw.x_q, fw.w_q, M, N, K, saved->scale_x, saved->scale_w, y, *dev, st));
}

extern "C" {

const char *f8_status_string(f8_status s)
{
    switch (s) {
    case F8_OK: return "F8_OK";
    case F8_ERR_INVALID: return "F8_ERR_INVALID: invalid argument";
    case F8_ERR_ALIGN: return "F8_ERR_ALIGN: misaligned pointer";
    case F8_ERR_SHAPE: return "F8_ERR_SHAPE: unsupported shape";
    case F8_ERR_CUDA: return "F8_ERR_CUDA: CUDA runtime error";
    case F8_ERR_TIMEOUT: return "F8_ERR_TIMEOUT: device wait exceeded its time limit";
    case F8_ERR_NONFINITE: return "F8_ERR_NONFINITE: non-finite value in an amax input";
    case F8_ERR_UNSUPPORTED: return "F8_ERR_UNSUPPORTED: needs an sm_103 device and driver";
    case F8_ERR_BOUNDS: return "F8_ERR_BOUNDS: an index left its buffer (checked build)";
    }
    return "F8_ERR_UNKNOWN";
}

void f8_set_wait_limit_ns(uint64_t limit_ns)
{
    g_wait_limit_ns.store(limit_ns ? limit_ns : kDefaultWaitLimitNs, std::memory_order_relaxed);
}

f8_status f8_amax(const void *x, int64_t n, float *amax_out, void *stream)
{
    if (n < 0 || amax_out == nullptr || (n > 0 && x == nullptr))
        return F8_ERR_INVALID;
    if (!aligned(x, 16) || !aligned(amax_out, 4))
        return F8_ERR_ALIGN;
    const DeviceInfo *dev;
    F8_TRY(get_device(&dev));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (n == 0)
        return from_cuda(cudaMemsetAsync(amax_out, 0, sizeof(float), st));
    return from_cuda(launch_amax(x, n, amax_out, *dev, st));
}

f8_status f8_cast_transpose(const void *x, int64_t rows, int64_t cols, const float *amax,
                            float *scale_out, uint8_t *q, uint8_t *q_t, void *stream)
{
    F8_TRY(check_cast_args(x, rows, cols, amax, scale_out, q, q_t));
    const DeviceInfo *dev;
    F8_TRY(get_device(&dev));
    return from_cuda(launch_cast_transpose(x, rows, cols, amax, nullptr, 0, nullptr, scale_out, q,
                                           q_t, 0, *dev, static_cast<cudaStream_t>(stream)));
}

size_t f8_quantize_workspace_bytes(void) { return kPartialsBytes; }

static f8_status quantize_impl(const void *x, int64_t rows, int64_t cols, int fmt, float *amax_out,
                               float *scale_out, uint8_t *q, uint8_t *q_t, void *workspace,
                               size_t workspace_bytes, void *stream)
{
    if (rows < 0 || cols < 0 || amax_out == nullptr || workspace == nullptr ||
        (rows > 0 && cols > 0 && x == nullptr) || (fmt != F8_E4M3 && fmt != F8_E5M2))
        return F8_ERR_INVALID;
    if (workspace_bytes < kPartialsBytes)
        return F8_ERR_INVALID;
    if (!aligned(x, 16) || !aligned(q, 16) || !aligned(q_t, 16) || !aligned(amax_out, 4) ||
        !aligned(scale_out, 4) || !aligned(workspace, 16))
        return F8_ERR_ALIGN;
    const DeviceInfo *dev;
    F8_TRY(get_device(&dev));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned *parts = static_cast<unsigned *>(workspace);
    int np = 0;
    F8_TRY_CUDA(launch_amax_partials(x, rows * cols, parts, &np, *dev, st));
    return from_cuda(launch_cast_transpose(x, rows, cols, nullptr, parts, np, amax_out, scale_out,
                                           q, q_t, fmt, *dev, st, true));
}

f8_status f8_quantize(const void *x, int64_t rows, int64_t cols, float *amax_out,
                      float *scale_out, uint8_t *q, uint8_t *q_t, void *workspace,
                      size_t workspace_bytes, void *stream)
{
    return quantize_impl(x, rows, cols, F8_E4M3, amax_out, scale_out, q, q_t, workspace,
                         workspace_bytes, stream);
}

f8_status f8_quantize_fmt(const void *x, int64_t rows, int64_t cols, f8_format fmt,
                          float *amax_out, float *scale_out, uint8_t *q, uint8_t *q_t,
                          void *workspace, size_t workspace_bytes, void *stream)
{
    return quantize_impl(x, rows, cols, fmt, amax_out, scale_out, q, q_t, workspace,
                         workspace_bytes, stream);
}

static f8_status gemm_impl(const uint8_t *a, int fa, const uint8_t *b, int fb, int64_t M, int64_t N,
                           int64_t K, const float *scale_a, const float *scale_b, void *c,
                           void *stream)
{
    if ((fa != F8_E4M3 && fa != F8_E5M2) || (fb != F8_E4M3 && fb != F8_E5M2))
        return F8_ERR_INVALID;
    F8_TRY(check_gemm_args(a, b, M, N, K, scale_a, scale_b, c));
    const DeviceInfo *dev;
    F8_TRY(get_device(&dev));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (M == 0 || N == 0)
        return F8_OK;
    if (K == 0)
        return from_cuda(cudaMemsetAsync(c, 0, static_cast<size_t>(M) * N * 2, st));
    return from_cuda(launch_gemm(a, b, M, N, K, scale_a, scale_b, c, *dev, st, fa, fb));
}

f8_status f8_gemm(const uint8_t *a, const uint8_t *b, int64_t M, int64_t N, int64_t K,
                  const float *scale_a, const float *scale_b, void *c, void *stream)
{
    return gemm_impl(a, F8_E4M3, b, F8_E4M3, M, N, K, scale_a, scale_b, c, stream);
}

f8_status f8_gemm_fmt(const uint8_t *a, f8_format fmt_a, const uint8_t *b, f8_format fmt_b,
                      int64_t M, int64_t N, int64_t K, const float *scale_a, const float *scale_b,
                      void *c, void *stream)
{
    return gemm_impl(a, fmt_a, b, fmt_b, M, N, K, scale_a, scale_b, c, stream);
}

f8_status f8_gemm_grouped(const f8_gemm_problem *problems, int count, void *stream)
{
    if (problems == nullptr || count < 1 || count > F8_MAX_GROUPED_GEMMS)
        return F8_ERR_INVALID;
    bool separate = count == 1;
    for (int i = 0; i < count; ++i) {
        const f8_gemm_problem &p = problems[i];
        if ((p.fmt_a != F8_E4M3 && p.fmt_a != F8_E5M2) ||
            (p.fmt_b != F8_E4M3 && p.fmt_b != F8_E5M2))
            return F8_ERR_INVALID;
        F8_TRY(check_gemm_args(p.a, p.b, p.M, p.N, p.K, p.scale_a, p.scale_b, p.c));
        if (p.M == 0 || p.N == 0 || p.K == 0)
            separate = true;
    }
    if (separate) {
        for (int i = 0; i < count; ++i) {
            const f8_gemm_problem &p = problems[i];
            F8_TRY(gemm_impl(p.a, p.fmt_a, p.b, p.fmt_b, p.M, p.N, p.K, p.scale_a, p.scale_b, p.c,
                             stream));
        }
        return F8_OK;
    }
    const DeviceInfo *dev;
    F8_TRY(get_device(&dev));
    GemmDesc g[F8_MAX_GROUPED_GEMMS];
    for (int i = 0; i < count; ++i) {
        const f8_gemm_problem &p = problems[i];
        g[i] = GemmDesc{p.a, p.b, p.M, p.N, p.K, p.scale_a, p.scale_b, p.c, p.fmt_a, p.fmt_b};
    }
    return from_cuda(launch_gemm_multi(g, count, *dev, static_cast<cudaStream_t>(stream)));
}

size_t f8_quantize_multi_workspace_bytes(void) { return kPartialsBytes; }

static f8_status check_quant_tensor(const f8_quant_tensor &t)
{
    if (t.rows < 0 || t.cols < 0 || t.amax_out == nullptr || (t.rows > 0 && t.cols > 0 && t.x == nullptr))
        return F8_ERR_INVALID;
    if (!aligned(t.x, 16) || !aligned(t.q, 16) || !aligned(t.q_t, 16) || !aligned(t.amax_out, 4) ||
        !aligned(t.scale_out, 4))
        return F8_ERR_ALIGN;
    return F8_OK;
}

f8_status f8_quantize_multi(const f8_quant_tensor *tensors, int count, f8_format fmt,
                            void *workspace, size_t workspace_bytes, void *stream)
{
    if (tensors == nullptr || count < 1 || count > F8_MAX_MULTI_TENSORS || workspace == nullptr ||
        (fmt != F8_E4M3 && fmt != F8_E5M2))
        return F8_ERR_INVALID;
    if (workspace_bytes < kPartialsBytes)
        return F8_ERR_INVALID;
    if (!aligned(workspace, 16))
        return F8_ERR_ALIGN;
    for (int i = 0; i < count; ++i)
        F8_TRY(check_quant_tensor(tensors[i]));
    const DeviceInfo *dev;
    F8_TRY(get_device(&dev));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    QuantDesc d[F8_MAX_MULTI_TENSORS];
    for (int i = 0; i < count; ++i) {
        const f8_quant_tensor &t = tensors[i];
        d[i] = QuantDesc{t.x, t.rows, t.cols, t.amax_out, t.scale_out, t.q, t.q_t};
    }
    return from_cuda(quantize_batches(d, count, fmt, static_cast<unsigned *>(workspace),
                                      quant_batch_bytes(kPairMaxBytes), *dev, st));
}

size_t f8_linear_workspace_bytes(int64_t M, int64_t N, int64_t K)
{
    if (M <= 0 || N <= 0 || K <= 0)
        return 0;
    size_t f = fwd_ws_bytes(M, N, K), b = bwd_ws_bytes(M, N);
    return f > b ? f : b;
}

f8_status f8_linear_fwd(const void *x, const void *w, int64_t M, int64_t N, int64_t K, void *y,
                        const f8_linear_saved *saved, void *workspace, size_t workspace_bytes,
                        void *stream)
{
    return linear_fwd_impl(x, w, M, N, K, y, saved, workspace, workspace_bytes,
                           static_cast<cudaStream_t>(stream));
}

static f8_status linear_bwd_impl(const void *dy, int fdy, const f8_linear_saved *saved, int64_t M,
                                 int64_t N, int64_t K, void *dx, void *dw, void *workspace,
                                 size_t workspace_bytes, void *stream)
{
    if (fdy != F8_E4M3 && fdy != F8_E5M2)
        return F8_ERR_INVALID;
    F8_TRY(check_linear_shape(M, N, K));
    F8_TRY(check_saved(saved));
    if (dy == nullptr || workspace == nullptr)
        return F8_ERR_INVALID;
    if (workspace_bytes < bwd_ws_bytes(M, N))
        return F8_ERR_INVALID;
    if (!aligned(dy, 16) || !aligned(dx, 16) || !aligned(dw, 16) || !aligned(workspace, 256))
        return F8_ERR_ALIGN;
    const DeviceInfo *dev;
    F8_TRY(get_device(&dev));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const BwdWs bw = bwd_ws(workspace, M, N);
    int np = 0;
    F8_TRY_CUDA(launch_amax_partials(dy, M * N, bw.parts_dy, &np, *dev, st));
    F8_TRY_CUDA(launch_cast_transpose(dy, M, N, nullptr, bw.parts_dy, np, bw.amax_dy, bw.scale_dy,
                                      dx ? bw.dy_q : nullptr, dw ? bw.dy_t : nullptr, fdy, *dev, st,
                                      true));
    return from_cuda(launch_bwd_gemms(bw, saved, M, N, K, fdy, dx, dw, *dev, st));
}

f8_status f8_linear_bwd(const void *dy, const f8_linear_saved *saved, int64_t M, int64_t N,
                        int64_t K, void *dx, void *dw, void *workspace, size_t workspace_bytes,
                        void *stream)
{
    return linear_bwd_impl(dy, F8_E4M3, saved, M, N, K, dx, dw, workspace, workspace_bytes, stream);
}

f8_status f8_linear_bwd_fmt(const void *dy, f8_format fmt_dy, const f8_linear_saved *saved,
                            int64_t M, int64_t N, int64_t K, void *dx, void *dw, void *workspace,
                            size_t workspace_bytes, void *stream)
{
    return linear_bwd_impl(dy, fmt_dy, saved, M, N, K, dx, dw, workspace, workspace_bytes, stream);
}

// Workspace of a group forward: q(X) [M, K], q(W_i) [N_i, K], partial
// maxima.  Of a group backward: per member q(dY_i) [M, N_i], q(dY_i)^T and
// 256 bytes of scalars (amax, scale), then partial maxima.
static size_t group_fwd_ws_bytes(int64_t M, int64_t K, const int64_t *N, int count)
{
    size_t b = round256(static_cast<size_t>(M) * K) + kPartialsBytes;
    for (int i = 0; i < count; ++i)
        b += round256(static_cast<size_t>(N[i]) * K);
    return b;
}

static size_t group_bwd_ws_bytes(int64_t M, const int64_t *N, int count)
{
    size_t b = kPartialsBytes;
    for (int i = 0; i < count; ++i)
        b += 2 * round256(static_cast<size_t>(M) * N[i]) + 256;
    return b;
}

// Shapes and the shared-X rule of a group; fills N[].
static f8_status check_group(const f8_group_linear *m, int count, int64_t M, int64_t K, int64_t *N)
{
    if (m == nullptr || count < 1 || count > F8_MAX_GROUP_LINEARS)
        return F8_ERR_INVALID;
    for (int i = 0; i < count; ++i) {
        F8_TRY(check_linear_shape(M, m[i].N, K));
        F8_TRY(check_saved(&m[i].saved));
        const f8_linear_saved &s0 = m[0].saved, &si = m[i].saved;
        if (si.x_t != s0.x_t || si.amax_x != s0.amax_x || si.scale_x != s0.scale_x)
            return F8_ERR_INVALID;
        N[i] = m[i].N;
    }
    return F8_OK;
}

size_t f8_linear_group_workspace_bytes(int64_t M, int64_t K, const int64_t *N, int count)
{
    if (N == nullptr || count < 1 || count > F8_MAX_GROUP_LINEARS || M <= 0 || K <= 0)
        return 0;
    for (int i = 0; i < count; ++i)
        if (N[i] <= 0)
            return 0;
    const size_t f = group_fwd_ws_bytes(M, K, N, count), b = group_bwd_ws_bytes(M, N, count);
    return f > b ? f : b;
}

f8_status f8_linear_fwd_group(const void *x, int64_t M, int64_t K, const f8_group_linear *members,
                              int count, void *workspace, size_t workspace_bytes, void *stream)
{
    int64_t N[F8_MAX_GROUP_LINEARS];
    F8_TRY(check_group(members, count, M, K, N));
    if (x == nullptr || workspace == nullptr)
        return F8_ERR_INVALID;
    for (int i = 0; i < count; ++i)
        if (members[i].w == nullptr || members[i].y == nullptr)
            return F8_ERR_INVALID;
    if (workspace_bytes < group_fwd_ws_bytes(M, K, N, count))
        return F8_ERR_INVALID;
    if (!aligned(x, 16) || !aligned(workspace, 256))
        return F8_ERR_ALIGN;
    for (int i = 0; i < count; ++i)
        if (!aligned(members[i].w, 16) || !aligned(members[i].y, 16))
            return F8_ERR_ALIGN;
    const DeviceInfo *dev;
    F8_TRY(get_device(&dev));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // workspace: q(X), q(W_0), ..., partials
    uint8_t *p = static_cast<uint8_t *>(workspace);
    uint8_t *x_q = p;
    p += round256(static_cast<size_t>(M) * K);
    uint8_t *w_q[F8_MAX_GROUP_LINEARS];
    for (int i = 0; i < count; ++i) {
        w_q[i] = p;
        p += round256(static_cast<size_t>(N[i]) * K);
    }
    unsigned *parts = reinterpret_cast<unsigned *>(p);
    const f8_linear_saved &s0 = members[0].saved;
    QuantDesc d[1 + F8_MAX_GROUP_LINEARS];
    d[0] = QuantDesc{x, M, K, s0.amax_x, s0.scale_x, x_q, s0.x_t};
    for (int i = 0; i < count; ++i) {
        const f8_linear_saved &si = members[i].saved;
        d[1 + i] = QuantDesc{members[i].w, N[i], K, si.amax_w, si.scale_w, w_q[i], si.w_t};
    }
    F8_TRY_CUDA(quantize_batches(d, 1 + count, F8_E4M3, parts, quant_batch_bytes(kPairMaxBytes),
                                 *dev, st));
    GemmDesc g[F8_MAX_GROUP_LINEARS];
    for (int i = 0; i < count; ++i)
        g[i] = GemmDesc{x_q, w_q[i], M, N[i], K, s0.scale_x, members[i].saved.scale_w,
                        members[i].y, F8_E4M3, F8_E4M3};
    return from_cuda(launch_gemm_multi(g, count, *dev, st));
}

f8_status f8_linear_bwd_group(const f8_group_linear *members, int count, int64_t M, int64_t K,
                              f8_format fmt_dy, void *workspace, size_t workspace_bytes,
                              void *stream)
{
    int64_t N[F8_MAX_GROUP_LINEARS];
    F8_TRY(check_group(members, count, M, K, N));
    if (workspace == nullptr || (fmt_dy != F8_E4M3 && fmt_dy != F8_E5M2))
        return F8_ERR_INVALID;
    for (int i = 0; i < count; ++i)
        if (members[i].dy == nullptr)
            return F8_ERR_INVALID;
    if (workspace_bytes < group_bwd_ws_bytes(M, N, count))
        return F8_ERR_INVALID;
    if (!aligned(workspace, 256))
        return F8_ERR_ALIGN;
    for (int i = 0; i < count; ++i)
        if (!aligned(members[i].dy, 16) || !aligned(members[i].dx, 16) ||
            !aligned(members[i].dw, 16))
            return F8_ERR_ALIGN;
    const DeviceInfo *dev;
    F8_TRY(get_device(&dev));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t *p = static_cast<uint8_t *>(workspace);
    uint8_t *dy_q[F8_MAX_GROUP_LINEARS], *dy_t[F8_MAX_GROUP_LINEARS];
    float *amax[F8_MAX_GROUP_LINEARS], *scale[F8_MAX_GROUP_LINEARS];
    for (int i = 0; i < count; ++i) {
        const size_t mn = round256(static_cast<size_t>(M) * N[i]);
        dy_q[i] = p;
        dy_t[i] = p + mn;
        amax[i] = reinterpret_cast<float *>(p + 2 * mn);
        scale[i] = reinterpret_cast<float *>(p + 2 * mn + 128);
        p += 2 * mn + 256;
    }
    unsigned *parts = reinterpret_cast<unsigned *>(p);
    QuantDesc d[F8_MAX_GROUP_LINEARS];
    for (int i = 0; i < count; ++i)
        d[i] = QuantDesc{members[i].dy, M, N[i], amax[i], scale[i],
                         members[i].dx ? dy_q[i] : nullptr, members[i].dw ? dy_t[i] : nullptr};
    F8_TRY_CUDA(quantize_batches(d, count, fmt_dy, parts, quant_batch_bytes(kPairMaxBytes), *dev,
                                 st));
    // dX_i [M,K] = q(dY_i) [M,N_i] . (q(W_i)^T [K,N_i])^T;  dW_i [N_i,K] = q(dY_i)^T . (q(X)^T [K,M])^T
    GemmDesc g[2 * F8_MAX_GROUP_LINEARS];
    int n = 0;
    for (int i = 0; i < count; ++i) {
        const f8_linear_saved &si = members[i].saved;
        if (members[i].dx != nullptr)
            g[n++] = GemmDesc{dy_q[i], si.w_t, M, K, N[i], scale[i], si.scale_w, members[i].dx,
                              fmt_dy, F8_E4M3};
        if (members[i].dw != nullptr)
            g[n++] = GemmDesc{dy_t[i], si.x_t, N[i], K, M, scale[i], si.scale_x, members[i].dw,
                              fmt_dy, F8_E4M3};
    }
    if (n == 0)
        return F8_OK;
    return from_cuda(launch_gemm_multi(g, n, *dev, st));
}

f8_status f8_transpose_u8(const uint8_t *in, int64_t rows, int64_t cols, uint8_t *out, void *stream)
{
    if (rows < 0 || cols < 0 || (rows > 0 && cols > 0 && (in == nullptr || out == nullptr)))
        return F8_ERR_INVALID;
    if (rows == 0 || cols == 0)
        return F8_OK;
    const DeviceInfo *dev;
    F8_TRY(get_device(&dev));
    return from_cuda(launch_transpose_u8(in, rows, cols, out, *dev, static_cast<cudaStream_t>(stream)));
}

size_t f8_linear_fwd_qw_workspace_bytes(int64_t M, int64_t K)
{
    if (M <= 0 || K <= 0)
        return 0;
    return round256(static_cast<size_t>(M) * K) + kPartialsBytes;
}

f8_status f8_linear_fwd_qw(const void *x, const uint8_t *w_q, int64_t M, int64_t N, int64_t K,
                           void *y, const f8_linear_saved *saved, void *workspace,
                           size_t workspace_bytes, void *stream)
{
    F8_TRY(check_linear_shape(M, N, K));
    F8_TRY(check_saved(saved));
    if (x == nullptr || w_q == nullptr || y == nullptr || workspace == nullptr)
        return F8_ERR_INVALID;
    if (workspace_bytes < f8_linear_fwd_qw_workspace_bytes(M, K))
        return F8_ERR_INVALID;
    if (!aligned(x, 16) || !aligned(w_q, 16) || !aligned(y, 16) || !aligned(workspace, 256))
        return F8_ERR_ALIGN;
    const DeviceInfo *dev;
    F8_TRY(get_device(&dev));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t *x_q = static_cast<uint8_t *>(workspace);
    unsigned *parts = reinterpret_cast<unsigned *>(x_q + round256(static_cast<size_t>(M) * K));
    int np = 0;
    F8_TRY_CUDA(launch_amax_partials(x, M * K, parts, &np, *dev, st));
    F8_TRY_CUDA(launch_cast_transpose(x, M, K, nullptr, parts, np, saved->amax_x, saved->scale_x,
                                      x_q, saved->x_t, 0, *dev, st, true));
    return from_cuda(launch_gemm(x_q, w_q, M, N, K, saved->scale_x, saved->scale_w, y, *dev, st));
}

f8_status f8_quantize_swiglu(const void *a, const void *b, void *h, int64_t rows, int64_t cols,
                             float *amax_out, float *scale_out, uint8_t *q, uint8_t *q_t,
                             void *workspace, size_t workspace_bytes, void *stream)
{
    if (rows < 0 || cols < 0 || amax_out == nullptr || workspace == nullptr ||
        (rows > 0 && cols > 0 && (a == nullptr || b == nullptr || h == nullptr)))
        return F8_ERR_INVALID;
    if (workspace_bytes < kPartialsBytes)
        return F8_ERR_INVALID;
    if (!aligned(a, 16) || !aligned(b, 16) || !aligned(h, 16) || !aligned(q, 16) ||
        !aligned(q_t, 16) || !aligned(amax_out, 4) || !aligned(scale_out, 4) ||
        !aligned(workspace, 16))
        return F8_ERR_ALIGN;
    const DeviceInfo *dev;
    F8_TRY(get_device(&dev));
    return from_cuda(launch_quantize_swiglu(a, b, h, rows, cols, static_cast<unsigned *>(workspace),
                                            amax_out, scale_out, q, q_t, *dev,
                                            static_cast<cudaStream_t>(stream)));
}

f8_status f8_linear_fwd_swiglu(const void *a, const void *b, void *h, const void *w, int64_t M,
                               int64_t N, int64_t K, void *y, const f8_linear_saved *saved,
                               void *workspace, size_t workspace_bytes, void *stream)
{
    F8_TRY(check_linear_shape(M, N, K));
    F8_TRY(check_saved(saved));
    if (a == nullptr || b == nullptr || h == nullptr || w == nullptr || y == nullptr ||
        workspace == nullptr)
        return F8_ERR_INVALID;
    if (workspace_bytes < fwd_ws_bytes(M, N, K))
        return F8_ERR_INVALID;
    if (!aligned(a, 16) || !aligned(b, 16) || !aligned(h, 16) || !aligned(w, 16) ||
        !aligned(y, 16) || !aligned(workspace, 256))
        return F8_ERR_ALIGN;
    const DeviceInfo *dev;
    F8_TRY(get_device(&dev));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const FwdWs fw = fwd_ws(workspace, M, N, K);
    int np = 0;
    F8_TRY_CUDA(launch_quantize_swiglu(a, b, h, M, K, fw.parts_x, saved->amax_x, saved->scale_x,
                                       fw.x_q, saved->x_t, *dev, st));
    F8_TRY_CUDA(launch_amax_partials(w, N * K, fw.parts_w, &np, *dev, st));
    F8_TRY_CUDA(launch_cast_transpose(w, N, K, nullptr, fw.parts_w, np, saved->amax_w,
                                      saved->scale_w, fw.w_q, saved->w_t, 0, *dev, st, true));
    return from_cuda(launch_gemm(fw.x_q, fw.w_q, M, N, K, saved->scale_x, saved->scale_w, y, *dev, st));
}

f8_status f8_linear_fwd_w13_swiglu(const void *x, const void *w13, int64_t M, int64_t F,
                                   int64_t K, void *ab, void *h, const f8_linear_saved *saved,
                                   float *amax_h, float *scale_h, uint8_t *h_q, uint8_t *h_t,
                                   void *workspace, size_t workspace_bytes, void *stream)
{
    if (M <= 0 || F <= 0 || K <= 0)
        return F8_ERR_INVALID;
    if (F % 128 || F > INT32_MAX / 4)
        return F8_ERR_SHAPE;
    const int64_t N = 2 * F;
    F8_TRY(check_linear_shape(M, N, K));
    F8_TRY(check_saved(saved));
    if (x == nullptr || w13 == nullptr || ab == nullptr || h == nullptr || amax_h == nullptr ||
        scale_h == nullptr || h_q == nullptr || h_t == nullptr || workspace == nullptr)
        return F8_ERR_INVALID;
    if (workspace_bytes < fwd_ws_bytes(M, N, K))
        return F8_ERR_INVALID;
    if (!aligned(x, 16) || !aligned(w13, 16) || !aligned(ab, 16) || !aligned(h, 16) ||
        !aligned(h_q, 16) || !aligned(h_t, 16) || !aligned(amax_h, 4) || !aligned(scale_h, 4) ||
        !aligned(workspace, 256))
        return F8_ERR_ALIGN;
    const DeviceInfo *dev;
    F8_TRY(get_device(&dev));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const FwdWs fw = fwd_ws(workspace, M, N, K);
    int np = 0;
    F8_TRY_CUDA(launch_amax_partials(x, M * K, fw.parts_x, &np, *dev, st));
    F8_TRY_CUDA(launch_cast_transpose(x, M, K, nullptr, fw.parts_x, np, saved->amax_x,
                                      saved->scale_x, fw.x_q, saved->x_t, 0, *dev, st, true));
    F8_TRY_CUDA(launch_amax_partials(w13, N * K, fw.parts_w, &np, *dev, st));
    F8_TRY_CUDA(launch_cast_transpose(w13, N, K, nullptr, fw.parts_w, np, saved->amax_w,
                                      saved->scale_w, fw.w_q, saved->w_t, 0, *dev, st, true));
    // the X partials were consumed by the cast of X, which the GEMM's
    // dependency wait orders before it: they take h's partials
    int nh = 0;
    F8_TRY_CUDA(launch_gemm_w13_swiglu(fw.x_q, fw.w_q, M, F, K, saved->scale_x, saved->scale_w, ab,
                                       h, fw.parts_x, &nh, *dev, st));
    return from_cuda(launch_cast_transpose(h, M, F, nullptr, fw.parts_x, nh, amax_h, scale_h, h_q,
                                           h_t, 0, *dev, st));
}

f8_status f8_quantize_swiglu_bwd(const void *dh, const void *ab, int64_t M, int64_t F, void *dab,
                                 f8_format fmt, float *amax_out, float *scale_out, uint8_t *q,
                                 uint8_t *q_t, void *workspace, size_t workspace_bytes,
                                 void *stream)
{
    if (M <= 0 || F <= 0 || (fmt != F8_E4M3 && fmt != F8_E5M2))
        return F8_ERR_INVALID;
    if (F % 128 || F > INT32_MAX / 4 || M > INT32_MAX / 2)
        return F8_ERR_SHAPE;
    if (dh == nullptr || ab == nullptr || dab == nullptr || amax_out == nullptr ||
        workspace == nullptr)
        return F8_ERR_INVALID;
    if (workspace_bytes < kPartialsBytes)
        return F8_ERR_INVALID;
    if (!aligned(dh, 16) || !aligned(ab, 16) || !aligned(dab, 16) || !aligned(q, 16) ||
        !aligned(q_t, 16) || !aligned(amax_out, 4) || !aligned(scale_out, 4) ||
        !aligned(workspace, 16))
        return F8_ERR_ALIGN;
    const DeviceInfo *dev;
    F8_TRY(get_device(&dev));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned *parts = static_cast<unsigned *>(workspace);
    int np = 0;
    F8_TRY_CUDA(launch_swiglu_bwd_amax(dh, ab, dab, M, F, parts, &np, *dev, st));
    return from_cuda(launch_cast_transpose(dab, M, 2 * F, nullptr, parts, np, amax_out, scale_out, q,
                                           q_t, fmt, *dev, st));
}

f8_status f8_linear_bwd_w13_swiglu(const void *dh, const void *ab, const f8_linear_saved *saved,
                                   int64_t M, int64_t F, int64_t K, void *dab, f8_format fmt_dab,
                                   void *dx, void *dw13, void *workspace, size_t workspace_bytes,
                                   void *stream)
{
    if (M <= 0 || F <= 0 || K <= 0 || (fmt_dab != F8_E4M3 && fmt_dab != F8_E5M2))
        return F8_ERR_INVALID;
    if (F % 128 || F > INT32_MAX / 4)
        return F8_ERR_SHAPE;
    const int64_t N = 2 * F;
    F8_TRY(check_linear_shape(M, N, K));
    F8_TRY(check_saved(saved));
    if (dh == nullptr || ab == nullptr || dab == nullptr || workspace == nullptr)
        return F8_ERR_INVALID;
    if (workspace_bytes < bwd_ws_bytes(M, N))
        return F8_ERR_INVALID;
    if (!aligned(dh, 16) || !aligned(ab, 16) || !aligned(dab, 16) || !aligned(dx, 16) ||
        !aligned(dw13, 16) || !aligned(workspace, 256))
        return F8_ERR_ALIGN;
    const DeviceInfo *dev;
    F8_TRY(get_device(&dev));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const BwdWs bw = bwd_ws(workspace, M, N);
    int np = 0;
    F8_TRY_CUDA(launch_swiglu_bwd_amax(dh, ab, dab, M, F, bw.parts_dy, &np, *dev, st));
    F8_TRY_CUDA(launch_cast_transpose(dab, M, N, nullptr, bw.parts_dy, np, bw.amax_dy, bw.scale_dy,
                                      dx ? bw.dy_q : nullptr, dw13 ? bw.dy_t : nullptr, fmt_dab,
                                      *dev, st));
    return from_cuda(launch_bwd_gemms(bw, saved, M, N, K, fmt_dab, dx, dw13, *dev, st));
}

f8_status f8_gemm_w13_swiglu(const uint8_t *x_q, const uint8_t *w13_q, int64_t M, int64_t F,
                             int64_t K, const float *scale_x, const float *scale_w13, void *ab,
                             void *h, float *amax_h, void *stream)
{
    if (M <= 0 || F <= 0 || K <= 0)
        return F8_ERR_INVALID;
    if (F % 128 || F > INT32_MAX / 4)
        return F8_ERR_SHAPE;
    F8_TRY(check_linear_shape(M, 2 * F, K));
    if (x_q == nullptr || w13_q == nullptr || scale_x == nullptr || scale_w13 == nullptr ||
        ab == nullptr || h == nullptr || amax_h == nullptr)
        return F8_ERR_INVALID;
    if (!aligned(x_q, 16) || !aligned(w13_q, 16) || !aligned(ab, 16) || !aligned(h, 16) ||
        !aligned(scale_x, 4) || !aligned(scale_w13, 4) || !aligned(amax_h, 4))
        return F8_ERR_ALIGN;
    const DeviceInfo *dev;
    F8_TRY(get_device(&dev));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    F8_TRY_CUDA(cudaMemsetAsync(amax_h, 0, sizeof(float), st));
    int nh = 0;
    return from_cuda(launch_gemm_w13_swiglu(x_q, w13_q, M, F, K, scale_x, scale_w13, ab, h,
                                            reinterpret_cast<unsigned *>(amax_h), &nh, *dev, st,
                                            true));
}

unsigned long long f8_kernel_launches(void)
{
    return g_kernel_launches.load(std::memory_order_relaxed);
}

f8_status f8_last_device_status(void *stream)
{
    const DeviceInfo *dev = device_info();
    if (dev == nullptr)
        return F8_ERR_CUDA;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return F8_ERR_CUDA;
    unsigned word = 0;
    if (cudaMemcpy(&word, dev->status, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
        return F8_ERR_CUDA;
    const unsigned zero = 0;
    if (cudaMemcpy(dev->status, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
        return F8_ERR_CUDA;
    if (word & kStatusBounds)
        return F8_ERR_BOUNDS;
    if (word & kStatusTimeout)
        return F8_ERR_TIMEOUT;
    if (word & kStatusNonfinite)
        return F8_ERR_NONFINITE;
    return F8_OK;
}

f8_status f8_selftest_bounds(void *stream)
{
    if (!bounds_checked_build())
        return F8_ERR_UNSUPPORTED;
    const DeviceInfo *dev;
    F8_TRY(get_device(&dev));
    return from_cuda(launch_bounds_selftest(*dev, static_cast<cudaStream_t>(stream)));
}

f8_status f8_selftest_wait_timeout(uint64_t limit_ns, void *stream)
{
    const DeviceInfo *dev;
    F8_TRY(get_device(&dev));
    return from_cuda(launch_wait_selftest(limit_ns, *dev, static_cast<cudaStream_t>(stream)));
}

} // extern "C"
