// Launchers shared between the translation units of libf8 (host side only).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cstdlib>
#include <cuda.h>
#include <cuda_runtime.h>
#include <atomic>
#include <utility>

#include "f8.h"

namespace f8 {

struct DeviceInfo {
    int ordinal = -1;
    int sm_count = 0;
    int cc_major = 0;
    int cc_minor = 0;
    unsigned *status = nullptr; // device address of this device's status word
};

// Per-device facts, filled on first use of a device (thread-safe).
// Returns nullptr if the device cannot be queried.
const DeviceInfo *device_info();

// Time limit of the GEMM pipeline's device waits.
uint64_t wait_limit_ns();

// 2-D row-major tensor [rows, cols] of `esize`-byte elements as a TMA tensor
// map with a box_cols x box_rows box; false if the driver entry point is
// missing or the encoding is refused.
bool make_tensor_map_2d(CUtensorMap *map, CUtensorMapDataType dtype, int esize, const void *ptr,
                        int64_t rows, int64_t cols, int box_cols, int box_rows,
                        CUtensorMapSwizzle swizzle);

// The TMA-fed cast is used unless F8_CAST_TMA=0 (for measurement).
inline bool cast_tma_enabled()
{
    const char *e = std::getenv("F8_CAST_TMA");
    return e == nullptr || e[0] != '0';
}

// The TMA cast takes its tiles last first (so that its re-read starts
// with what the amax pass left in L2) unless F8_CAST_REVERSE=0.
inline bool cast_reverse_enabled()
{
    const char *e = std::getenv("F8_CAST_REVERSE");
    return e == nullptr || e[0] != '0';
}

// Largest bf16 total (bytes) one multi-tensor quantisation launch pair
// takes; larger lists are split into consecutive batches within it, and a
// tensor larger than it is quantised alone.  F8_QUANT_BATCH_MB overrides
// the default (for measurement).
inline int64_t quant_batch_bytes(int64_t dflt)
{
    const char *e = std::getenv("F8_QUANT_BATCH_MB");
    return e == nullptr ? dflt : static_cast<int64_t>(std::atoll(e)) << 20;
}

// X and W of a small linear are quantised together (one amax launch, one
// cast launch) unless F8_QUANT_PAIR=0.
inline bool quant_pair_enabled()
{
    const char *e = std::getenv("F8_QUANT_PAIR");
    return e == nullptr || e[0] != '0';
}

// Whether launch_gemm_multi puts several GEMMs in one launch:
// F8_GEMM_GROUP=0 never, =2 always (all in one launch where one launch can
// take them), otherwise (1 or unset) as sched_partition plans it: shared
// launches only where the predicted time beats one launch per GEMM by the
// planner's margin.
constexpr int kGroupNever = 0;
constexpr int kGroupAuto = 1;
constexpr int kGroupAlways = 2;
inline int gemm_group_mode()
{
    const char *e = std::getenv("F8_GEMM_GROUP");
    if (e == nullptr)
        return kGroupAuto;
    if (e[0] == '0')
        return kGroupNever;
    return e[0] == '2' ? kGroupAlways : kGroupAuto;
}

// Kernels this library has launched in this process (every launch site adds
// one; defined in f8_api.cu).
extern std::atomic<unsigned long long> g_kernel_launches;

inline void count_launch() { g_kernel_launches.fetch_add(1, std::memory_order_relaxed); }

// Programmatic dependent launch is on unless F8_PDL=0.
inline bool pdl_enabled()
{
    const char *e = std::getenv("F8_PDL");
    return e == nullptr || e[0] != '0';
}

// Launch with programmatic stream serialization, so the kernel's prologue
// may overlap the tail of the previous kernel in the stream.  Every kernel
// launched this way calls griddep_wait() before reading dependent data.
// `cluster_x` > 1 launches clusters of that many CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                               cudaStream_t stream, unsigned cluster_x, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (pdl_enabled()) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    count_launch();
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args)
{
    return launch_pdl_cluster(kernel, grid, block, smem, stream, 1u, std::forward<Args>(args)...);
}

// Most partial maxima one amax launch writes (its largest grid).
constexpr int kMaxAmaxPartials = 4096;

// amax over n bf16 values into one fp32 (zeroed here, then atomicMax);
// n >= 1, x 16-byte aligned.
cudaError_t launch_amax(const void *x, int64_t n, float *amax_out, const DeviceInfo &dev,
                        cudaStream_t stream);

// amax over n bf16 values as per-block partial maxima (fp32 bit patterns),
// no zeroing needed; *nparts receives the number written (<= kMaxAmaxPartials).
cudaError_t launch_amax_partials(const void *x, int64_t n, unsigned *partials, int *nparts,
                                 const DeviceInfo &dev, cudaStream_t stream);

// Scale + cast + (optional) transpose of a [rows, cols] bf16 tensor.  The
// amax comes either from `amax` (one fp32) or, if `partials` is non-null,
// from the maximum of `nparts` partial maxima, which is then also stored to
// `amax_out` (if non-null).
// fmt: 0 = E4M3 (scale 448/amax), 1 = E5M2 (scale 57344/amax).
// early: the launch just before this one on the stream only read x (its
// amax pass), so x is complete when this kernel starts and its first tiles
// may be loaded before the dependency wait.  Leave it false after a kernel
// that writes x.
cudaError_t launch_cast_transpose(const void *x, int64_t rows, int64_t cols, const float *amax,
                                  const unsigned *partials, int nparts, float *amax_out,
                                  float *scale_out, uint8_t *q, uint8_t *q_t, int fmt,
                                  const DeviceInfo &dev, cudaStream_t stream, bool early = false);

// Most tensors one multi-tensor quantisation launch pair takes.
constexpr int kMaxQuantTensors = 8;

// One tensor of a multi-tensor quantisation: bf16 [rows, cols] in, its amax
// and scale (device fp32) and its codes (either may be null) out.
struct QuantDesc {
    const void *x;
    int64_t rows, cols;
    float *amax_out, *scale_out;
    uint8_t *q, *q_t;
};

// Whether launch_quantize_multi takes these tensors (every side a multiple
// of 128, the TMA cast enabled, 1 <= n <= kMaxQuantTensors).
bool quantize_multi_castable(const QuantDesc *t, int n);

// Dynamic tensorwise quantisation of n tensors, each with its own amax and
// scale, in two launches: one amax launch whose blocks are split between the
// tensors in proportion to their sizes (partial maxima in `parts`, which
// holds kMaxAmaxPartials), then one TMA cast launch over all their tiles.
// cudaErrorNotSupported (nothing launched) unless quantize_multi_castable.
cudaError_t launch_quantize_multi(const QuantDesc *t, int n, int fmt, unsigned *parts,
                                  const DeviceInfo &dev, cudaStream_t stream);

// h = bf16(silu(a) * b) for two [rows, cols] bf16 tensors written to `h`
// together with its amax partials (one pass), then its E4M3 cast.
cudaError_t launch_quantize_swiglu(const void *a, const void *b, void *h, int64_t rows,
                                   int64_t cols, unsigned *partials, float *amax_out,
                                   float *scale_out, uint8_t *q, uint8_t *q_t, const DeviceInfo &dev,
                                   cudaStream_t stream);

// C[M,N] = bf16(A[M,K] B[N,K]^T / (sa sb)); M, N, K >= 1, K % 16 == 0.
// fa, fb: operand formats (0 = E4M3, 1 = E5M2).
// Returns cudaErrorNotSupported if the tensor-map encoder is unavailable.
cudaError_t launch_gemm(const uint8_t *a, const uint8_t *b, int64_t M, int64_t N, int64_t K,
                        const float *sa, const float *sb, void *c, const DeviceInfo &dev,
                        cudaStream_t stream, int fa = 0, int fb = 0);

// One GEMM as launch_gemm_multi takes it: C[M,N] = bf16(A[M,K] B[N,K]^T / (sa sb)).
struct GemmDesc {
    const uint8_t *a;
    const uint8_t *b;
    int64_t M, N, K;
    const float *sa;
    const float *sb;
    void *c;
    int fa, fb;
};

// n (<= 8) independent GEMMs in as few persistent launches as pay:
// f8_sched.h's sched_partition groups problems of at most two tile costs
// (K extents) into launches of up to four; within a launch the costlier
// class is dealt round-robin over the CTAs and the other class's tiles then
// go, in order, to the CTA that frees up first (a static list schedule each
// CTA evaluates in closed form).  Problems that need different kernels (the
// CTA-pair kernel for M >= 256, the single-CTA one below) never share a
// launch.
cudaError_t launch_gemm_multi(const GemmDesc *g, int n, const DeviceInfo &dev, cudaStream_t stream);

// launch_gemm_multi of two problems.
cudaError_t launch_gemm2(const GemmDesc &g0, const GemmDesc &g1, const DeviceInfo &dev,
                         cudaStream_t stream);

// The W13 GEMM of a SwiGLU FFN: AB[M, 2F] = bf16(X W13^T / (sx sw)) with
// W13 interleaved by 128 rows (W1 block, W3 block, ...), and h[M, F] =
// bf16(silu(a) b) from its epilogue with one |h| partial maximum per CTA in
// hparts (*nparts receives their count), or with hatomic one atomicMax per
// CTA into hparts[0] (a zeroed fp32 amax).  F % 128 == 0.
cudaError_t launch_gemm_w13_swiglu(const uint8_t *x_q, const uint8_t *w13_q, int64_t M, int64_t F,
                                   int64_t K, const float *sx, const float *sw, void *ab, void *h,
                                   unsigned *hparts, int *nparts, const DeviceInfo &dev,
                                   cudaStream_t stream, bool hatomic = false);

// d(AB) [M, 2F] (AB's column order) of the w1+w3 group from the gradient dh
// [M, F] of h = silu(a) b and the forward's AB, with one |d(AB)| partial
// maximum per CTA in partials (*nparts receives their count).  F % 128 == 0.
cudaError_t launch_swiglu_bwd_amax(const void *dh, const void *ab, void *dab, int64_t M, int64_t F,
                                   unsigned *partials, int *nparts, const DeviceInfo &dev,
                                   cudaStream_t stream);

// out[c, r] = in[r, c] for a [rows, cols] uint8 tensor (rows, cols >= 1).
cudaError_t launch_transpose_u8(const uint8_t *in, int64_t rows, int64_t cols, uint8_t *out,
                                const DeviceInfo &dev, cudaStream_t stream);

// The argument rules of a linear (M, N, K multiples of 16 and > 0, tile
// counts within the kernels' 32-bit index) and of its saved tensors, as
// f8_linear_fwd / f8_linear_bwd apply them.
f8_status check_linear_shape(int64_t M, int64_t N, int64_t K);
f8_status check_saved(const f8_linear_saved *s);

// Workspace bytes f8_linear_fwd needs (its row-major E4M3 copies of X and W
// and the amax partial maxima), for a shape that passed check_linear_shape.
size_t linear_fwd_ws_bytes(int64_t M, int64_t N, int64_t K);

// f8_linear_fwd itself: argument checks, then its launches with `workspace`.
f8_status linear_fwd_impl(const void *x, const void *w, int64_t M, int64_t N, int64_t K, void *y,
                          const f8_linear_saved *saved, void *workspace, size_t workspace_bytes,
                          cudaStream_t stream);

// Whether this library was built with the device bounds checks
// (-DF8_BOUNDS_CHECK), and a one-thread kernel that makes one such check
// fail without touching memory (it sets kStatusBounds in a checked build).
bool bounds_checked_build();
cudaError_t launch_bounds_selftest(const DeviceInfo &dev, cudaStream_t stream);

// One CTA waiting on an mbarrier that is never signalled (failure-path test).
cudaError_t launch_wait_selftest(uint64_t limit_ns, const DeviceInfo &dev, cudaStream_t stream);

} // namespace f8
