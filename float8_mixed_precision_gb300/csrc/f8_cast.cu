// The HBM-bound steps of dynamic tensorwise scaling: amax, and the fused
// scale + cast + transpose (bf16 -> E4M3 or E5M2); also the SwiGLU passes
// that produce a tensor together with its amax.
//
// amax_kernel: every thread streams 16-byte vectors of 8 bf16 values with
// eight independent (predicated) loads in flight, also in the last round,
// and keeps the maximum of the magnitude bits (bits & 0x7FFF: for
// non-negative IEEE values the integer order is the numeric order, and
// inf/NaN sort above every finite value).  It reduces through redux.sync
// within the warp and shared memory within the block, then either folds the
// block result into the output with one atomicMax on the fp32 bit pattern,
// or (inside a linear) writes one partial maximum per block, so that no
// output has to be zeroed first; the cast kernel reduces the partials in its
// prologue.  amax_multi_kernel does the same for up to eight tensors in one
// launch, its blocks split between them in proportion to their sizes.
//
// cast_transpose_kernel: a CTA owns a 128 x 128 tile.  Phase 1 reads it with
// 16-byte loads (each thread 16 consecutive bf16 of one row), scales in
// fp32, converts with the hardware's saturating RNE conversion, writes the
// row-major codes with 16-byte stores and parks them in a 16 KB shared tile
// whose 16-byte chunks are XOR-swizzled by (row / 16) % 8.  Phase 2 gives
// each thread a 16-row x 4-column block: 16 conflict-free 4-byte shared
// loads, a byte transpose with PRMT, and four 16-byte stores of the
// column-major copy (8 consecutive threads write 128 contiguous bytes of one
// column).  cast_transpose_tma_kernel does the same with the bf16 tiles
// brought in by TMA through a 3-stage ring, for one tensor or up to eight
// (each with its own scale) whose sides are multiples of 128; the register
// kernel takes the other shapes.
//
// swiglu_amax_kernel / swiglu_bwd_amax_kernel: h = silu(a) b, and the
// gradient d(AB) of the w1+w3 group, each produced in one pass that also
// writes one partial maximum per CTA for the cast that follows.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <mutex>

#include "f8_internal.h"
#include "f8_ptx.cuh"
#include "f8_swiglu.cuh"

namespace f8 {
namespace {

using swiglu::swiglu_x2;

constexpr int kAmaxThreads = 256;
constexpr int kAmaxUnroll = 8;

__device__ __forceinline__ uint32_t max_u16x2(uint32_t acc, uint4 v)
{
    acc = __vmaxu2(acc, v.x & 0x7FFF7FFFu);
    acc = __vmaxu2(acc, v.y & 0x7FFF7FFFu);
    acc = __vmaxu2(acc, v.z & 0x7FFF7FFFu);
    acc = __vmaxu2(acc, v.w & 0x7FFF7FFFu);
    return acc;
}

template <bool kPartials>
__global__ void __launch_bounds__(kAmaxThreads, 4)
amax_kernel(const uint4 *__restrict__ x, int64_t nvec, const uint16_t *__restrict__ tail, int ntail,
            unsigned *__restrict__ out_bits, unsigned *__restrict__ status)
{
    griddep_wait();
    griddep_launch_dependents();
    uint32_t m2 = 0;
    const int64_t S = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; base < nvec;
         base += kAmaxUnroll * S) {
        uint4 v[kAmaxUnroll];
#pragma unroll
        for (int u = 0; u < kAmaxUnroll; ++u) {
            const int64_t i = base + u * S;
            v[u] = i < nvec && in_range(i, 1, nvec, status) ? __ldg(x + i) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kAmaxUnroll; ++u)
            m2 = max_u16x2(m2, v[u]);
    }
    uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
    if (blockIdx.x == 0 && threadIdx.x < ntail && in_range(threadIdx.x, 1, ntail, status))
        m = max(m, static_cast<uint32_t>(tail[threadIdx.x]) & 0x7FFFu);

    m = __reduce_max_sync(0xFFFFFFFFu, m);
    __shared__ uint32_t warp_max[kAmaxThreads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0)
        warp_max[warp] = m;
    __syncthreads();
    if (warp == 0) {
        m = lane < kAmaxThreads / 32 ? warp_max[lane] : 0u;
        m = __reduce_max_sync(0xFFFFFFFFu, m);
        if (lane == 0) {
            if (m >= 0x7F80u)
                atomicOr(status, kStatusNonfinite);
            if (kPartials)
                out_bits[blockIdx.x] = m << 16;
            else
                atomicMax(out_bits, m << 16);
        }
    }
}

// Partial maxima of up to kMaxQuantTensors tensors in one launch (no tails:
// every length is a multiple of 8): blocks [first_block[i],
// first_block[i + 1]) take tensor i, each tensor with its own grid stride;
// block j of a tensor writes that tensor's partial j.
struct AmaxSegs {
    const uint4 *x[kMaxQuantTensors];
    int64_t nvec[kMaxQuantTensors];
    unsigned *parts[kMaxQuantTensors];
    int first_block[kMaxQuantTensors + 1];
    int nseg;
};

__global__ void __launch_bounds__(kAmaxThreads, 4)
amax_multi_kernel(const __grid_constant__ AmaxSegs segs, unsigned *__restrict__ status)
{
    griddep_wait();
    griddep_launch_dependents();
    int seg = 0;
#pragma unroll
    for (int i = 1; i < kMaxQuantTensors; ++i)
        seg += (i < segs.nseg && static_cast<int>(blockIdx.x) >= segs.first_block[i]) ? 1 : 0;
    const uint4 *__restrict__ x = segs.x[seg];
    const int64_t nvec = segs.nvec[seg];
    const int bid = static_cast<int>(blockIdx.x) - segs.first_block[seg];
    const int nblk = segs.first_block[seg + 1] - segs.first_block[seg];
    uint32_t m2 = 0;
    const int64_t S = static_cast<int64_t>(nblk) * blockDim.x;
    for (int64_t base = static_cast<int64_t>(bid) * blockDim.x + threadIdx.x; base < nvec;
         base += kAmaxUnroll * S) {
        uint4 v[kAmaxUnroll];
#pragma unroll
        for (int u = 0; u < kAmaxUnroll; ++u) {
            const int64_t i = base + u * S;
            v[u] = i < nvec && in_range(i, 1, nvec, status) ? __ldg(x + i) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kAmaxUnroll; ++u)
            m2 = max_u16x2(m2, v[u]);
    }
    uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    __shared__ uint32_t warp_max[kAmaxThreads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0)
        warp_max[warp] = m;
    __syncthreads();
    if (warp == 0) {
        m = lane < kAmaxThreads / 32 ? warp_max[lane] : 0u;
        m = __reduce_max_sync(0xFFFFFFFFu, m);
        if (lane == 0) {
            if (m >= 0x7F80u)
                atomicOr(status, kStatusNonfinite);
            segs.parts[seg][bid] = m << 16;
        }
    }
}

// ----------------------------------------------------------------- cast
constexpr int kTile = 128;
constexpr int kCastThreads = 256;
constexpr int kCastThreadsMax = 256;

// Largest finite value of the target format: 448 (E4M3, FMT 0) or 57344
// (E5M2, FMT 1).
template <int FMT>
__device__ __forceinline__ float scale_of(float amax)
{
    return __fdiv_rn(FMT == 1 ? 57344.0f : 448.0f, fmaxf(amax, 1e-12f));
}

// Maximum of the partial maxima (fp32 bit patterns of non-negative values),
// reduced by the whole block; every thread gets the result.
__device__ __forceinline__ float reduce_partials(const unsigned *partials, int n)
{
    __shared__ uint32_t red[kCastThreadsMax / 32];
    uint32_t m = 0;
    for (int i = threadIdx.x; i < n; i += blockDim.x)
        m = max(m, partials[i]);
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0)
        red[warp] = m;
    __syncthreads();
    m = lane < static_cast<int>(blockDim.x >> 5) ? red[lane] : 0u;
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    __syncthreads();
    return __uint_as_float(m);
}

// Saturating RNE conversion of two fp32 values to two FP8 codes (lo in the
// low byte).
template <int FMT>
__device__ __forceinline__ uint16_t cvt2(float lo, float hi)
{
    return static_cast<uint16_t>(__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE,
                                                          FMT == 1 ? __NV_E5M2 : __NV_E4M3));
}

template <int FMT>
__device__ __forceinline__ uint32_t bf16x2_to_fp8x2(uint32_t w, float s)
{
    const float lo = __uint_as_float(w << 16);
    const float hi = __uint_as_float(w & 0xFFFF0000u);
    return cvt2<FMT>(__fmul_rn(lo, s), __fmul_rn(hi, s));
}

// 8 bf16 (one uint4) -> 8 FP8 codes (one uint2), element order preserved.
template <int FMT>
__device__ __forceinline__ uint2 cvt8(uint4 v, float s)
{
    uint2 r;
    r.x = bf16x2_to_fp8x2<FMT>(v.x, s) | (bf16x2_to_fp8x2<FMT>(v.y, s) << 16);
    r.y = bf16x2_to_fp8x2<FMT>(v.z, s) | (bf16x2_to_fp8x2<FMT>(v.w, s) << 16);
    return r;
}

template <int FMT>
__device__ __forceinline__ uint8_t cvt1(uint16_t b, float s)
{
    const float v = __fmul_rn(__uint_as_float(static_cast<uint32_t>(b) << 16), s);
    return static_cast<uint8_t>(cvt2<FMT>(v, 0.0f) & 0xFFu);
}

// h = silu(a) * b for the whole [n] tensors, written once as bf16, with one
// partial maximum of |h| per CTA (as amax_kernel<true>): the amax comes out
// of the pass that produces h, so h is read only by the cast.
__global__ void __launch_bounds__(kAmaxThreads)
swiglu_amax_kernel(const uint4 *__restrict__ a, const uint4 *__restrict__ b, uint4 *__restrict__ h,
                   int64_t nvec, const uint16_t *__restrict__ a_tail, const uint16_t *__restrict__ b_tail,
                   uint16_t *__restrict__ h_tail, int ntail, unsigned *__restrict__ partials,
                   unsigned *__restrict__ status)
{
    griddep_wait();
    griddep_launch_dependents();
    constexpr int kU = 4;
    uint32_t m2 = 0;
    const int64_t S = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; base < nvec;
         base += kU * S) {
        uint4 va[kU], vb[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int64_t i = base + u * S;
            const bool in = i < nvec && in_range(i, 1, nvec, status);
            va[u] = in ? __ldg(a + i) : make_uint4(0, 0, 0, 0);
            vb[u] = in ? __ldg(b + i) : make_uint4(0, 0, 0, 0);
        }
        uint32_t amag = 0;
#pragma unroll
        for (int u = 0; u < kU; ++u)
            amag = swiglu::fold_abs(amag, va[u]);
        uint4 hv[kU];
        // one branch per 32 elements, so that their chains interleave
        if (swiglu::small87(amag)) {
#pragma unroll
            for (int u = 0; u < kU; ++u)
                hv[u] = swiglu::swiglu8<false>(va[u], vb[u]);
        } else {
#pragma unroll
            for (int u = 0; u < kU; ++u)
                hv[u] = swiglu::swiglu8<true>(va[u], vb[u]);
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int64_t i = base + u * S;
            if (i < nvec && in_range(i, 1, nvec, status)) {
                h[i] = hv[u];
                m2 = max_u16x2(m2, hv[u]);
            }
        }
    }
    uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
    if (blockIdx.x == 0 && threadIdx.x < ntail && in_range(threadIdx.x, 1, ntail, status)) {
        const uint32_t hv = swiglu_x2<true>(a_tail[threadIdx.x], b_tail[threadIdx.x]) & 0xFFFFu;
        h_tail[threadIdx.x] = static_cast<uint16_t>(hv);
        m = max(m, hv & 0x7FFFu);
    }
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    __shared__ uint32_t warp_max[kAmaxThreads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0)
        warp_max[warp] = m;
    __syncthreads();
    if (warp == 0) {
        m = lane < kAmaxThreads / 32 ? warp_max[lane] : 0u;
        m = __reduce_max_sync(0xFFFFFFFFu, m);
        if (lane == 0) {
            if (m >= 0x7F80u)
                atomicOr(status, kStatusNonfinite);
            partials[blockIdx.x] = m << 16;
        }
    }
}

// d(AB) of the w1+w3 group from the gradient dh [M, F] of h and the
// forward's AB [M, 2F] (a and b in column blocks of 128, alternating): for
// the 16-byte vector v of dh, a is vector v + 16 (v / 16) of AB and b the
// one 16 vectors further; da and db are written at those same places of
// dAB.  One partial maximum of |d(AB)| per CTA, as amax_kernel<true>.
__global__ void __launch_bounds__(kAmaxThreads)
swiglu_bwd_amax_kernel(const uint4 *__restrict__ dh, const uint4 *__restrict__ ab,
                       uint4 *__restrict__ dab, int64_t nvec, unsigned *__restrict__ partials,
                       unsigned *__restrict__ status)
{
    griddep_wait();
    griddep_launch_dependents();
    constexpr int kU = 2;
    uint32_t m2 = 0;
    const int64_t S = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; base < nvec;
         base += kU * S) {
        uint4 vd[kU], va[kU], vb[kU];
        int64_t ia[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int64_t i = base + u * S;
            ia[u] = i + ((i >> 4) << 4);
            const bool in = i < nvec && in_range(i, 1, nvec, status) &&
                            in_range(ia[u], 1, 2 * nvec, status) &&
                            in_range(ia[u] + 16, 1, 2 * nvec, status);
            vd[u] = in ? __ldg(dh + i) : make_uint4(0, 0, 0, 0);
            va[u] = in ? __ldg(ab + ia[u]) : make_uint4(0, 0, 0, 0);
            vb[u] = in ? __ldg(ab + ia[u] + 16) : make_uint4(0, 0, 0, 0);
        }
        uint32_t amag = 0;
#pragma unroll
        for (int u = 0; u < kU; ++u)
            amag = swiglu::fold_abs(amag, va[u]);
        uint4 ga[kU], gb[kU];
        // one branch per 16 elements, so that their chains interleave
        if (swiglu::small87(amag)) {
#pragma unroll
            for (int u = 0; u < kU; ++u)
                swiglu::swiglu_bwd8<false>(vd[u], va[u], vb[u], ga[u], gb[u]);
        } else {
#pragma unroll
            for (int u = 0; u < kU; ++u)
                swiglu::swiglu_bwd8<true>(vd[u], va[u], vb[u], ga[u], gb[u]);
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            if (base + u * S < nvec && in_range(ia[u] + 16, 1, 2 * nvec, status)) {
                dab[ia[u]] = ga[u];
                dab[ia[u] + 16] = gb[u];
                m2 = max_u16x2(max_u16x2(m2, ga[u]), gb[u]);
            }
        }
    }
    uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    __shared__ uint32_t warp_max[kAmaxThreads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0)
        warp_max[warp] = m;
    __syncthreads();
    if (warp == 0) {
        m = lane < kAmaxThreads / 32 ? warp_max[lane] : 0u;
        m = __reduce_max_sync(0xFFFFFFFFu, m);
        if (lane == 0) {
            if (m >= 0x7F80u)
                atomicOr(status, kStatusNonfinite);
            partials[blockIdx.x] = m << 16;
        }
    }
}

// Phase 2 of a full tile: thread t takes a 16-row x 4-column block of the
// parked codes (16 conflict-free 4-byte shared loads), transposes it with
// PRMT and writes four 16-byte column segments of q^T (8 consecutive threads
// write 128 contiguous bytes of one column).
__device__ __forceinline__ void transpose_out(const uint8_t *tile, uint8_t *__restrict__ qt,
                                              int64_t rows, int64_t cols, int64_t r0, int64_t c0,
                                              int t, unsigned *status)
{
    const int rs = t & 7;          // 16-row segment
    const int cg = t >> 3;         // 4-column group (0..31)
    const int chunk = cg >> 2;     // 16-byte chunk holding the 4 columns
    const int word = cg & 3;       // 4-byte word within the chunk
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int row = rs * 16 + i;
        const int pch = chunk ^ ((row >> 4) & 7);
        w[i] = *reinterpret_cast<const uint32_t *>(tile + row * kTile + pch * 16 + word * 4);
    }
    uint32_t col[4][4];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const uint32_t a = w[4 * g], b = w[4 * g + 1], c = w[4 * g + 2], d = w[4 * g + 3];
        const uint32_t t0 = __byte_perm(a, b, 0x5140), t1 = __byte_perm(c, d, 0x5140);
        const uint32_t t2 = __byte_perm(a, b, 0x7362), t3 = __byte_perm(c, d, 0x7362);
        col[0][g] = __byte_perm(t0, t1, 0x5410);
        col[1][g] = __byte_perm(t0, t1, 0x7632);
        col[2][g] = __byte_perm(t2, t3, 0x5410);
        col[3][g] = __byte_perm(t2, t3, 0x7632);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int64_t o = (c0 + cg * 4 + j) * rows + r0 + rs * 16;
        if (in_range(o, 16, rows * cols, status))
            *reinterpret_cast<uint4 *>(qt + o) =
                make_uint4(col[j][0], col[j][1], col[j][2], col[j][3]);
    }
}

template <int FMT>
__global__ void __launch_bounds__(kCastThreads)
cast_transpose_kernel(const uint16_t *__restrict__ x, int64_t rows, int64_t cols,
                      const float *__restrict__ amax, const unsigned *__restrict__ partials,
                      int nparts, float *__restrict__ amax_out, float *__restrict__ scale_out,
                      uint8_t *__restrict__ q, uint8_t *__restrict__ qt, int vector_ok,
                      unsigned *__restrict__ status)
{
    __shared__ __align__(16) uint8_t tile[kTile * kTile];
    griddep_wait();
    griddep_launch_dependents();
    const float a = partials != nullptr ? reduce_partials(partials, nparts) : *amax;
    const float s = scale_of<FMT>(a);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        if (scale_out != nullptr)
            *scale_out = s;
        if (amax_out != nullptr)
            *amax_out = a;
    }

    const int64_t tiles_c = (cols + kTile - 1) / kTile;
    const int64_t tiles_r = (rows + kTile - 1) / kTile;
    const int64_t ntiles = tiles_r * tiles_c;
    const int t = threadIdx.x;

    for (int64_t tix = blockIdx.x; tix < ntiles; tix += gridDim.x) {
        const int64_t r0 = (tix / tiles_c) * kTile;
        const int64_t c0 = (tix % tiles_c) * kTile;
        const bool full = vector_ok && r0 + kTile <= rows && c0 + kTile <= cols;
        if (full) {
            // ---- phase 1: rows in, row-major codes out, park in smem
#pragma unroll
            for (int it = 0; it < 4; ++it) {
                const int k = t + it * kCastThreads;  // 16-element chunk id in the tile
                const int row = k >> 3, ch = k & 7;
                const int64_t o = (r0 + row) * cols + c0 + ch * 16;
                const bool ok = in_range(o, 16, rows * cols, status);
                const uint16_t *src = x + o;
                const uint4 v0 = ok ? __ldg(reinterpret_cast<const uint4 *>(src)) : make_uint4(0, 0, 0, 0);
                const uint4 v1 = ok ? __ldg(reinterpret_cast<const uint4 *>(src + 8)) : make_uint4(0, 0, 0, 0);
                const uint2 a = cvt8<FMT>(v0, s), b = cvt8<FMT>(v1, s);
                const uint4 codes = make_uint4(a.x, a.y, b.x, b.y);
                if (q != nullptr && ok)
                    *reinterpret_cast<uint4 *>(q + o) = codes;
                const int pch = ch ^ ((row >> 4) & 7);
                *reinterpret_cast<uint4 *>(tile + row * kTile + pch * 16) = codes;
            }
            if (qt != nullptr) {
                __syncthreads();
                transpose_out(tile, qt, rows, cols, r0, c0, t, status);
            }
            __syncthreads();
        } else {
            // ragged or unaligned tile: one element at a time
            for (int e = t; e < kTile * kTile; e += kCastThreads) {
                const int64_t r = r0 + e / kTile, c = c0 + e % kTile;
                if (r < rows && c < cols && in_range(r * cols + c, 1, rows * cols, status) &&
                    in_range(c * rows + r, 1, rows * cols, status)) {
                    const uint8_t b = cvt1<FMT>(x[r * cols + c], s);
                    if (q != nullptr)
                        q[r * cols + c] = b;
                    if (qt != nullptr)
                        qt[c * rows + r] = b;
                }
            }
        }
    }
}

// The same cast for tensors whose sides are multiples of 128, with the bf16
// tiles brought in by TMA: a CTA keeps kInStages 32 KB input buffers and
// loads tiles k+1 .. k+kInStages-1 while it converts and transposes tile k,
// so the work of a tile overlaps the latency of the next ones.  Phase 1
// reads the tile from shared memory (16 bytes per thread, consecutive
// threads on consecutive bytes).  Two CTAs fit on an SM.
constexpr int kInBytes = kTile * kTile * 2;
constexpr int kInStages = 3;
constexpr int kTmaCastSmem = kInStages * kInBytes + kTile * kTile + 64 + 128;

// One tensor's share of a cast launch: shape, where its amax comes from and
// where its outputs go (outputs may be NULL).
struct CastSeg {
    int64_t rows, cols;
    const float *amax;
    const unsigned *partials;
    int nparts;
    float *amax_out, *scale_out;
    uint8_t *q, *qt;
};

// The tensors of one TMA cast launch: NS = 1, one tensor; NS =
// kMaxQuantTensors, nseg tensors whose tiles are numbered one after the
// other (first_tile[i] = tensor i's first tile).
template <int NS>
struct CastSet {
    CUtensorMap map[NS];
    CastSeg seg[NS];
    int64_t first_tile[NS + 1];
    int nseg;
    int early;   // 1: the inputs are complete before the dependency wait (the
                 // previous launch only read them: their amax pass)
    int reverse; // 1: tiles last first
};

// Tiles are taken in reverse launch order (the last tile first): the amax
// pass that precedes a cast walks each tensor front to back, so the tail of
// a tensor larger than L2 is what L2 still holds when the cast starts.
template <int FMT, int NS>
__global__ void __launch_bounds__(kCastThreads)
cast_transpose_tma_kernel(const __grid_constant__ CastSet<NS> set, unsigned *__restrict__ status,
                          uint64_t limit_ns)
{
    extern __shared__ uint8_t cast_smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(cast_smem_raw) + 127) &
                                              ~static_cast<uintptr_t>(127));
    uint8_t *tile = sm + kInStages * kInBytes;
    uint64_t *bar = reinterpret_cast<uint64_t *>(tile + kTile * kTile);
    __shared__ int abort_flag;
    __shared__ float s_scale[NS];
    const int t = threadIdx.x;
    const int nseg = NS == 1 ? 1 : set.nseg;
    const int64_t ntiles = set.first_tile[nseg];
    const int64_t nmine = ntiles > blockIdx.x ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    // the k-th tile of this CTA -> (tensor, tile row start, tile column start)
    auto locate = [&](int64_t k, int &sg, int64_t &r0, int64_t &c0) {
        const int64_t fwd = blockIdx.x + k * gridDim.x;
        const int64_t tix = set.reverse ? ntiles - 1 - fwd : fwd;
        sg = 0;
#pragma unroll
        for (int i = 1; i < NS; ++i)
            sg += (i < nseg && tix >= set.first_tile[i]) ? 1 : 0;
        const int64_t lt = tix - set.first_tile[sg];
        const int64_t tc = set.seg[sg].cols / kTile;
        r0 = (lt / tc) * kTile;
        c0 = (lt % tc) * kTile;
    };
    auto issue = [&](int64_t k) {
        int sg;
        int64_t r0, c0;
        locate(k, sg, r0, c0);
        const int b = static_cast<int>(k % kInStages);
        fence_proxy_async_shared();  // earlier generic reads of this buffer come first
        mbar_arrive_expect_tx(&bar[b], kInBytes);
        tma_load_2d(sm + b * kInBytes, &set.map[sg], &bar[b], static_cast<int32_t>(c0),
                    static_cast<int32_t>(r0));
    };
    if (t == 0) {
        for (int b = 0; b < kInStages; ++b)
            mbar_init(&bar[b], 1);
        abort_flag = 0;
        fence_mbar_init();
        for (int i = 0; i < nseg; ++i)
            tma_prefetch_desc(&set.map[i]);
        if (set.early)
            for (int64_t j = 0; j < nmine && j < kInStages - 1; ++j)
                issue(j);
    }
    __syncthreads();
    griddep_wait();
    griddep_launch_dependents();
    if (t == 0 && !set.early)
        for (int64_t j = 0; j < nmine && j < kInStages - 1; ++j)
            issue(j);
    // each tensor's amax: the block reduces its partial maxima (fp32 bit
    // patterns of non-negative values, so integer order is numeric order),
    // then its scale
    __shared__ unsigned s_amax[NS];
    if (t < nseg)
        s_amax[t] = 0u;
    __syncthreads();
    for (int i = 0; i < nseg; ++i) {
        const CastSeg &sg = set.seg[i];
        uint32_t m = 0;
        if (sg.partials != nullptr) {
            for (int j = t; j < sg.nparts; j += kCastThreads)
                m = max(m, sg.partials[j]);
        } else if (t == 0) {
            m = __float_as_uint(*sg.amax);
        }
        m = __reduce_max_sync(0xFFFFFFFFu, m);
        if ((t & 31) == 0 && m != 0u)
            atomicMax(&s_amax[i], m);
    }
    __syncthreads();
    if (t < nseg) {
        const float a = __uint_as_float(s_amax[t]);
        const float sc = scale_of<FMT>(a);
        s_scale[t] = sc;
        if (blockIdx.x == 0) {
            if (set.seg[t].scale_out != nullptr)
                *set.seg[t].scale_out = sc;
            if (set.seg[t].amax_out != nullptr)
                *set.seg[t].amax_out = a;
        }
    }
    __syncthreads();

    int64_t k = 0;
    for (; k < nmine; ++k) {
        if (t == 0 && k + kInStages - 1 < nmine)
            issue(k + kInStages - 1);  // its buffer was released at the end of iteration k - 1
        const int b = static_cast<int>(k % kInStages);
        if (!mbar_wait(&bar[b], static_cast<uint32_t>((k / kInStages) & 1), &abort_flag, limit_ns)) {
            abort_flag = 1;
            atomicOr(status, kStatusTimeout);
        }
        if (__syncthreads_or(abort_flag))
            break;
        int sg;
        int64_t r0, c0;
        locate(k, sg, r0, c0);
        const CastSeg &seg = set.seg[sg];
        const float s = s_scale[sg];
        const int64_t rows = seg.rows;
        const int64_t cols = seg.cols;
        uint8_t *q = seg.q;
        uint8_t *qt = seg.qt;
        const uint8_t *src = sm + b * kInBytes;
        // ---- phase 1: 8 passes of 16 rows; thread t converts 8 consecutive bf16
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            const int idx = p * kCastThreads + t;
            const int row = idx >> 4, c8 = idx & 15;
            const uint4 v = *reinterpret_cast<const uint4 *>(src + row * (kTile * 2) + c8 * 16);
            const uint2 codes = cvt8<FMT>(v, s);
            const int64_t o = (r0 + row) * cols + c0 + c8 * 8;
            if (q != nullptr && in_range(o, 8, rows * cols, status))
                *reinterpret_cast<uint2 *>(q + o) = codes;
            const int pch = (c8 >> 1) ^ ((row >> 4) & 7);
            *reinterpret_cast<uint2 *>(tile + row * kTile + pch * 16 + (c8 & 1) * 8) = codes;
        }
        __syncthreads();
        if (qt != nullptr)
            transpose_out(tile, qt, rows, cols, r0, c0, t, status);
        __syncthreads();  // the input buffer and the parked tile are free again
    }
    if (t == 0) {
        // gave up: the loads still in flight must land before the CTA exits
        // (loads are issued up to kInStages - 1 tiles ahead of k)
        for (int64_t j = k; j < nmine && j < k + kInStages; ++j)
            if (k < nmine)
                mbar_wait(&bar[j % kInStages], static_cast<uint32_t>((j / kInStages) & 1), nullptr,
                          limit_ns);
    }
}
} // namespace

namespace {

// Resident CTAs per SM of each kernel on each device (occupancy API, cached).
struct Occupancy {
    int amax_atomic = 0, amax_partials = 0, cast = 0, cast_tma = 0, swiglu = 0, swiglu_bwd = 0;
};
std::mutex g_occ_mutex;
Occupancy g_occ[64];

const Occupancy &occupancy(const DeviceInfo &dev)
{
    std::lock_guard<std::mutex> lock(g_occ_mutex);
    Occupancy &o = g_occ[dev.ordinal & 63];
    if (o.cast == 0) {
        int n = 0;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, amax_kernel<false>, kAmaxThreads, 0);
        o.amax_atomic = n > 0 ? n : 1;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, amax_kernel<true>, kAmaxThreads, 0);
        o.amax_partials = n > 0 ? n : 1;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, cast_transpose_kernel<0>, kCastThreads, 0);
        o.cast = n > 0 ? n : 1;
        cudaFuncSetAttribute(cast_transpose_tma_kernel<0, 1>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kTmaCastSmem);
        cudaFuncSetAttribute(cast_transpose_tma_kernel<1, 1>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kTmaCastSmem);
        cudaFuncSetAttribute(cast_transpose_tma_kernel<0, kMaxQuantTensors>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kTmaCastSmem);
        cudaFuncSetAttribute(cast_transpose_tma_kernel<1, kMaxQuantTensors>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kTmaCastSmem);
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, cast_transpose_tma_kernel<0, 1>,
                                                      kCastThreads, kTmaCastSmem);
        o.cast_tma = n > 0 ? n : 1;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, swiglu_amax_kernel, kAmaxThreads, 0);
        o.swiglu = n > 0 ? n : 1;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, swiglu_bwd_amax_kernel, kAmaxThreads, 0);
        o.swiglu_bwd = n > 0 ? n : 1;
    }
    return o;
}

bool tma_castable(int64_t rows, int64_t cols)
{
    return rows % kTile == 0 && cols % kTile == 0 && rows > 0 && cols > 0 && cast_tma_enabled();
}

int64_t amax_grid(int64_t nvec, int per_sm, const DeviceInfo &dev)
{
    int64_t blocks = (nvec + kAmaxThreads * kAmaxUnroll - 1) / (kAmaxThreads * kAmaxUnroll);
    const int64_t cap = static_cast<int64_t>(dev.sm_count) * per_sm;
    if (blocks > cap)
        blocks = cap;
    if (blocks > kMaxAmaxPartials)
        blocks = kMaxAmaxPartials;
    return blocks < 1 ? 1 : blocks;
}

} // namespace

cudaError_t launch_amax(const void *x, int64_t n, float *amax_out, const DeviceInfo &dev,
                        cudaStream_t stream)
{
    cudaError_t err = cudaMemsetAsync(amax_out, 0, sizeof(float), stream);
    if (err != cudaSuccess)
        return err;
    const int64_t nvec = n / 8;
    const int ntail = static_cast<int>(n % 8);
    const uint16_t *tail = static_cast<const uint16_t *>(x) + nvec * 8;
    const int64_t blocks = amax_grid(nvec, occupancy(dev).amax_atomic, dev);
    // follows a memset, so it is launched without programmatic serialization
    count_launch();
    amax_kernel<false><<<static_cast<unsigned>(blocks), kAmaxThreads, 0, stream>>>(
        static_cast<const uint4 *>(x), nvec, tail, ntail, reinterpret_cast<unsigned *>(amax_out),
        dev.status);
    return cudaGetLastError();
}

cudaError_t launch_amax_partials(const void *x, int64_t n, unsigned *partials, int *nparts,
                                 const DeviceInfo &dev, cudaStream_t stream)
{
    const int64_t nvec = n / 8;
    const int ntail = static_cast<int>(n % 8);
    const uint16_t *tail = static_cast<const uint16_t *>(x) + nvec * 8;
    const int64_t blocks = amax_grid(nvec, occupancy(dev).amax_partials, dev);
    *nparts = static_cast<int>(blocks);
    return launch_pdl(amax_kernel<true>, dim3(static_cast<unsigned>(blocks)), dim3(kAmaxThreads), 0,
                      stream, static_cast<const uint4 *>(x), nvec, tail, ntail, partials,
                      dev.status);
}

cudaError_t launch_cast_transpose(const void *x, int64_t rows, int64_t cols, const float *amax,
                                  const unsigned *partials, int nparts, float *amax_out,
                                  float *scale_out, uint8_t *q, uint8_t *q_t, int fmt,
                                  const DeviceInfo &dev, cudaStream_t stream, bool early)
{
    const int64_t ntiles = ((rows + kTile - 1) / kTile) * ((cols + kTile - 1) / kTile);
    CUtensorMap map;
    if (tma_castable(rows, cols) &&
        make_tensor_map_2d(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, rows, cols, kTile, kTile,
                           CU_TENSOR_MAP_SWIZZLE_NONE)) {
        int64_t blocks = ntiles;
        const int64_t cap = static_cast<int64_t>(dev.sm_count) * occupancy(dev).cast_tma;
        if (blocks > cap)
            blocks = cap;
        CastSet<1> set;
        set.map[0] = map;
        set.seg[0] = CastSeg{rows, cols, amax, partials, nparts, amax_out, scale_out, q, q_t};
        set.first_tile[0] = 0;
        set.first_tile[1] = ntiles;
        set.nseg = 1;
        set.early = early ? 1 : 0;
        set.reverse = cast_reverse_enabled() ? 1 : 0;
        return launch_pdl(fmt == 1 ? cast_transpose_tma_kernel<1, 1> : cast_transpose_tma_kernel<0, 1>,
                          dim3(static_cast<unsigned>(blocks)), dim3(kCastThreads), kTmaCastSmem,
                          stream, set, dev.status, wait_limit_ns());
    }
    int64_t blocks = ntiles;
    const int64_t cap = static_cast<int64_t>(dev.sm_count) * occupancy(dev).cast;
    if (blocks > cap)
        blocks = cap;
    if (blocks < 1)
        blocks = 1;
    const int vector_ok = (rows % 16 == 0) && (cols % 16 == 0);
    return launch_pdl(fmt == 1 ? cast_transpose_kernel<1> : cast_transpose_kernel<0>,
                      dim3(static_cast<unsigned>(blocks)), dim3(kCastThreads),
                      0, stream, static_cast<const uint16_t *>(x), rows, cols, amax, partials, nparts,
                      amax_out, scale_out, q, q_t, vector_ok, dev.status);
}

cudaError_t launch_quantize_swiglu(const void *a, const void *b, void *h, int64_t rows,
                                   int64_t cols, unsigned *partials, float *amax_out,
                                   float *scale_out, uint8_t *q, uint8_t *q_t, const DeviceInfo &dev,
                                   cudaStream_t stream)
{
    const int64_t n = rows * cols;
    const int64_t nvec = n / 8;
    const int ntail = static_cast<int>(n % 8);
    int64_t blocks = (nvec + kAmaxThreads * 4 - 1) / (kAmaxThreads * 4);
    const int64_t cap = static_cast<int64_t>(dev.sm_count) * occupancy(dev).swiglu;
    if (blocks > cap)
        blocks = cap;
    if (blocks > kMaxAmaxPartials)
        blocks = kMaxAmaxPartials;
    if (blocks < 1)
        blocks = 1;
    const uint16_t *a16 = static_cast<const uint16_t *>(a), *b16 = static_cast<const uint16_t *>(b);
    uint16_t *h16 = static_cast<uint16_t *>(h);
    cudaError_t e = launch_pdl(swiglu_amax_kernel, dim3(static_cast<unsigned>(blocks)),
                               dim3(kAmaxThreads), 0, stream, static_cast<const uint4 *>(a),
                               static_cast<const uint4 *>(b), static_cast<uint4 *>(h), nvec,
                               a16 + nvec * 8, b16 + nvec * 8, h16 + nvec * 8, ntail, partials,
                               dev.status);
    if (e != cudaSuccess)
        return e;
    return launch_cast_transpose(h, rows, cols, nullptr, partials, static_cast<int>(blocks), amax_out,
                                 scale_out, q, q_t, 0, dev, stream);
}

cudaError_t launch_swiglu_bwd_amax(const void *dh, const void *ab, void *dab, int64_t M, int64_t F,
                                   unsigned *partials, int *nparts, const DeviceInfo &dev,
                                   cudaStream_t stream)
{
    const int64_t nvec = M * F / 8;
    int64_t blocks = (nvec + kAmaxThreads * 2 - 1) / (kAmaxThreads * 2);
    const int64_t cap = static_cast<int64_t>(dev.sm_count) * occupancy(dev).swiglu_bwd;
    if (blocks > cap)
        blocks = cap;
    if (blocks > kMaxAmaxPartials)
        blocks = kMaxAmaxPartials;
    if (blocks < 1)
        blocks = 1;
    *nparts = static_cast<int>(blocks);
    return launch_pdl(swiglu_bwd_amax_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kAmaxThreads),
                      0, stream, static_cast<const uint4 *>(dh), static_cast<const uint4 *>(ab),
                      static_cast<uint4 *>(dab), nvec, partials, dev.status);
}

cudaError_t launch_quantize_multi(const QuantDesc *t, int n, int fmt, unsigned *parts,
                                  const DeviceInfo &dev, cudaStream_t stream)
{
    if (n < 1 || n > kMaxQuantTensors || (fmt != 0 && fmt != 1))
        return cudaErrorInvalidValue;
    CastSet<kMaxQuantTensors> set;
    AmaxSegs segs;
    int64_t nvec_total = 0;
    for (int i = 0; i < n; ++i) {
        if (!tma_castable(t[i].rows, t[i].cols) ||
            !make_tensor_map_2d(&set.map[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, t[i].x, t[i].rows,
                                t[i].cols, kTile, kTile, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorNotSupported;
        segs.x[i] = static_cast<const uint4 *>(t[i].x);
        segs.nvec[i] = t[i].rows * t[i].cols / 8;
        nvec_total += segs.nvec[i];
    }
    const Occupancy &occ = occupancy(dev);
    // the amax blocks, shared in proportion to the tensors' sizes (each at
    // least one, at most kMaxAmaxPartials / kMaxQuantTensors)
    const int64_t total = amax_grid(nvec_total, occ.amax_partials, dev);
    constexpr int kPartsPer = kMaxAmaxPartials / kMaxQuantTensors;
    segs.first_block[0] = 0;
    set.first_tile[0] = 0;
    for (int i = 0; i < n; ++i) {
        int64_t b = (total * segs.nvec[i] + nvec_total / 2) / nvec_total;
        b = b < 1 ? 1 : (b > kPartsPer ? kPartsPer : b);
        segs.first_block[i + 1] = segs.first_block[i] + static_cast<int>(b);
        segs.parts[i] = parts + static_cast<size_t>(i) * kPartsPer;
        set.seg[i] = CastSeg{t[i].rows, t[i].cols, nullptr, segs.parts[i], static_cast<int>(b),
                             t[i].amax_out, t[i].scale_out, t[i].q, t[i].q_t};
        set.first_tile[i + 1] = set.first_tile[i] + (t[i].rows / kTile) * (t[i].cols / kTile);
    }
    for (int i = n; i < kMaxQuantTensors; ++i) {  // unused entries: copies, never read
        segs.x[i] = segs.x[0];
        segs.nvec[i] = 0;
        segs.parts[i] = segs.parts[0];
        segs.first_block[i + 1] = segs.first_block[n];
        set.map[i] = set.map[0];
        set.seg[i] = set.seg[0];
        set.first_tile[i + 1] = set.first_tile[n];
    }
    segs.nseg = n;
    set.nseg = n;
    set.early = 1;  // the amax launch just before only reads the inputs
    set.reverse = cast_reverse_enabled() ? 1 : 0;
    cudaError_t e = launch_pdl(amax_multi_kernel, dim3(static_cast<unsigned>(segs.first_block[n])),
                               dim3(kAmaxThreads), 0, stream, segs, dev.status);
    if (e != cudaSuccess)
        return e;
    int64_t blocks = set.first_tile[n];
    const int64_t cap = static_cast<int64_t>(dev.sm_count) * occ.cast_tma;
    if (blocks > cap)
        blocks = cap;
    return launch_pdl(fmt == 1 ? cast_transpose_tma_kernel<1, kMaxQuantTensors>
                               : cast_transpose_tma_kernel<0, kMaxQuantTensors>,
                      dim3(static_cast<unsigned>(blocks)), dim3(kCastThreads), kTmaCastSmem, stream,
                      set, dev.status, wait_limit_ns());
}

bool quantize_multi_castable(const QuantDesc *t, int n)
{
    for (int i = 0; i < n; ++i)
        if (!tma_castable(t[i].rows, t[i].cols))
            return false;
    return n >= 1 && n <= kMaxQuantTensors;
}

namespace {
// Byte transpose out[c, r] = in[r, c] of a [rows, cols] uint8 tensor, 64 x 64
// tiles through shared memory (a padded row pitch keeps the column reads
// conflict-free); byte-wide, coalesced accesses.  Used on the FP8 weight
// all-gather path (q(W)^T of a gathered q(W)), not inside the linear.
constexpr int kTrTile = 64;
constexpr int kTrThreads = 256;

__global__ void __launch_bounds__(kTrThreads)
transpose_u8_kernel(const uint8_t *__restrict__ in, int64_t rows, int64_t cols,
                    uint8_t *__restrict__ out, unsigned *__restrict__ status)
{
    __shared__ uint8_t tile[kTrTile][kTrTile + 1];
    griddep_wait();
    griddep_launch_dependents();
    const int64_t tiles_c = (cols + kTrTile - 1) / kTrTile;
    const int64_t ntiles = ((rows + kTrTile - 1) / kTrTile) * tiles_c;
    const int64_t n = rows * cols;
    for (int64_t tix = blockIdx.x; tix < ntiles; tix += gridDim.x) {
        const int64_t r0 = (tix / tiles_c) * kTrTile, c0 = (tix % tiles_c) * kTrTile;
        for (int e = threadIdx.x; e < kTrTile * kTrTile; e += kTrThreads) {
            const int r = e / kTrTile, c = e % kTrTile;
            const int64_t o = (r0 + r) * cols + c0 + c;
            if (r0 + r < rows && c0 + c < cols && in_range(o, 1, n, status))
                tile[r][c] = in[o];
        }
        __syncthreads();
        for (int e = threadIdx.x; e < kTrTile * kTrTile; e += kTrThreads) {
            const int c = e / kTrTile, r = e % kTrTile;
            const int64_t o = (c0 + c) * rows + r0 + r;
            if (r0 + r < rows && c0 + c < cols && in_range(o, 1, n, status))
                out[o] = tile[r][c];
        }
        __syncthreads();
    }
}

// The same transpose for rows and cols multiples of 128 and 16-byte aligned
// buffers: 128 x 128 tiles, each row read as 16-byte chunks into the
// swizzled shared tile of the TMA cast, then written by the cast's PRMT
// transpose (transpose_out) as 16-byte column segments.
__global__ void __launch_bounds__(kCastThreads)
transpose_u8_tile_kernel(const uint8_t *__restrict__ in, int64_t rows, int64_t cols,
                         uint8_t *__restrict__ out, unsigned *__restrict__ status)
{
    __shared__ __align__(16) uint8_t tile[kTile * kTile];
    griddep_wait();
    griddep_launch_dependents();
    const int t = threadIdx.x;
    const int64_t tiles_c = cols / kTile;
    const int64_t ntiles = (rows / kTile) * tiles_c;
    const int64_t n = rows * cols;
    for (int64_t tix = blockIdx.x; tix < ntiles; tix += gridDim.x) {
        const int64_t r0 = (tix / tiles_c) * kTile, c0 = (tix % tiles_c) * kTile;
#pragma unroll
        for (int p = 0; p < kTile * kTile / 16 / kCastThreads; ++p) {
            const int idx = p * kCastThreads + t;
            const int row = idx >> 3, ch = idx & 7;   // 8 threads read one 128-byte row
            const int64_t o = (r0 + row) * cols + c0 + ch * 16;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (in_range(o, 16, n, status))
                v = *reinterpret_cast<const uint4 *>(in + o);
            *reinterpret_cast<uint4 *>(tile + row * kTile + ((ch ^ ((row >> 4) & 7)) * 16)) = v;
        }
        __syncthreads();
        transpose_out(tile, out, rows, cols, r0, c0, t, status);
        __syncthreads();  // the tile is free again
    }
}
} // namespace

cudaError_t launch_transpose_u8(const uint8_t *in, int64_t rows, int64_t cols, uint8_t *out,
                                const DeviceInfo &dev, cudaStream_t stream)
{
    if (rows % kTile == 0 && cols % kTile == 0 && reinterpret_cast<uintptr_t>(in) % 16 == 0 &&
        reinterpret_cast<uintptr_t>(out) % 16 == 0) {
        int64_t blocks = (rows / kTile) * (cols / kTile);
        const int64_t cap = static_cast<int64_t>(dev.sm_count) * 4;
        if (blocks > cap)
            blocks = cap;
        return launch_pdl(transpose_u8_tile_kernel, dim3(static_cast<unsigned>(blocks)),
                          dim3(kCastThreads), 0, stream, in, rows, cols, out, dev.status);
    }
    const int64_t ntiles = ((rows + kTrTile - 1) / kTrTile) * ((cols + kTrTile - 1) / kTrTile);
    int64_t blocks = ntiles;
    const int64_t cap = static_cast<int64_t>(dev.sm_count) * 8;
    if (blocks > cap)
        blocks = cap;
    if (blocks < 1)
        blocks = 1;
    return launch_pdl(transpose_u8_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kTrThreads), 0,
                      stream, in, rows, cols, out, dev.status);
}

namespace {
// One thread asks in_range about an element past the end of a 1-element
// buffer and touches no memory: the checked build records kStatusBounds.
__global__ void bounds_selftest_kernel(unsigned *status) { (void)in_range(1, 1, 1, status); }
} // namespace

bool bounds_checked_build() { return kBoundsCheck; }

cudaError_t launch_bounds_selftest(const DeviceInfo &dev, cudaStream_t stream)
{
    count_launch();
    bounds_selftest_kernel<<<1, 1, 0, stream>>>(dev.status);
    return cudaGetLastError();
}

} // namespace f8
