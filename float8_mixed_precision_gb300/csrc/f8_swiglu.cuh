// SwiGLU of bf16 pairs, shared by the producing pass (f8_cast.cu) and the
// W13 GEMM epilogue (f8_gemm.cu).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace f8 {
namespace swiglu {

// ---- the SwiGLU input of the w2 linear, h = bf16(silu(a) * b), and its
// gradient, evaluated in fp32 to within one bf16 ulp of the definition
// (silu(a) = a / (1 + exp(-a)) and its derivative in exact arithmetic,
// rounded once to bf16).  exp(x) is Cody and Waite's range reduction
// (x = n ln2 + r, ln2 split into a head exact in fp32 and a tail) with the
// degree-7 Taylor polynomial of exp(r) in Horner form, scaled by 2^n;
// silu(a) = a * (1 / (1 + exp(-a))) with the correctly rounded reciprocal.
// Two elements go through each packed fp32x2 instruction (per lane the
// numerics of the scalar _rn operation).  n = rint(x log2e) is taken as
// (p + 1.5 2^23) - 1.5 2^23, exact round-to-nearest-even for |p| < 2^22, and
// 2^n is read off the low mantissa bits of the rounded sum.
// Below a = -87, sigma(a) = e^a / (1 + e^a) rounds to e^a in fp32 and falls
// into fp32's subnormal range, where forming it would lose the bits that
// a sigma(a) b (a bf16 normal down to a = -92) still needs: there e^a =
// p 2^n is applied as 2^(n+64) before the products and 2^-64 after them
// (neg_tail), so every intermediate stays a normal fp32.
__device__ __forceinline__ float2 splat(float v) { return make_float2(v, v); }

__device__ __forceinline__ float exp_special(float x, float e)
{
    if (x != x)
        return x;
    if (x > 88.0f)
        return __int_as_float(0x7F800000);
    if (x < -87.0f)
        return 0.0f;
    return e;
}

// kChecked = false: the caller has shown -87 <= x <= 87 for both lanes (no
// NaN), where the special cases cannot arise and n stays in [-126, 126].
template <bool kChecked>
__device__ __forceinline__ float2 exp_cw2(float2 x)
{
    constexpr float kRound = 12582912.0f;  // 1.5 * 2^23
    const float2 p = __fmul2_rn(x, splat(1.44269502f));
    const float2 t = __fadd2_rn(p, splat(kRound));
    const float2 mn = __fadd2_rn(splat(kRound), make_float2(-t.x, -t.y));  // -rint(p)
    float2 r = __ffma2_rn(mn, splat(0.693145751953125f), x);
    r = __ffma2_rn(mn, splat(1.42860677e-06f), r);
    float2 q = __ffma2_rn(splat(0x1.a01a02p-13f), r, splat(0x1.6c16c2p-10f));
    q = __ffma2_rn(q, r, splat(0x1.111112p-7f));
    q = __ffma2_rn(q, r, splat(0x1.555556p-5f));
    q = __ffma2_rn(q, r, splat(0x1.555556p-3f));
    q = __ffma2_rn(q, r, splat(0.5f));
    q = __ffma2_rn(q, r, splat(1.0f));
    q = __ffma2_rn(q, r, splat(1.0f));
    // bits(t) = 0x4B400000 + n, and 0x4B400000 << 23 vanishes mod 2^32
    const float2 two_n = make_float2(__int_as_float((__float_as_int(t.x) << 23) + 0x3F800000),
                                     __int_as_float((__float_as_int(t.y) << 23) + 0x3F800000));
    const float2 e = __fmul2_rn(q, two_n);
    if (!kChecked)
        return e;
    return make_float2(exp_special(x.x, e.x), exp_special(x.y, e.y));
}

// 1/d correctly rounded, two lanes, for d in [1, 2^126): the hardware's
// approximate reciprocal refined by two Newton-Raphson steps in Markstein's
// residual form (e = 1 - d y by one FMA, then y + y e), and d = (2 - 2^-23)
// 2^k, the one input class the refinement can leave one ulp off, set to its
// correctly rounded reciprocal (1 + 2^-23) 2^-(k+1) directly.  Every
// significand of d has been checked against IEEE division with seeds up to
// 8 ulp off.  Branch-free, so consecutive elements interleave.
__device__ __forceinline__ float rcp_approx(float x)
{
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ float fix_all_ones(float d, float y)
{
    const uint32_t bd = __float_as_uint(d);
    return (bd & 0x7FFFFFu) == 0x7FFFFFu ? __uint_as_float(0x7E800001u - (bd & 0x7F800000u)) : y;
}

__device__ __forceinline__ float2 rcp2_refined(float2 d)
{
    const float2 nd = make_float2(-d.x, -d.y);
    float2 y = make_float2(rcp_approx(d.x), rcp_approx(d.y));
    float2 e = __ffma2_rn(nd, y, splat(1.0f));
    y = __ffma2_rn(y, e, y);
    e = __ffma2_rn(nd, y, splat(1.0f));
    y = __ffma2_rn(y, e, y);
    return make_float2(fix_all_ones(d.x, y.x), fix_all_ones(d.y, y.y));
}

// For a in [-110, -87): p 2^(n + 64) with e^a = p 2^n (n in [-159, -125],
// so 2^(n + 64) is a normal fp32).  Below -110, e^a < 2^-158 and 0 is
// returned: every product that uses it is then a signed zero (or NaN for an
// infinite factor), as the definition's is after rounding.
__device__ __forceinline__ float neg_tail_exp_scaled(float a)
{
    if (a < -110.0f)
        return 0.0f;
    constexpr float kRound = 12582912.0f;  // 1.5 * 2^23
    const float t = __fadd_rn(__fmul_rn(a, 1.44269502f), kRound);
    const float n = __fadd_rn(t, -kRound);
    float r = __fmaf_rn(-n, 0.693145751953125f, a);
    r = __fmaf_rn(-n, 1.42860677e-06f, r);
    float q = __fmaf_rn(0x1.a01a02p-13f, r, 0x1.6c16c2p-10f);
    q = __fmaf_rn(q, r, 0x1.111112p-7f);
    q = __fmaf_rn(q, r, 0x1.555556p-5f);
    q = __fmaf_rn(q, r, 0x1.555556p-3f);
    q = __fmaf_rn(q, r, 0.5f);
    q = __fmaf_rn(q, r, 1.0f);
    q = __fmaf_rn(q, r, 1.0f);
    const int ni = static_cast<int>(n);
    return __fmul_rn(q, __int_as_float((ni + 64 + 127) << 23));
}

// h for a < -87: (a e^a b), e^a applied as 2^(n+64) p, then 2^-64.
__device__ __forceinline__ float neg_tail_h(float a, float b)
{
    return __fmul_rn(__fmul_rn(__fmul_rn(a, neg_tail_exp_scaled(a)), b), 0x1p-64f);
}

// two packed bf16 of a and of b -> two packed bf16 of h.  kChecked = false
// requires |a| <= 87 in both lanes: exp needs no special values and
// 1 + exp(-a) lies in [1, 2^126), the refined reciprocal's range.
template <bool kChecked>
__device__ __forceinline__ uint32_t swiglu_x2(uint32_t a, uint32_t b)
{
    const float2 fa = make_float2(__uint_as_float(a << 16), __uint_as_float(a & 0xFFFF0000u));
    const float2 fb = make_float2(__uint_as_float(b << 16), __uint_as_float(b & 0xFFFF0000u));
    const float2 e = exp_cw2<kChecked>(make_float2(-fa.x, -fa.y));
    const float2 d = __fadd2_rn(splat(1.0f), e);
    const float2 r = kChecked ? make_float2(__frcp_rn(d.x), __frcp_rn(d.y)) : rcp2_refined(d);
    float2 hf = __fmul2_rn(__fmul2_rn(fa, r), fb);
    if (kChecked) {
        if (fa.x < -87.0f)
            hf.x = neg_tail_h(fa.x, fb.x);
        if (fa.y < -87.0f)
            hf.y = neg_tail_h(fa.y, fb.y);
    }
    const __nv_bfloat162 h = __floats2bfloat162_rn(hf.x, hf.y);
    return *reinterpret_cast<const uint32_t *>(&h);
}

template <bool kChecked>
__device__ __forceinline__ uint4 swiglu8(uint4 a, uint4 b)
{
    return make_uint4(swiglu_x2<kChecked>(a.x, b.x), swiglu_x2<kChecked>(a.y, b.y),
                      swiglu_x2<kChecked>(a.z, b.z), swiglu_x2<kChecked>(a.w, b.w));
}

// Packed maximum of |a| over eight bf16, to gate a group onto the fast path
// (every |a| <= 87, bf16 0x42AE, when small87 of the fold is true).
__device__ __forceinline__ uint32_t fold_abs(uint32_t m, uint4 a)
{
    constexpr uint32_t kMag = 0x7FFF7FFFu;
    return __vmaxu2(__vmaxu2(m, __vmaxu2(a.x & kMag, a.y & kMag)), __vmaxu2(a.z & kMag, a.w & kMag));
}

__device__ __forceinline__ bool small87(uint32_t m) { return __vcmpgtu2(m, 0x42AE42AEu) == 0; }

// The gradient of h = silu(a) b for two packed bf16 lanes of the upstream
// gradient dh: db = bf16(dh s) with s = a sigma, and da = bf16((dh b) ds)
// with ds = sigma fma(a, 1 - sigma, 1) = silu'(a); sigma as in the forward.
// Below a = -87 (kChecked only), sigma = e^a and 1 - sigma = 1 in fp32, so
// db = (a e^a) dh and da = ((1 + a) e^a) (dh b), with e^a applied as in
// neg_tail_h.  dh b is formed first in every case (exact in fp32 for
// bf16 factors unless it leaves fp32's range).
template <bool kChecked>
__device__ __forceinline__ void swiglu_bwd_x2(uint32_t dh, uint32_t a, uint32_t b, uint32_t &da,
                                              uint32_t &db)
{
    const float2 fa = make_float2(__uint_as_float(a << 16), __uint_as_float(a & 0xFFFF0000u));
    const float2 fb = make_float2(__uint_as_float(b << 16), __uint_as_float(b & 0xFFFF0000u));
    const float2 fd = make_float2(__uint_as_float(dh << 16), __uint_as_float(dh & 0xFFFF0000u));
    const float2 e = exp_cw2<kChecked>(make_float2(-fa.x, -fa.y));
    const float2 d = __fadd2_rn(splat(1.0f), e);
    const float2 sg = kChecked ? make_float2(__frcp_rn(d.x), __frcp_rn(d.y)) : rcp2_refined(d);
    float2 vdb = __fmul2_rn(fd, __fmul2_rn(fa, sg));
    const float2 t = __fadd2_rn(splat(1.0f), make_float2(-sg.x, -sg.y));
    const float2 ds = __fmul2_rn(sg, __ffma2_rn(fa, t, splat(1.0f)));
    const float2 g = __fmul2_rn(fd, fb);
    float2 vda = __fmul2_rn(g, ds);
    if (kChecked) {
        if (fa.x < -87.0f) {
            const float s = neg_tail_exp_scaled(fa.x);
            vdb.x = __fmul_rn(__fmul_rn(__fmul_rn(fa.x, s), fd.x), 0x1p-64f);
            vda.x = __fmul_rn(__fmul_rn(__fmul_rn(__fadd_rn(1.0f, fa.x), s), g.x), 0x1p-64f);
        }
        if (fa.y < -87.0f) {
            const float s = neg_tail_exp_scaled(fa.y);
            vdb.y = __fmul_rn(__fmul_rn(__fmul_rn(fa.y, s), fd.y), 0x1p-64f);
            vda.y = __fmul_rn(__fmul_rn(__fmul_rn(__fadd_rn(1.0f, fa.y), s), g.y), 0x1p-64f);
        }
    }
    const __nv_bfloat162 ha = __floats2bfloat162_rn(vda.x, vda.y);
    const __nv_bfloat162 hb = __floats2bfloat162_rn(vdb.x, vdb.y);
    da = *reinterpret_cast<const uint32_t *>(&ha);
    db = *reinterpret_cast<const uint32_t *>(&hb);
}

template <bool kChecked>
__device__ __forceinline__ void swiglu_bwd8(uint4 dh, uint4 a, uint4 b, uint4 &da, uint4 &db)
{
    swiglu_bwd_x2<kChecked>(dh.x, a.x, b.x, da.x, db.x);
    swiglu_bwd_x2<kChecked>(dh.y, a.y, b.y, da.y, db.y);
    swiglu_bwd_x2<kChecked>(dh.z, a.z, b.z, da.z, db.z);
    swiglu_bwd_x2<kChecked>(dh.w, a.w, b.w, da.w, db.w);
}

// |h| of a packed bf16 pair folded into a running packed maximum (bit order
// is numeric order for non-negative bf16; NaN and inf sort above all finite).
__device__ __forceinline__ uint32_t max_abs2(uint32_t m, uint32_t h2)
{
    return __vmaxu2(m, h2 & 0x7FFF7FFFu);
}

} // namespace swiglu
} // namespace f8
