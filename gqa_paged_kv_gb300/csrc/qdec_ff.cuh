// qdec_ff.cuh -- float-float arithmetic and the appended key row, shared by
// the decode and prefill kernels of libqdec.  Not part of the ABI.
//
// The appended key is bf16(k_rot) rounded to nearest-even from the exact
// value: norm and rotation are carried in unevaluated float pairs (about 48
// significant bits, fp32 operations only -- the GPU's fp64 rate is a small
// fraction of its fp32 rate) and rounded once.
#pragma once

#include "qdec_internal.h"

namespace qdec {

// ----------------------------------------------------- float-float math --
// Unevaluated sums hi + lo of two floats (Dekker 1971; Knuth's TwoSum):
// ~48 significant bits from fp32 arithmetic, so the appended key can be
// rounded to bf16 as if from the exact value without fp64 (which GB300
// executes at a small fraction of its fp32 rate).
struct ff {
    float hi, lo;
};
static __device__ __forceinline__ ff two_sum(float a, float b) {
    const float s = a + b;
    const float bb = s - a;
    return {s, (a - (s - bb)) + (b - bb)};
}
static __device__ __forceinline__ ff fast_two_sum(float a, float b) {  // |a| >= |b|
    const float s = a + b;
    return {s, b - (s - a)};
}
static __device__ __forceinline__ ff two_prod(float a, float b) {
    const float p = a * b;
    return {p, fmaf(a, b, -p)};
}
static __device__ __forceinline__ ff ff_add(ff a, ff b) {
    ff s = two_sum(a.hi, b.hi);
    const ff t = two_sum(a.lo, b.lo);
    s.lo += t.hi;
    s = fast_two_sum(s.hi, s.lo);
    s.lo += t.lo;
    return fast_two_sum(s.hi, s.lo);
}
static __device__ __forceinline__ ff ff_neg(ff a) { return {-a.hi, -a.lo}; }
static __device__ __forceinline__ ff ff_mul(ff a, ff b) {
    ff p = two_prod(a.hi, b.hi);
    p.lo += a.hi * b.lo + a.lo * b.hi;
    return fast_two_sum(p.hi, p.lo);
}
static __device__ __forceinline__ ff ff_mul_f(ff a, float b) {
    ff p = two_prod(a.hi, b);
    p.lo += a.lo * b;
    return fast_two_sum(p.hi, p.lo);
}
// Round hi + lo to bf16, nearest-even: hi is the float nearest to the exact
// sum, so the two differ in bf16 only when hi sits exactly on a bf16
// midpoint, where the sign of lo decides.
static __device__ __forceinline__ __nv_bfloat16 ff_to_bf16(ff y) {
    const uint32_t u = __float_as_uint(y.hi);
    if ((u & 0xFFFFu) == 0x8000u && y.lo != 0.0f) {
        const uint32_t toward_zero = u & 0xFFFF0000u;
        const bool away = (y.lo > 0.0f) == (y.hi > 0.0f);
        return __ushort_as_bfloat16(
            static_cast<unsigned short>((away ? toward_zero + 0x10000u : toward_zero) >> 16));
    }
    return __float2bfloat16_rn(y.hi);
}

// ---------------------------------------------- cos and sin, float-float --
// (cos theta, sin theta) as normalised float pairs (about 46 significant
// bits), from fp32 arithmetic after a double-precision argument reduction
// (the GPU's fp64 rate makes a double sincos per angle the bound of a kernel
// that needs many angles).  Reduction (Cody and Waite 1980): k = the integer
// nearest theta * 2/pi, r = theta - k pi/2 with pi/2 the sum of two doubles,
// both products through fused multiply-adds, so |r| <= pi/4 (plus rounding)
// with an absolute error near 1e-16 for |k| < 2^31.  Then the Taylor series
// about 0 in x = r (a float pair) and x^2: sin x = x + x x^2 P(x^2), cos x =
// 1 + x^2 Q(x^2), P and Q with the coefficients (-1)^n / (2n+1)! and
// (-1)^n / (2n+2)!; the terms whose magnitude stays below 1e-7 are summed in
// float, the rest in float-float.  The remainders after x^17 and x^18 are
// below 1e-19 for |x| <= pi/4.  The quadrant k mod 4 swaps and negates.
static __device__ __forceinline__ ff ff_const(double d) {
    const float h = static_cast<float>(d);
    return {h, static_cast<float>(d - static_cast<double>(h))};
}
static __device__ RopeEntry ff_sincos(double theta) {
    constexpr double kHalfPiHi = 1.5707963267948966;      // pi/2 rounded to a double
    constexpr double kHalfPiLo = 6.123233995736766e-17;   // pi/2 minus that, rounded
    constexpr double kTwoOverPi = 0.6366197723675814;
    const double kq = rint(theta * kTwoOverPi);
    double r = fma(-kq, kHalfPiHi, theta);
    r = fma(-kq, kHalfPiLo, r);
    const int q = static_cast<int>(static_cast<long long>(kq) & 3);
    const float rh = static_cast<float>(r);
    const ff x = {rh, static_cast<float>(r - static_cast<double>(rh))};
    const ff x2 = ff_mul(x, x);
    const float z = x2.hi;
    // 1/n! for n = 2 .. 18
    constexpr double f2 = 1.0 / 2, f3 = f2 / 3, f4 = f3 / 4, f5 = f4 / 5, f6 = f5 / 6,
                     f7 = f6 / 7, f8 = f7 / 8, f9 = f8 / 9, f10 = f9 / 10, f11 = f10 / 11,
                     f12 = f11 / 12, f13 = f12 / 13, f14 = f13 / 14, f15 = f14 / 15,
                     f16 = f15 / 16, f17 = f16 / 17, f18 = f17 / 18;
    // sin: P = -f3 + z (f5 + z (-f7 + z (f9 + z (-f11 + z (f13 + z (-f15 + z f17))))))
    const float ts = static_cast<float>(-f11) +
                     z * (static_cast<float>(f13) +
                          z * (static_cast<float>(-f15) + z * static_cast<float>(f17)));
    ff ps = ff_add(ff_const(f9), ff_mul_f(x2, ts));
    ps = ff_add(ff_const(-f7), ff_mul(x2, ps));
    ps = ff_add(ff_const(f5), ff_mul(x2, ps));
    ps = ff_add(ff_const(-f3), ff_mul(x2, ps));
    const ff sn = ff_add(x, ff_mul(x, ff_mul(x2, ps)));
    // cos: Q = -f2 + z (f4 + z (-f6 + z (f8 + z (-f10 + z (f12 + z (-f14 + z (f16 - z f18)))))))
    const float tc = static_cast<float>(f12) +
                     z * (static_cast<float>(-f14) +
                          z * (static_cast<float>(f16) + z * static_cast<float>(-f18)));
    ff pc = ff_add(ff_const(-f10), ff_mul_f(x2, tc));
    pc = ff_add(ff_const(f8), ff_mul(x2, pc));
    pc = ff_add(ff_const(-f6), ff_mul(x2, pc));
    pc = ff_add(ff_const(f4), ff_mul(x2, pc));
    pc = ff_add(ff_const(-f2), ff_mul(x2, pc));
    const ff cs = ff_add(ff{1.0f, 0.0f}, ff_mul(x2, pc));
    // theta = r + q pi/2
    const ff c = (q == 0) ? cs : (q == 1) ? ff_neg(sn) : (q == 2) ? ff_neg(cs) : sn;
    const ff s = (q == 0) ? sn : (q == 1) ? cs : (q == 2) ? ff_neg(sn) : ff_neg(cs);
    return {c.hi, c.lo, s.hi, s.lo};
}

// Whether every value within err of y has the same nearest-even bf16 as y:
// y is a normal float, no bf16 rounding boundary (the midpoint of two
// consecutive bf16 values) lies within err of it, and err is below an eighth
// of its bf16 spacing (so the boundaries of the neighbouring intervals, at
// least a quarter spacing away, are out of reach too).
static __device__ __forceinline__ bool bf16_rounding_certain(float y, float err) {
    const uint32_t a = __float_as_uint(y) & 0x7FFFFFFFu;
    if (a < 0x00800000u || a >= 0x7F800000u) return false;  // zero, subnormal, inf, NaN
    const float mid = __uint_as_float((a & 0xFFFF0000u) | 0x8000u);
    const float eighth = __uint_as_float(a & 0x7F800000u) * 0x1p-10f;  // 2^e x 2^-7 / 8
    return fabsf(__uint_as_float(a) - mid) > err && err < eighth;  // the difference is exact
}

// The new key row (sequence b, KV head g) on one warp, lane l holding dims
// 2l, 2l+1, 64+2l, 65+2l: RMSNorm and RoPE, one rounding to bf16, the
// nearest-even bf16 of the exact value.  x*w is exact in fp32 (two bf16
// values), so is x^2.
//
// First in fp32, with an a-priori bound on the error (u = 2^-24): the sum of
// squares passes through at most 7 roundings (8u relative, all terms
// positive); v = ss/D + eps one more (9u); r = 1/sqrt(v) by IEEE square root
// and division (6.5u); n = (x w) r one more (7.5u); the rotated element
// y = n_a c - n_b s as fma(n_a, c, -fl(n_b s)) with c, s the float parts of
// the angle (u each): |y32 - y| <= 9.6u (|n_a c| + |n_b s|) + 1.01u |y32|,
// below 16u (|n_a c| + |n_b s| + |y32|) as computed.  When no element of the
// row lies that close to a bf16 rounding boundary (most rows), its rounding
// is final; otherwise the whole row is redone in float-float arithmetic
// (about 48 significant bits).  Rows with a sum of squares under 2^-100 (or
// not finite) take the float-float path as well, where the bound's premises
// (no underflow in x^2 or x w) could fail.
static __device__ void key_row(float eps, __nv_bfloat162 ka, __nv_bfloat162 kc, __nv_bfloat162 wa,
                        __nv_bfloat162 wc, const RopeEntry &e0, const RopeEntry &e1,
                        __nv_bfloat16 (&kb)[4]) {
    const float x[4] = {__low2float(ka), __high2float(ka), __low2float(kc), __high2float(kc)};
    const float wv[4] = {__low2float(wa), __high2float(wa), __low2float(wc), __high2float(wc)};
    {
        float sq = __fadd_rn(__fadd_rn(__fmul_rn(x[0], x[0]), __fmul_rn(x[1], x[1])),
                             __fadd_rn(__fmul_rn(x[2], x[2]), __fmul_rn(x[3], x[3])));
#pragma unroll
        for (int o = 16; o; o >>= 1) sq = __fadd_rn(sq, __shfl_xor_sync(0xffffffffu, sq, o));
        const float v = fmaf(sq, 1.0f / kHeadDim, eps);
        const float r = __fdiv_rn(1.0f, __fsqrt_rn(v));
        float n[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) n[e] = __fmul_rn(__fmul_rn(x[e], wv[e]), r);
        // element e rotates n[e] and n[e ^ 2] by angle e & 1
        float y[4];
        bool ok = sq >= 0x1p-100f && sq <= 0x1p100f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float c = (e & 1) ? e1.c_hi : e0.c_hi, sn = (e & 1) ? e1.s_hi : e0.s_hi;
            const float a = n[e], b = n[e ^ 2];
            // e < 2: a c - b s; e >= 2: a c + b s (b is the first half)
            const float t = __fmul_rn(b, sn);
            y[e] = fmaf(a, c, e < 2 ? -t : t);
            const float mag = __fadd_rn(fabsf(__fmul_rn(a, c)), fabsf(t));
            ok = ok && bf16_rounding_certain(y[e], 0x1p-20f * __fadd_rn(mag, fabsf(y[e])));
        }
        if (__all_sync(0xffffffffu, ok)) {
#pragma unroll
            for (int e = 0; e < 4; ++e) kb[e] = __float2bfloat16_rn(y[e]);
            return;
        }
    }
    ff ss = {x[0] * x[0], 0.f};
#pragma unroll
    for (int e = 1; e < 4; ++e) ss = ff_add(ss, ff{x[e] * x[e], 0.f});
#pragma unroll
    for (int o = 16; o; o >>= 1)
        ss = ff_add(ss, ff{__shfl_xor_sync(0xffffffffu, ss.hi, o), __shfl_xor_sync(0xffffffffu, ss.lo, o)});
    const ff v = ff_add(ff{ss.hi * (1.0f / kHeadDim), ss.lo * (1.0f / kHeadDim)}, ff{eps, 0.f});
    // r = 1/sqrt(v): one Newton step from rsqrtf in float-float
    const float r0 = rsqrtf(v.hi);
    const ff t = ff_mul(v, two_prod(r0, r0));          // v * r0^2, close to 1
    const float h = (1.0f - t.hi) - t.lo;              // 1 - t.hi is exact there
    const ff r = fast_two_sum(r0, 0.5f * r0 * h);
    ff xh[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) xh[e] = ff_mul_f(r, x[e] * wv[e]);
    const ff c0 = {e0.c_hi, e0.c_lo}, s0 = {e0.s_hi, e0.s_lo};
    const ff c1 = {e1.c_hi, e1.c_lo}, s1 = {e1.s_hi, e1.s_lo};
    kb[0] = ff_to_bf16(ff_add(ff_mul(xh[0], c0), ff_neg(ff_mul(xh[2], s0))));
    kb[2] = ff_to_bf16(ff_add(ff_mul(xh[2], c0), ff_mul(xh[0], s0)));
    kb[1] = ff_to_bf16(ff_add(ff_mul(xh[1], c1), ff_neg(ff_mul(xh[3], s1))));
    kb[3] = ff_to_bf16(ff_add(ff_mul(xh[3], c1), ff_mul(xh[1], s1)));
}


}  // namespace qdec
