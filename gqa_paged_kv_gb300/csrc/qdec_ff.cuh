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

// The new key row (sequence b, KV head g) on one warp, lane l holding dims
// 2l, 2l+1, 64+2l, 65+2l: RMSNorm and RoPE in float-float arithmetic, then
// one rounding to bf16.  x*w is exact in fp32 (two bf16 values), so is x^2.
static __device__ void key_row(float eps, __nv_bfloat162 ka, __nv_bfloat162 kc, __nv_bfloat162 wa,
                        __nv_bfloat162 wc, const RopeEntry &e0, const RopeEntry &e1,
                        __nv_bfloat16 (&kb)[4]) {
    const float x[4] = {__low2float(ka), __high2float(ka), __low2float(kc), __high2float(kc)};
    const float wv[4] = {__low2float(wa), __high2float(wa), __low2float(wc), __high2float(wc)};
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
