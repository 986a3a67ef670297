// Double-float arithmetic in fp32 instructions (sm_103a): exact error-free
// transformations (TwoSum, TwoProd by fma) and values hi + lo with
// ~2^-44 relative precision.  fp64 throughput is very low on this part, so
// the exact re-decisions use these instead.
#pragma once

#include <cuda_fp16.h>

namespace kvc {
namespace {

// s + e = a + b exactly (Knuth's TwoSum).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}

// Double-float values (hi + lo, |lo| <= ulp(hi) / 2): ~2^-44 relative
// precision with fp32 instructions only (fp64 throughput is very low here).
struct ff2 {
  float hi, lo;
};

__device__ __forceinline__ ff2 fast_two_sum(float a, float b) {  // |a| >= |b|
  const float s = a + b;
  return ff2{s, b - (s - a)};
}
__device__ __forceinline__ ff2 ff_add(ff2 a, ff2 b) {
  float s, e;
  two_sum(a.hi, b.hi, s, e);
  e += a.lo + b.lo;
  return fast_two_sum(s, e);
}
__device__ __forceinline__ ff2 ff_mul(ff2 a, ff2 b) {
  const float p = a.hi * b.hi;
  float e = fmaf(a.hi, b.hi, -p);
  e = fmaf(a.hi, b.lo, e);
  e = fmaf(a.lo, b.hi, e);
  return fast_two_sum(p, e);
}
__device__ __forceinline__ ff2 ff_sqrt(ff2 a) {  // a >= 0
  const float h = sqrtf(a.hi);
  if (h == 0.f) return ff2{0.f, 0.f};
  const float r = fmaf(-h, h, a.hi) + a.lo;
  return fast_two_sum(h, r / (2.f * h));
}
__device__ __forceinline__ bool ff_less(ff2 a, ff2 b) {
  return a.hi < b.hi || (a.hi == b.hi && a.lo < b.lo);
}

// a / b for an integer-valued b > 0, to ~2^-44.
__device__ __forceinline__ ff2 ff_div_f(ff2 a, float b) {
  const float q1 = a.hi / b;
  const float r = fmaf(-q1, b, a.hi) + a.lo;
  return fast_two_sum(q1, r / b);
}
// a / b, to ~2^-44 (b != 0).
__device__ __forceinline__ ff2 ff_div(ff2 a, ff2 b) {
  const float q1 = a.hi / b.hi;
  const ff2 r = ff_add(a, ff_mul(ff2{-q1, 0.f}, b));
  return fast_two_sum(q1, r.hi / b.hi);
}
__device__ __forceinline__ ff2 ff_abs(ff2 a) { return a.hi < 0.f ? ff2{-a.hi, -a.lo} : a; }
// rint(hi + lo), half to even: f = hi - rint(hi) is exact; lo matters only at
// an exact half of hi.
__device__ __forceinline__ float ff_rint(ff2 a) {
  const float r = rintf(a.hi), f = a.hi - r;
  if (f == 0.5f && a.lo > 0.f) return r + 1.f;
  if (f == -0.5f && a.lo < 0.f) return r - 1.f;
  return r;
}
// fp16 of hi + lo (>= 0): hi's rounding, unless hi is exactly halfway between
// two fp16 values, where lo's sign decides (lo = 0: hi's own tie rule).
__device__ __forceinline__ __half ff_to_half(ff2 a) {
  __half h = __float2half_rn(a.hi);
  const float hf = __half2float(h);
  if (hf != a.hi && a.lo != 0.f) {
    const unsigned short hb = __half_as_ushort(h);
    const unsigned short ob = hf < a.hi ? (unsigned short)(hb + 1) : (unsigned short)(hb - 1);
    const float of = __half2float(__ushort_as_half(ob));
    if (0.5f * (hf + of) == a.hi && ((of > hf) == (a.lo > 0.f))) h = __ushort_as_half(ob);
  }
  return h;
}

}  // namespace
}  // namespace kvc
