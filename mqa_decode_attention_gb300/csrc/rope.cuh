// RoPE angle helpers shared by the append kernel and the decode kernels.
#pragma once

#include <cuda_bf16.h>

namespace mqa {

// 2 pi = kTwoPi1 + kTwoPi2 + kTwoPi3 (leading double, then the next two
// 53-bit pieces of the remainder).
constexpr double kTwoPi1 = 6.283185307179586232;
constexpr double kTwoPi2 = 2.4492935982947063545e-16;
constexpr double kTwoPi3 = -5.9895396194366793e-33;
constexpr double kInvTwoPi = 0.15915494309189533577;

// Cody-Waite additive range reduction: x - k 2 pi with k the nearest integer
// to x / (2 pi), the product folded in piece by piece with fused
// multiply-adds. |x| < 2^40 here (position < 2^31, theta <= 1).
__device__ __forceinline__ double reduce_two_pi(double x) {
  const double k = rint(x * kInvTwoPi);
  double r = fma(-k, kTwoPi1, x);
  r = fma(-k, kTwoPi2, r);
  r = fma(-k, kTwoPi3, r);
  return r;
}

// cos / sin of pos * theta_i in fp64 (reduced argument), i = threadIdx-chosen
__device__ __forceinline__ void rope_cos_sin(int pos, double theta, double* c, double* s) {
  sincos(reduce_two_pi(static_cast<double>(pos) * theta), s, c);
}

// The key pair (x, y) turned by the reduced angle `ang` and rounded once to
// bf16: bit for bit the rounding of the fp64 rotation (fp64 sine and cosine
// of ang, round-to-nearest products and sum), at a fraction of its cost on a
// part whose fp64 rate is low. The rotation is formed first in fp32, from the
// fp32 sine and cosine of ang rounded to fp32, and again in fp64 only when
// the fp32 result's error interval holds a bf16 rounding boundary, or when
// s = |x| + |y| is zero, tiny, huge or not finite.
//
// Error bound, fp32 result against fp64 result: rounding |ang| <= pi + ulp to
// fp32 moves it by <= 2^-23; sincosf is within 2 ulp (<= 2^-22 here); so the
// fp32 cosine and sine are within 3.6e-7 of the fp64 ones. The product and
// the fused multiply-add add <= 2^-24 (|y| + s) <= 1.2e-7 s, the fp64
// arithmetic < 4e-16 s: |r32 - r64| < 4.8e-7 s. The bound used is 8e-7 s.
// Rounding to nearest is monotonic, so when r32 - bound and r32 + bound
// (each rounded outward) round to the same bf16, r64 rounds to it as well.
//
// rope_k_bf16_fast is the fp32 stage alone, given cf / sf = the fp32 cosine /
// sine of the reduced angle rounded to fp32: true, with *r set, when it
// decides the rounding; rope_k_bf16_fp64 the fp64 stage; rope_k_bf16 both.
__device__ __forceinline__ bool rope_k_bf16_fast(float x, float y, float cf, float sf, __nv_bfloat162* r) {
  const float s = fabsf(x) + fabsf(y);
  if (!(s >= 0x1p-100f && s <= 1e37f)) return false;
  const float xr = fmaf(x, cf, -(y * sf));
  const float yr = fmaf(x, sf, y * cf);
  const float e = s * 8e-7f;
  const __nv_bfloat16 xl = __float2bfloat16_rn(__fsub_rd(xr, e)), xh = __float2bfloat16_rn(__fadd_ru(xr, e));
  const __nv_bfloat16 yl = __float2bfloat16_rn(__fsub_rd(yr, e)), yh = __float2bfloat16_rn(__fadd_ru(yr, e));
  if (__bfloat16_as_ushort(xl) != __bfloat16_as_ushort(xh) || __bfloat16_as_ushort(yl) != __bfloat16_as_ushort(yh))
    return false;
  r->x = xl;
  r->y = yl;
  return true;
}

__device__ __forceinline__ __nv_bfloat162 rope_k_bf16_fp64(float x, float y, double ang) {
  double c, sn;
  sincos(ang, &sn, &c);
  const double xd = x, yd = y;
  __nv_bfloat162 r;
  r.x = __double2bfloat16(__dsub_rn(__dmul_rn(xd, c), __dmul_rn(yd, sn)));
  r.y = __double2bfloat16(__dadd_rn(__dmul_rn(xd, sn), __dmul_rn(yd, c)));
  return r;
}

__device__ __forceinline__ __nv_bfloat162 rope_k_bf16(float x, float y, double ang) {
  __nv_bfloat162 r;
  const float s = fabsf(x) + fabsf(y);
  if (s >= 0x1p-100f && s <= 1e37f) {
    float sf, cf;
    sincosf(static_cast<float>(ang), &sf, &cf);
    if (rope_k_bf16_fast(x, y, cf, sf, &r)) return r;
  }
  return rope_k_bf16_fp64(x, y, ang);
}

}  // namespace mqa
