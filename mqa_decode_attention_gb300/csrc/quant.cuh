// Byte-cache encoders shared by the append kernel and the decode kernels
// that perform the append themselves (fused step): both write the same bytes.
#pragma once

#include <cuda_fp16.h>

namespace mqa {

// uint8 quantisation of one (token, kv head) row in float32, in the order
// scale = (max - min) / 255 (1 if 0), zero = rint(-min / scale) clamped,
// code = rint(x / scale + zero) clamped (rint: nearest, ties to even).
__device__ __forceinline__ float2 u8_params(float mn, float mx) {
  float sc = __fdiv_rn(__fsub_rn(mx, mn), 255.0f);
  if (sc == 0.0f) sc = 1.0f;
  const float zp = fminf(fmaxf(rintf(__fdiv_rn(-mn, sc)), 0.0f), 255.0f);
  return make_float2(sc, zp);
}

__device__ __forceinline__ uint32_t u8_code(float x, float2 sz) {
  return static_cast<uint32_t>(fminf(fmaxf(rintf(__fadd_rn(__fdiv_rn(x, sz.x), sz.y)), 0.0f), 255.0f));
}

// fp8 e5m2 code of x: 1 sign, 5 exponent (bias 15), 2 mantissa bits. x is
// rounded once, to nearest with ties to even, at a quantum of 2 bits below
// its leading bit (never below the subnormal quantum 2^-16); magnitudes past
// the largest finite value 57344 saturate to it, NaN gives a NaN code. The
// rounded value is an IEEE half whose low byte is zero: its high byte is the
// code.
__device__ __forceinline__ uint32_t e5m2_code(double x) {
  uint32_t code = 0x7Fu;
  if (!isnan(x)) {
    const double ax = fabs(x);
    double r = 57344.0;
    if (ax < 57344.0) {
      const int e = ax > 0.0 ? ilogb(ax) : -14;
      const int qe = (e < -14 ? -14 : e) - 2;
      r = fmin(ldexp(rint(ldexp(ax, -qe)), qe), 57344.0);
    }
    code = static_cast<uint32_t>(__half_as_ushort(__double2half(r))) >> 8;
  }
  return code | (signbit(x) ? 0x80u : 0u);
}

}  // namespace mqa
