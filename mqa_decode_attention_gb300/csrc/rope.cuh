// RoPE angle helpers shared by the append kernel and the decode kernels.
#pragma once

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

}  // namespace mqa
