// Byte-cache encoders shared by the append kernel and the decode kernels
// that perform the append themselves (fused step): both write the same bytes.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "rope.cuh"

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

// The fused append of a one-byte cache: sequence b's new token at `pos`, kv
// head j, element offset `row` of its cache row (negative: nothing is
// written), by one whole warp (lane i owns rotation pairs i, i + 32, ...),
// with the append kernel's bytes: k turned in fp64 by the fp64 sine and cosine
// of the reduced angle (round-to-nearest products); uint8: k rounded to fp32
// and v taken as fp32, each row quantised with its own (scale, zero point)
// from its minimum and maximum; e5m2: k (fp64) and v each rounded once to
// e5m2. The rows are then fenced for TMA loads (async proxy) that follow the
// warp's arrival on a barrier. P: the kernel's parameters (theta, k_new,
// v_new [B, H_kv, D] bf16, h_kv, k_cache, v_cache, k_sz, v_sz).
template <int D, bool F8, class P>
__device__ __forceinline__ void append_row_q(const P& p, int b, int j, int pos, long long row, int lane) {
  constexpr int kPer = D / 64;  // rotation pairs per lane
  if (row >= 0) {  // the same for every lane
    uint32_t k[kPer], v[kPer];
    double theta[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      theta[i] = p.theta[lane + 32 * i];
      const long long src = (static_cast<long long>(b) * p.h_kv + j) * D + 2 * (lane + 32 * i);
      k[i] = *reinterpret_cast<const uint32_t*>(static_cast<const __nv_bfloat16*>(p.k_new) + src);
      v[i] = *reinterpret_cast<const uint32_t*>(static_cast<const __nv_bfloat16*>(p.v_new) + src);
    }
    double xr[kPer], yr[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      double c, sn;
      sincos(reduce_two_pi(static_cast<double>(pos) * theta[i]), &sn, &c);
      const double x = bf16lo_to_f32(k[i]), y = bf16hi_to_f32(k[i]);
      xr[i] = __dsub_rn(__dmul_rn(x, c), __dmul_rn(y, sn));
      yr[i] = __dadd_rn(__dmul_rn(x, sn), __dmul_rn(y, c));
    }
    uint8_t* kc = static_cast<uint8_t*>(const_cast<void*>(p.k_cache)) + row;
    uint8_t* vc = static_cast<uint8_t*>(const_cast<void*>(p.v_cache)) + row;
    if constexpr (F8) {
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int t = lane + 32 * i;
        *reinterpret_cast<uint16_t*>(kc + 2 * t) = static_cast<uint16_t>(e5m2_code(xr[i]) | (e5m2_code(yr[i]) << 8));
        *reinterpret_cast<uint16_t*>(vc + 2 * t) =
            static_cast<uint16_t>(e5m2_code(bf16lo_to_f32(v[i])) | (e5m2_code(bf16hi_to_f32(v[i])) << 8));
      }
    } else {
      float kx[kPer], ky[kPer], vx[kPer], vy[kPer];
      float kmn = INFINITY, kmx = -INFINITY, vmn = INFINITY, vmx = -INFINITY;
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        kx[i] = __double2float_rn(xr[i]);
        ky[i] = __double2float_rn(yr[i]);
        vx[i] = bf16lo_to_f32(v[i]);
        vy[i] = bf16hi_to_f32(v[i]);
        kmn = fminf(kmn, fminf(kx[i], ky[i]));
        kmx = fmaxf(kmx, fmaxf(kx[i], ky[i]));
        vmn = fminf(vmn, fminf(vx[i], vy[i]));
        vmx = fmaxf(vmx, fmaxf(vx[i], vy[i]));
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        kmn = fminf(kmn, __shfl_xor_sync(0xffffffffu, kmn, off));
        kmx = fmaxf(kmx, __shfl_xor_sync(0xffffffffu, kmx, off));
        vmn = fminf(vmn, __shfl_xor_sync(0xffffffffu, vmn, off));
        vmx = fmaxf(vmx, __shfl_xor_sync(0xffffffffu, vmx, off));
      }
      const float2 ksz = u8_params(kmn, kmx), vsz = u8_params(vmn, vmx);
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int t = lane + 32 * i;
        *reinterpret_cast<uint16_t*>(kc + 2 * t) =
            static_cast<uint16_t>(u8_code(kx[i], ksz) | (u8_code(ky[i], ksz) << 8));
        *reinterpret_cast<uint16_t*>(vc + 2 * t) =
            static_cast<uint16_t>(u8_code(vx[i], vsz) | (u8_code(vy[i], vsz) << 8));
      }
      if (lane == 0) {
        const_cast<float2*>(p.k_sz)[row / D] = ksz;
        const_cast<float2*>(p.v_sz)[row / D] = vsz;
      }
    }
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  __syncwarp();
}

}  // namespace mqa
