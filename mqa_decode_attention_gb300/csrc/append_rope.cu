// kv_append_rope kernel: RoPE on the new token's q and k, append of the rotated
// k and the v into the cache slot of position pos[b].
//
// Source: "KV Cache" explainer (lensaml.com), Langkah 3: each decode step
// writes one slice on the token axis of the [batch, kv_heads, tokens,
// head_dim] cache, and each key is rotated by its position once and stored
// rotated. Paged slot: "KV Cache 최적화 심층 분석" (youngju.dev), class
// PagedKVCache (block pos / block_size, row pos % block_size).
//
// Blocks cover (sequence, chunk of heads): first the query-head blocks (up to
// 8 heads each), then the kv-head blocks (2 heads each, so the fp64 key
// rotation is spread over many SMs). Every thread issues its global loads
// before the trigonometry so the two latencies overlap. Each block forms the
// d/2 angles pos * theta_i in fp64, reduces them to [-pi, pi] by Cody-Waite
// additive range reduction (2 pi split into three doubles, products folded in
// with fused multiply-adds) and takes their sine and cosine in fp64. The key
// is rotated in fp64 with explicit round-to-nearest products (no fused
// multiply-add), then rounded once to the cache dtype; the query is rotated
// in fp32 and written as fp32. bf16 and e5m2 caches keep the reduced angle
// and its fp32 cosine / sine instead: the key's rounding is decided from its
// fp32 rotation wherever an error bound settles it (the same bits as the
// fp64 path), the fp64 rotation taken only for the rest.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "../../include/mqa_decode.h"
#include "launch.h"
#include "ptx.cuh"
#include "quant.cuh"
#include "rope.cuh"

namespace mqa {
namespace {

// e5m2_code of a float, in float arithmetic: every step is exact for a float
// input (scalings by powers of two, one rint), so the code equals
// e5m2_code(double(x)) without fp64 work.
__device__ __forceinline__ uint32_t e5m2_code_f(float x) {
  uint32_t code = 0x7Fu;
  if (!isnan(x)) {
    const float ax = fabsf(x);
    float r = 57344.0f;
    if (ax < 57344.0f) {
      const int e = ax > 0.0f ? ilogbf(ax) : -14;
      const int qe = (e < -14 ? -14 : e) - 2;
      r = fminf(ldexpf(rintf(ldexpf(ax, -qe)), qe), 57344.0f);
    }
    code = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(r))) >> 8;
  }
  return code | (signbit(x) ? 0x80u : 0u);
}

// The key pair (x, y) turned by the reduced angle and rounded once to e5m2,
// decided in fp32 as rope_k_bf16_fast decides a bf16 rounding: the rotation
// from the fp32 cosine / sine cf, sf of the angle is within 8e-7 (|x| + |y|)
// of the fp64 rotation, and e5m2 rounding is monotonic, so when both ends of
// that interval (rounded outward) give one code the fp64 rotation gives it
// too. True with the codes in *codes (x in bits 0-7, y in 8-15); false
// leaves the pair to the fp64 rotation (e5m2_pair_fp64).
__device__ __forceinline__ bool rope_k_e5m2_fast(float x, float y, float cf, float sf, uint32_t* codes) {
  const float s = fabsf(x) + fabsf(y);
  if (!(s >= 0x1p-100f && s <= 1e37f)) return false;
  const float xr = fmaf(x, cf, -(y * sf));
  const float yr = fmaf(x, sf, y * cf);
  const float e = s * 8e-7f;
  const uint32_t xl = e5m2_code_f(__fsub_rd(xr, e)), xh = e5m2_code_f(__fadd_ru(xr, e));
  const uint32_t yl = e5m2_code_f(__fsub_rd(yr, e)), yh = e5m2_code_f(__fadd_ru(yr, e));
  if (xl != xh || yl != yh) return false;
  *codes = xl | (yl << 8);
  return true;
}

// The same pair from the fp64 rotation (fp64 sine and cosine of ang,
// round-to-nearest products and sum; the fused steps' append_row_q forms
// every pair this way), out of line: it runs only for the pairs whose fp32
// interval holds an e5m2 rounding boundary.
__device__ __noinline__ uint32_t e5m2_pair_fp64(float x, float y, double ang) {
  double c, sn;
  sincos(ang, &sn, &c);
  const double xd = x, yd = y;
  const double xr = __dsub_rn(__dmul_rn(xd, c), __dmul_rn(yd, sn));
  const double yr = __dadd_rn(__dmul_rn(xd, sn), __dmul_rn(yd, c));
  return e5m2_code(xr) | (e5m2_code(yr) << 8);
}

constexpr int kAppendThreads = 256;
constexpr int kQHeadsPerBlock = 8;   // 8 heads x 64 pairs = 2 pairs per thread at d = 128
constexpr int kKvHeadsPerBlock = 2;  // 2 heads x 64 pairs <= one pair per thread

template <typename T>
struct Elem;

template <>
struct Elem<__nv_bfloat16> {
  // two adjacent elements as fp32
  static __device__ __forceinline__ float2 load2(const __nv_bfloat16* p) {
    const uint32_t v = *reinterpret_cast<const uint32_t*>(p);
    return make_float2(bf16lo_to_f32(v), bf16hi_to_f32(v));
  }
  static __device__ __forceinline__ void store2_from_f64(__nv_bfloat16* p, double a, double b) {
    __nv_bfloat162 v;
    v.x = __double2bfloat16(a);
    v.y = __double2bfloat16(b);
    *reinterpret_cast<__nv_bfloat162*>(p) = v;
  }
  static __device__ __forceinline__ void copy2(__nv_bfloat16* dst, const __nv_bfloat16* src) {
    *reinterpret_cast<uint32_t*>(dst) = *reinterpret_cast<const uint32_t*>(src);
  }
};

template <>
struct Elem<float> {
  static __device__ __forceinline__ float2 load2(const float* p) { return *reinterpret_cast<const float2*>(p); }
  static __device__ __forceinline__ void store2_from_f64(float* p, double a, double b) {
    *reinterpret_cast<float2*>(p) = make_float2(__double2float_rn(a), __double2float_rn(b));
  }
  static __device__ __forceinline__ void copy2(float* dst, const float* src) {
    *reinterpret_cast<float2*>(dst) = *reinterpret_cast<const float2*>(src);
  }
};

template <typename T, bool QU8, bool F8 = false>
__global__ void __launch_bounds__(kAppendThreads) append_rope_kernel(const AppendParams p) {
  // bf16 and e5m2 caches: no fp64 sine / cosine table. q turns by the fp32
  // sine / cosine of the fp64-reduced angle (as the fused decode kernels form
  // q_rot) and k by rope_k_bf16 / rope_k_e5m2_fast (bit for bit the fp64
  // rotation rounded once); the fp32 and uint8 caches, whose stored values
  // depend on the exact fp32 rounding of the fp64 rotation, keep the fp64
  // table.
  constexpr bool kFast = std::is_same<T, __nv_bfloat16>::value && !QU8 && !F8;
  // the angle table (s_cos = the reduced angle, s_cf / s_sf its fp32 cosine /
  // sine): bf16 and e5m2 caches, whose keys take the fp32 stage first
  constexpr bool kAngle = kFast || F8;
  __shared__ double s_cos[kMaxHalfDim], s_sin[kMaxHalfDim];  // fp64 cos / sin; kFast: s_cos holds the angle
  __shared__ float s_cf[kMaxHalfDim], s_sf[kMaxHalfDim];    // kFast: fp32 cos / sin of the angle
  __shared__ float s_red[kAppendThreads / 32][4];  // uint8 cache: per-warp k/v min and max
  __shared__ long long s_row;     // element offset of the slot row of kv head 0
  __shared__ long long s_stride;  // element distance between kv heads at that slot
  __shared__ int s_ok;

  // Let a dependent decode launch start its prologue; it waits for this grid
  // before it reads q_rot or the appended slot.
  grid_dependents_launch();

  const int bt = blockIdx.x;  // (sequence, new token) = b * n_new + token
  const int b = bt / p.n_new;
  const int D = p.head_dim;
  const int half = D >> 1;
  const int n_qblocks = (p.h_q + kQHeadsPerBlock - 1) / kQHeadsPerBlock;
  const bool kv_block = static_cast<int>(blockIdx.y) >= n_qblocks;
  const int pos = p.pos[b] + (bt - b * p.n_new);

  // Issue this thread's loads first (at most 2 pairs per thread).
  int h_begin, h_end;
  if (!kv_block) {
    h_begin = blockIdx.y * kQHeadsPerBlock;
    h_end = min(h_begin + kQHeadsPerBlock, p.h_q);
  } else {
    h_begin = (blockIdx.y - n_qblocks) * kKvHeadsPerBlock;
    h_end = min(h_begin + kKvHeadsPerBlock, p.h_kv);
  }
  const int n_pairs = (h_end - h_begin) * half;
  const T* src = kv_block ? static_cast<const T*>(p.k_new) + static_cast<long long>(bt) * p.h_kv * D
                          : static_cast<const T*>(p.q_new) + static_cast<long long>(bt) * p.h_q * D;
  float2 x0 = make_float2(0.f, 0.f), x1 = make_float2(0.f, 0.f);
  const int i0 = threadIdx.x, i1 = threadIdx.x + kAppendThreads;
  if (i0 < n_pairs) x0 = Elem<T>::load2(src + (h_begin + i0 / half) * D + 2 * (i0 % half));
  if (i1 < n_pairs) x1 = Elem<T>::load2(src + (h_begin + i1 / half) * D + 2 * (i1 % half));

  if (threadIdx.x < half) {
    if constexpr (kAngle) {
      const double ang = reduce_two_pi(static_cast<double>(pos) * p.theta[threadIdx.x]);
      float sf, cf;
      sincosf(static_cast<float>(ang), &sf, &cf);
      s_cos[threadIdx.x] = ang;
      s_cf[threadIdx.x] = cf;
      s_sf[threadIdx.x] = sf;
    } else {
      double cs, sn;
      rope_cos_sin(pos, p.theta[threadIdx.x], &cs, &sn);
      s_cos[threadIdx.x] = cs;
      s_sin[threadIdx.x] = sn;
    }
  }
  if (threadIdx.x == 0 && kv_block) {
    int ok = 1;
    long long row = 0, stride = 0;
    const bool report = h_begin == 0;  // one block per sequence reports
    if (!p.paged) {
      if (pos < 0 || pos >= p.capacity) {
        ok = 0;
        if (report) atomicOr(p.err, static_cast<int>(MQA_DEVERR_POS_RANGE));
      } else {
        row = (static_cast<long long>(b) * p.h_kv * p.capacity + pos) * D;
        stride = p.capacity * D;
      }
    } else {
      const int lp = pos >= 0 ? pos / p.page_size : -1;
      if (pos < 0 || lp >= p.max_pages) {
        ok = 0;
        if (report) atomicOr(p.err, static_cast<int>(MQA_DEVERR_POS_RANGE));
      } else {
        const int page = p.block_table[static_cast<long long>(b) * p.max_pages + lp];
        if (page < 0 || page >= p.num_pages) {
          ok = 0;
          if (report) atomicOr(p.err, static_cast<int>(MQA_DEVERR_PAGE_RANGE));
        } else {
          row = (static_cast<long long>(page) * p.h_kv * p.page_size + (pos % p.page_size)) * D;
          stride = static_cast<long long>(p.page_size) * D;
        }
      }
    }
    s_ok = ok;
    s_row = row;
    s_stride = stride;
  }
  __syncthreads();

  if (!kv_block) {
    // q: fp32 rotation, fp32 output
    float* qr = p.q_rot + static_cast<long long>(bt) * p.h_q * D;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int idx = u == 0 ? i0 : i1;
      if (idx >= n_pairs) continue;
      const float2 x = u == 0 ? x0 : x1;
      const int h = h_begin + idx / half, i = idx % half;
      const float c = kAngle ? s_cf[i] : static_cast<float>(s_cos[i]);
      const float s = kAngle ? s_sf[i] : static_cast<float>(s_sin[i]);
      *reinterpret_cast<float2*>(qr + h * D + 2 * i) = make_float2(x.x * c - x.y * s, x.x * s + x.y * c);
    }
    return;
  }
  if (!s_ok) return;

  if constexpr (QU8) {
    // k: fp64 rotation rounded to fp32, then both rows quantised; one pair per thread
    const T* v = static_cast<const T*>(p.v_new) + static_cast<long long>(bt) * p.h_kv * D;
    const bool act = i0 < n_pairs;
    const int hl = act ? i0 / half : 0, i = i0 % half;
    float kx = 0.f, ky = 0.f, vx = 0.f, vy = 0.f;
    if (act) {
      const double xd = x0.x, yd = x0.y, c = s_cos[i], s = s_sin[i];
      kx = __double2float_rn(__dsub_rn(__dmul_rn(xd, c), __dmul_rn(yd, s)));
      ky = __double2float_rn(__dadd_rn(__dmul_rn(xd, s), __dmul_rn(yd, c)));
      const float2 vv = Elem<T>::load2(v + (h_begin + hl) * D + 2 * i);
      vx = vv.x;
      vy = vv.y;
    }
    float r[4] = {act ? fminf(kx, ky) : INFINITY, act ? fmaxf(kx, ky) : -INFINITY,
                  act ? fminf(vx, vy) : INFINITY, act ? fmaxf(vx, vy) : -INFINITY};
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {  // a warp never spans two heads (half is 32 or 64)
      r[0] = fminf(r[0], __shfl_xor_sync(0xffffffffu, r[0], off));
      r[1] = fmaxf(r[1], __shfl_xor_sync(0xffffffffu, r[1], off));
      r[2] = fminf(r[2], __shfl_xor_sync(0xffffffffu, r[2], off));
      r[3] = fmaxf(r[3], __shfl_xor_sync(0xffffffffu, r[3], off));
    }
    if ((threadIdx.x & 31) == 0) {
      s_red[threadIdx.x >> 5][0] = r[0];
      s_red[threadIdx.x >> 5][1] = r[1];
      s_red[threadIdx.x >> 5][2] = r[2];
      s_red[threadIdx.x >> 5][3] = r[3];
    }
    __syncthreads();
    if (!act) return;
    float kmn = INFINITY, kmx = -INFINITY, vmn = INFINITY, vmx = -INFINITY;
    for (int w = hl * half / 32; w < (hl + 1) * half / 32; ++w) {
      kmn = fminf(kmn, s_red[w][0]);
      kmx = fmaxf(kmx, s_red[w][1]);
      vmn = fminf(vmn, s_red[w][2]);
      vmx = fmaxf(vmx, s_red[w][3]);
    }
    const float2 ksz = u8_params(kmn, kmx), vsz = u8_params(vmn, vmx);
    const long long row = s_row + static_cast<long long>(h_begin + hl) * s_stride;  // element offset of the row
    uint8_t* kc = static_cast<uint8_t*>(p.k_cache) + row;
    uint8_t* vc = static_cast<uint8_t*>(p.v_cache) + row;
    *reinterpret_cast<uint16_t*>(kc + 2 * i) = static_cast<uint16_t>(u8_code(kx, ksz) | (u8_code(ky, ksz) << 8));
    *reinterpret_cast<uint16_t*>(vc + 2 * i) = static_cast<uint16_t>(u8_code(vx, vsz) | (u8_code(vy, vsz) << 8));
    if (i == 0) {
      p.k_sz[row / D] = ksz;
      p.v_sz[row / D] = vsz;
    }
    return;
  }

  if constexpr (F8) {
    // e5m2 cache: k from its rotation (rope_k_e5m2_fast, else the fp64 one)
    // and v from its bf16 value, each rounded once to e5m2
    const T* v = static_cast<const T*>(p.v_new) + static_cast<long long>(bt) * p.h_kv * D;
    uint8_t* kc = static_cast<uint8_t*>(p.k_cache) + s_row;
    uint8_t* vc = static_cast<uint8_t*>(p.v_cache) + s_row;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int idx = u == 0 ? i0 : i1;
      if (idx >= n_pairs) continue;
      const float2 x = u == 0 ? x0 : x1;
      const int h = h_begin + idx / half, i = idx % half;
      uint32_t kk;
      if (!rope_k_e5m2_fast(x.x, x.y, s_cf[i], s_sf[i], &kk)) kk = e5m2_pair_fp64(x.x, x.y, s_cos[i]);
      const float2 vv = Elem<T>::load2(v + h * D + 2 * i);
      *reinterpret_cast<uint16_t*>(kc + h * s_stride + 2 * i) = static_cast<uint16_t>(kk);
      *reinterpret_cast<uint16_t*>(vc + h * s_stride + 2 * i) =
          static_cast<uint16_t>(e5m2_code_f(vv.x) | (e5m2_code_f(vv.y) << 8));
    }
    return;
  }

  // k: fp64 rotation, one rounding to the cache dtype; v: bit copy
  const T* v = static_cast<const T*>(p.v_new) + static_cast<long long>(bt) * p.h_kv * D;
  T* kc = static_cast<T*>(p.k_cache) + s_row;
  T* vc = static_cast<T*>(p.v_cache) + s_row;
  const long long stride = s_stride;
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int idx = u == 0 ? i0 : i1;
    if (idx >= n_pairs) continue;
    const float2 x = u == 0 ? x0 : x1;
    const int h = h_begin + idx / half, i = idx % half;
    if constexpr (kFast) {
      *reinterpret_cast<__nv_bfloat162*>(kc + h * stride + 2 * i) = rope_k_bf16(x.x, x.y, s_cos[i]);
    } else {
      const double xd = x.x, yd = x.y, c = s_cos[i], s = s_sin[i];
      const double xr = __dsub_rn(__dmul_rn(xd, c), __dmul_rn(yd, s));
      const double yr = __dadd_rn(__dmul_rn(xd, s), __dmul_rn(yd, c));
      Elem<T>::store2_from_f64(kc + h * stride + 2 * i, xr, yr);
    }
    Elem<T>::copy2(vc + h * stride + 2 * i, v + h * D + 2 * i);
  }
}

// Many new tokens per sequence (prefill): one block per (sequence, token)
// that forms the token's d/2 fp64 sines and cosines once and rotates every
// query and kv head of it, with the arithmetic of append_rope_kernel (the
// per-head-block grid would evaluate the same fp64 table once per head block).
// BYTE: a uint8 (1) or e5m2 (2) cache: one warp per kv head row rotates k in
// fp64 and quantises the row as append_rope_kernel does (uint8: the row's
// minimum and maximum over a warp reduction, the same set of values, so the
// same scale and zero point).
template <typename T, int BYTE = 0>
__global__ void __launch_bounds__(kAppendThreads) append_rope_tokens_kernel(const AppendParams p) {
  constexpr bool kFast = std::is_same<T, __nv_bfloat16>::value && BYTE == 0;  // as in append_rope_kernel
  constexpr bool kAngle = kFast || BYTE == 2;
  __shared__ double s_cos[kMaxHalfDim], s_sin[kMaxHalfDim];  // fp64 cos / sin; kFast: s_cos holds the angle
  __shared__ float s_cf[kMaxHalfDim], s_sf[kMaxHalfDim];    // kFast: fp32 cos / sin of the angle
  __shared__ long long s_row, s_stride;
  __shared__ int s_ok;
  grid_dependents_launch();
  const int bt = blockIdx.x;
  const int b = bt / p.n_new;
  const int D = p.head_dim, half = D >> 1;
  const int pos = p.pos[b] + (bt - b * p.n_new);
  // bf16 q rows: 16-byte units of four rotation pairs; a thread's first two
  // units are requested before the table is formed, so that their latency
  // and the table's overlap
  constexpr bool kVec = std::is_same<T, __nv_bfloat16>::value;
  const int n_units = kVec ? p.h_q * D / 8 : 0;
  const uint4* qsrc = reinterpret_cast<const uint4*>(static_cast<const T*>(p.q_new) + static_cast<long long>(bt) * p.h_q * D);
  uint4 qpre0 = make_uint4(0u, 0u, 0u, 0u), qpre1 = make_uint4(0u, 0u, 0u, 0u);
  if (kVec && static_cast<int>(threadIdx.x) < n_units) qpre0 = qsrc[threadIdx.x];
  if (kVec && static_cast<int>(threadIdx.x) + kAppendThreads < n_units) qpre1 = qsrc[threadIdx.x + kAppendThreads];
  if (threadIdx.x < half) {
    if constexpr (kAngle) {
      const double ang = reduce_two_pi(static_cast<double>(pos) * p.theta[threadIdx.x]);
      float sf, cf;
      sincosf(static_cast<float>(ang), &sf, &cf);
      s_cos[threadIdx.x] = ang;
      s_cf[threadIdx.x] = cf;
      s_sf[threadIdx.x] = sf;
    } else {
      double cs, sn;
      rope_cos_sin(pos, p.theta[threadIdx.x], &cs, &sn);
      s_cos[threadIdx.x] = cs;
      s_sin[threadIdx.x] = sn;
    }
  }
  if (threadIdx.x == 0) {
    int ok = 1;
    long long row = 0, stride = 0;
    if (!p.paged) {
      if (pos < 0 || pos >= p.capacity) {
        ok = 0;
        atomicOr(p.err, static_cast<int>(MQA_DEVERR_POS_RANGE));
      } else {
        row = (static_cast<long long>(b) * p.h_kv * p.capacity + pos) * D;
        stride = p.capacity * D;
      }
    } else {
      const int lp = pos >= 0 ? pos / p.page_size : -1;
      if (pos < 0 || lp >= p.max_pages) {
        ok = 0;
        atomicOr(p.err, static_cast<int>(MQA_DEVERR_POS_RANGE));
      } else {
        const int page = p.block_table[static_cast<long long>(b) * p.max_pages + lp];
        if (page < 0 || page >= p.num_pages) {
          ok = 0;
          atomicOr(p.err, static_cast<int>(MQA_DEVERR_PAGE_RANGE));
        } else {
          row = (static_cast<long long>(page) * p.h_kv * p.page_size + (pos % p.page_size)) * D;
          stride = static_cast<long long>(p.page_size) * D;
        }
      }
    }
    s_ok = ok;
    s_row = row;
    s_stride = stride;
  }
  __syncthreads();
  // q: fp32 rotation, fp32 output
  const T* qs = static_cast<const T*>(p.q_new) + static_cast<long long>(bt) * p.h_q * D;
  float* qr = p.q_rot + static_cast<long long>(bt) * p.h_q * D;
  if constexpr (kVec) {
    auto rot_unit = [&](int w, uint4 raw) {  // elements 8 w .. 8 w + 7 (one head: D % 8 == 0)
      const int e0 = 8 * w, i0 = (e0 % D) >> 1;
      const uint32_t wd[4] = {raw.x, raw.y, raw.z, raw.w};
      float o[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float x = bf16lo_to_f32(wd[k]), y = bf16hi_to_f32(wd[k]);
        const float c = kAngle ? s_cf[i0 + k] : static_cast<float>(s_cos[i0 + k]);
        const float s = kAngle ? s_sf[i0 + k] : static_cast<float>(s_sin[i0 + k]);
        o[2 * k] = x * c - y * s;
        o[2 * k + 1] = x * s + y * c;
      }
      *reinterpret_cast<float4*>(qr + e0) = make_float4(o[0], o[1], o[2], o[3]);
      *reinterpret_cast<float4*>(qr + e0 + 4) = make_float4(o[4], o[5], o[6], o[7]);
    };
    if (static_cast<int>(threadIdx.x) < n_units) rot_unit(threadIdx.x, qpre0);
    if (static_cast<int>(threadIdx.x) + kAppendThreads < n_units) rot_unit(threadIdx.x + kAppendThreads, qpre1);
    for (int w = threadIdx.x + 2 * kAppendThreads; w < n_units; w += kAppendThreads) rot_unit(w, qsrc[w]);
  } else {
    for (int idx = threadIdx.x; idx < p.h_q * half; idx += kAppendThreads) {
      const int h = idx / half, i = idx - h * half;
      const float2 x = Elem<T>::load2(qs + h * D + 2 * i);
      const float c = kAngle ? s_cf[i] : static_cast<float>(s_cos[i]);
      const float s = kAngle ? s_sf[i] : static_cast<float>(s_sin[i]);
      *reinterpret_cast<float2*>(qr + h * D + 2 * i) = make_float2(x.x * c - x.y * s, x.x * s + x.y * c);
    }
  }
  if (!s_ok) return;
  const T* ks = static_cast<const T*>(p.k_new) + static_cast<long long>(bt) * p.h_kv * D;
  const T* vs = static_cast<const T*>(p.v_new) + static_cast<long long>(bt) * p.h_kv * D;
  if constexpr (BYTE != 0) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int h = warp; h < p.h_kv; h += kAppendThreads / 32) {
      const long long row = s_row + static_cast<long long>(h) * s_stride;  // element (byte) offset of the row
      uint8_t* kc = static_cast<uint8_t*>(p.k_cache) + row;
      uint8_t* vc = static_cast<uint8_t*>(p.v_cache) + row;
      float kmn = INFINITY, kmx = -INFINITY, vmn = INFINITY, vmx = -INFINITY;
      double xr[2], yr[2];
      float2 vv[2];
      for (int u = 0; u < 2; ++u) {
        const int i = lane + 32 * u;
        if (i >= half) break;
        const float2 x = Elem<T>::load2(ks + h * D + 2 * i);
        vv[u] = Elem<T>::load2(vs + h * D + 2 * i);
        if constexpr (BYTE == 2) {
          uint32_t kk;
          if (!rope_k_e5m2_fast(x.x, x.y, s_cf[i], s_sf[i], &kk)) kk = e5m2_pair_fp64(x.x, x.y, s_cos[i]);
          *reinterpret_cast<uint16_t*>(kc + 2 * i) = static_cast<uint16_t>(kk);
          *reinterpret_cast<uint16_t*>(vc + 2 * i) =
              static_cast<uint16_t>(e5m2_code_f(vv[u].x) | (e5m2_code_f(vv[u].y) << 8));
        } else {
          const double xd = x.x, yd = x.y, c = s_cos[i], sn = s_sin[i];
          xr[u] = __dsub_rn(__dmul_rn(xd, c), __dmul_rn(yd, sn));
          yr[u] = __dadd_rn(__dmul_rn(xd, sn), __dmul_rn(yd, c));
          const float kx = __double2float_rn(xr[u]), ky = __double2float_rn(yr[u]);
          kmn = fminf(kmn, fminf(kx, ky));
          kmx = fmaxf(kmx, fmaxf(kx, ky));
          vmn = fminf(vmn, fminf(vv[u].x, vv[u].y));
          vmx = fmaxf(vmx, fmaxf(vv[u].x, vv[u].y));
        }
      }
      if constexpr (BYTE == 1) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          kmn = fminf(kmn, __shfl_xor_sync(0xffffffffu, kmn, off));
          kmx = fmaxf(kmx, __shfl_xor_sync(0xffffffffu, kmx, off));
          vmn = fminf(vmn, __shfl_xor_sync(0xffffffffu, vmn, off));
          vmx = fmaxf(vmx, __shfl_xor_sync(0xffffffffu, vmx, off));
        }
        const float2 ksz = u8_params(kmn, kmx), vsz = u8_params(vmn, vmx);
        for (int u = 0; u < 2; ++u) {
          const int i = lane + 32 * u;
          if (i >= half) break;
          const float kx = __double2float_rn(xr[u]), ky = __double2float_rn(yr[u]);
          *reinterpret_cast<uint16_t*>(kc + 2 * i) = static_cast<uint16_t>(u8_code(kx, ksz) | (u8_code(ky, ksz) << 8));
          *reinterpret_cast<uint16_t*>(vc + 2 * i) =
              static_cast<uint16_t>(u8_code(vv[u].x, vsz) | (u8_code(vv[u].y, vsz) << 8));
        }
        if (lane == 0) {
          p.k_sz[row / D] = ksz;
          p.v_sz[row / D] = vsz;
        }
      }
    }
    return;
  }
  // k: fp64 rotation, one rounding to the cache dtype; v: bit copy
  T* kc = static_cast<T*>(p.k_cache) + s_row;
  T* vc = static_cast<T*>(p.v_cache) + s_row;
  for (int idx = threadIdx.x; idx < p.h_kv * half; idx += kAppendThreads) {
    const int h = idx / half, i = idx - h * half;
    const float2 x = Elem<T>::load2(ks + h * D + 2 * i);
    if constexpr (kFast) {
      *reinterpret_cast<__nv_bfloat162*>(kc + h * s_stride + 2 * i) = rope_k_bf16(x.x, x.y, s_cos[i]);
    } else {
      const double xd = x.x, yd = x.y, c = s_cos[i], s = s_sin[i];
      const double xr = __dsub_rn(__dmul_rn(xd, c), __dmul_rn(yd, s));
      const double yr = __dadd_rn(__dmul_rn(xd, s), __dmul_rn(yd, c));
      Elem<T>::store2_from_f64(kc + h * s_stride + 2 * i, xr, yr);
    }
    Elem<T>::copy2(vc + h * s_stride + 2 * i, vs + h * D + 2 * i);
  }
}

}  // namespace

KernelShape append_rope_shape() { return {kAppendThreads, 0, 0, 0}; }

cudaError_t launch_append_rope(const AppendParams& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  if (static_cast<long long>(p.batch) * p.n_new >= 256) {
    // one block per token forms its fp64 table once for all heads: from a few
    // hundred tokens the per-head-block tables' fp64 work costs more than the
    // parallelism they buy (measured, gqa4k shapes: 256 tokens 21.6 -> 17.3 µs;
    // at 64 and 128 tokens the per-head-block grid stays faster; one-byte
    // caches, whose tables are fp64 sines and cosines: 8 x 4096 tokens e5m2
    // 3.3 ms on the per-head-block grid)
    cfg.gridDim = dim3(p.batch * p.n_new);
    cfg.blockDim = dim3(kAppendThreads);
    cfg.stream = stream;
    if (p.cache_dtype == kDtypeU8) return cudaLaunchKernelEx(&cfg, append_rope_tokens_kernel<__nv_bfloat16, 1>, p);
    if (p.cache_dtype == kDtypeF8) return cudaLaunchKernelEx(&cfg, append_rope_tokens_kernel<__nv_bfloat16, 2>, p);
    if (p.cache_dtype == kDtypeBf16) return cudaLaunchKernelEx(&cfg, append_rope_tokens_kernel<__nv_bfloat16>, p);
    return cudaLaunchKernelEx(&cfg, append_rope_tokens_kernel<float>, p);
  }
  cfg.gridDim = dim3(p.batch * p.n_new, (p.h_q + kQHeadsPerBlock - 1) / kQHeadsPerBlock +
                                  (p.h_kv + kKvHeadsPerBlock - 1) / kKvHeadsPerBlock);
  cfg.blockDim = dim3(kAppendThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  if (p.cache_dtype == kDtypeU8) return cudaLaunchKernelEx(&cfg, append_rope_kernel<__nv_bfloat16, true>, p);
  if (p.cache_dtype == kDtypeF8) return cudaLaunchKernelEx(&cfg, append_rope_kernel<__nv_bfloat16, false, true>, p);
  if (p.cache_dtype == kDtypeBf16) return cudaLaunchKernelEx(&cfg, append_rope_kernel<__nv_bfloat16, false>, p);
  return cudaLaunchKernelEx(&cfg, append_rope_kernel<float, false>, p);
}

}  // namespace mqa
