// kv_append_rope kernel: RoPE on the new token's q and k, append of the rotated
// k and the v into the cache slot of position pos[b].
//
// Source: "KV Cache" explainer (lensaml.com), Langkah 3: each decode step
// writes one slice on the token axis of the [batch, kv_heads, tokens,
// head_dim] cache, and each key is rotated by its position once and stored
// rotated. Paged slot: "KV Cache 최적화 심층 분석" (youngju.dev), class
// PagedKVCache (block pos / block_size, row pos % block_size).
//
// One block per sequence. The d/2 angles pos * theta_i are formed and their
// sine and cosine taken in fp64 once per sequence, shared by all heads. The
// key is rotated in fp64 with explicit round-to-nearest products (no fused
// multiply-add), then rounded once to the cache dtype; the query is rotated
// in fp32 and written as fp32.
#include <cuda_bf16.h>

#include "../../include/mqa_decode.h"
#include "launch.h"
#include "ptx.cuh"

namespace mqa {
namespace {

constexpr int kAppendThreads = 256;

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

template <typename T>
__global__ void __launch_bounds__(kAppendThreads) append_rope_kernel(const AppendParams p) {
  __shared__ double s_cos[kMaxHalfDim], s_sin[kMaxHalfDim];
  __shared__ long long s_row;     // element offset of the slot row of kv head 0
  __shared__ long long s_stride;  // element distance between kv heads at that slot
  __shared__ int s_ok;

  // Let a dependent decode launch start its prologue; it waits for this grid
  // before it reads q_rot or the cache.
  grid_dependents_launch();

  const int b = blockIdx.x;
  const int D = p.head_dim;
  const int half = D >> 1;
  const int pos = p.pos[b];

  if (threadIdx.x < half) {
    double sn, cs;
    sincos(static_cast<double>(pos) * p.theta[threadIdx.x], &sn, &cs);
    s_cos[threadIdx.x] = cs;
    s_sin[threadIdx.x] = sn;
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
  const T* q = static_cast<const T*>(p.q_new) + static_cast<long long>(b) * p.h_q * D;
  float* qr = p.q_rot + static_cast<long long>(b) * p.h_q * D;
  for (int idx = threadIdx.x; idx < p.h_q * half; idx += kAppendThreads) {
    const int h = idx / half, i = idx - h * half;
    const float2 x = Elem<T>::load2(q + h * D + 2 * i);
    const float c = static_cast<float>(s_cos[i]), s = static_cast<float>(s_sin[i]);
    *reinterpret_cast<float2*>(qr + h * D + 2 * i) = make_float2(x.x * c - x.y * s, x.x * s + x.y * c);
  }
  if (!s_ok) return;

  // k: fp64 rotation, one rounding to the cache dtype; v: bit copy
  const T* k = static_cast<const T*>(p.k_new) + static_cast<long long>(b) * p.h_kv * D;
  const T* v = static_cast<const T*>(p.v_new) + static_cast<long long>(b) * p.h_kv * D;
  T* kc = static_cast<T*>(p.k_cache) + s_row;
  T* vc = static_cast<T*>(p.v_cache) + s_row;
  const long long stride = s_stride;
  for (int idx = threadIdx.x; idx < p.h_kv * half; idx += kAppendThreads) {
    const int h = idx / half, i = idx - h * half;
    const float2 x = Elem<T>::load2(k + h * D + 2 * i);
    const double xd = x.x, yd = x.y, c = s_cos[i], s = s_sin[i];
    const double xr = __dsub_rn(__dmul_rn(xd, c), __dmul_rn(yd, s));
    const double yr = __dadd_rn(__dmul_rn(xd, s), __dmul_rn(yd, c));
    Elem<T>::store2_from_f64(kc + h * stride + 2 * i, xr, yr);
    Elem<T>::copy2(vc + h * stride + 2 * i, v + h * D + 2 * i);
  }
}

}  // namespace

KernelShape append_rope_shape() { return {kAppendThreads, 0, 0}; }

cudaError_t launch_append_rope(const AppendParams& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.batch);
  cfg.blockDim = dim3(kAppendThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  if (p.cache_dtype == kDtypeBf16) return cudaLaunchKernelEx(&cfg, append_rope_kernel<__nv_bfloat16>, p);
  return cudaLaunchKernelEx(&cfg, append_rope_kernel<float>, p);
}

}  // namespace mqa
