// splitkv_combine kernel: log-sum-exp merge of per-split results.
//
// Split s of row (b, h) holds the normalised output O_s over its token range
// and lse_s = log sum exp(score) over that range. With M = max_s lse_s,
//   LSE = M + log sum_s exp(lse_s - M),  O = sum_s exp(lse_s - M) O_s / sum_s exp(lse_s - M).
// A split with no tokens has lse_s = -inf and weight 0.
//
// One warp per (b, h) row, eight rows per block; lane l holds head dims
// (D / 32) l .. + D / 32 and walks the splits in order with vector loads of
// O_s (the same order of the sum as one thread per element).
#include <cuda_bf16.h>

#include "launch.h"

namespace mqa {
namespace {

constexpr int kRowsPerBlock = 8;
constexpr int kUnroll = 8;  // splits whose loads are issued together

template <int V>  // head dims per lane: 4 (d = 128) or 2 (d = 64)
__global__ void __launch_bounds__(32 * kRowsPerBlock) combine_kernel(const CombineParams p) {
  // The next launch (the next step) may be scheduled now: it waits for this
  // whole grid before it touches anything. Then wait for the decode grid that
  // wrote the partials (both no-ops without programmatic dependent launch).
  asm volatile("griddepcontrol.launch_dependents;");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kRowsPerBlock + warp;
  if (row >= p.rows) return;
  const int S = p.num_splits, D = p.head_dim;
  const float* lse = p.lse_part + static_cast<long long>(row) * S;
  const float* o = p.o_part + static_cast<long long>(row) * S * D + V * lane;

  float m = -INFINITY;
  for (int s = lane; s < S; s += 32) m = fmaxf(m, lse[s]);
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, w));

  float wsum = 0.f, acc[V];
#pragma unroll
  for (int v = 0; v < V; ++v) acc[v] = 0.f;
  if (m != -INFINITY) {
    // batches of kUnroll splits: their loads all in flight before the sums
    for (int s0 = 0; s0 < S; s0 += kUnroll) {
      float lv[kUnroll], ov[kUnroll][V];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        lv[u] = -INFINITY;
#pragma unroll
        for (int v = 0; v < V; ++v) ov[u][v] = 0.f;
        if (s0 + u < S) {
          lv[u] = lse[s0 + u];
          const float* src = o + static_cast<long long>(s0 + u) * D;
          if constexpr (V == 4) {
            const float4 t = *reinterpret_cast<const float4*>(src);
            ov[u][0] = t.x, ov[u][1] = t.y, ov[u][2] = t.z, ov[u][3] = t.w;
          } else {
            const float2 t = *reinterpret_cast<const float2*>(src);
            ov[u][0] = t.x, ov[u][1] = t.y;
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        if (s0 + u < S) {
          const float w = expf(lv[u] - m);  // exp(-inf) = 0 for empty splits
          wsum += w;
#pragma unroll
          for (int v = 0; v < V; ++v) acc[v] = fmaf(w, ov[u][v], acc[v]);
        }
      }
    }
  }
  const long long idx = static_cast<long long>(row) * D + V * lane;
  float val[V];
#pragma unroll
  for (int v = 0; v < V; ++v) val[v] = wsum > 0.f ? acc[v] / wsum : 0.f;
  if (p.out_dtype == kDtypeBf16) {
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + idx;
#pragma unroll
    for (int v = 0; v < V; v += 2) *reinterpret_cast<__nv_bfloat162*>(dst + v) = __floats2bfloat162_rn(val[v], val[v + 1]);
  } else {
    float* dst = static_cast<float*>(p.out) + idx;
#pragma unroll
    for (int v = 0; v < V; ++v) dst[v] = val[v];
  }
  if (lane == 0 && p.lse_out != nullptr) p.lse_out[row] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
}

}  // namespace

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((p.rows + kRowsPerBlock - 1) / kRowsPerBlock);
  cfg.blockDim = dim3(32 * kRowsPerBlock);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  // resident while the decode grid finishes; griddepcontrol.wait holds it
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return p.head_dim == 128 ? cudaLaunchKernelEx(&cfg, combine_kernel<4>, p) : cudaLaunchKernelEx(&cfg, combine_kernel<2>, p);
}

}  // namespace mqa
