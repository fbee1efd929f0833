// splitkv_combine kernel: log-sum-exp merge of per-split results.
//
// Split s of row (b, h) holds the normalised output O_s over its token range
// and lse_s = log sum exp(score) over that range. With M = max_s lse_s,
//   LSE = M + log sum_s exp(lse_s - M),  O = sum_s exp(lse_s - M) O_s / sum_s exp(lse_s - M).
// A split with no tokens has lse_s = -inf and weight 0.
//
// One block per (b, h) row, one thread per output element; each thread walks
// the splits with independent, coalesced loads of O_s[d].
#include <cuda_bf16.h>

#include "launch.h"

namespace mqa {
namespace {

constexpr int kCombineUnroll = 8;

__global__ void __launch_bounds__(128) combine_kernel(const CombineParams p) {
  // Wait for the decode grid that wrote the partials (no-op without PDL).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int row = blockIdx.x;
  const int S = p.num_splits;
  const float* lse = p.lse_part + static_cast<long long>(row) * S;
  const float* o = p.o_part + static_cast<long long>(row) * S * p.head_dim;

  float m = -INFINITY;
  for (int s = 0; s < S; ++s) m = fmaxf(m, lse[s]);

  for (int d = threadIdx.x; d < p.head_dim; d += blockDim.x) {
    float wsum = 0.f, acc = 0.f;
    if (m != -INFINITY) {
      int s = 0;
      for (; s + kCombineUnroll <= S; s += kCombineUnroll) {
        float ov[kCombineUnroll], lv[kCombineUnroll];
#pragma unroll
        for (int u = 0; u < kCombineUnroll; ++u) {
          lv[u] = lse[s + u];
          ov[u] = o[static_cast<long long>(s + u) * p.head_dim + d];
        }
#pragma unroll
        for (int u = 0; u < kCombineUnroll; ++u) {
          const float w = expf(lv[u] - m);  // exp(-inf) = 0 for empty splits
          wsum += w;
          acc = fmaf(w, ov[u], acc);
        }
      }
      for (; s < S; ++s) {
        const float w = expf(lse[s] - m);
        wsum += w;
        acc = fmaf(w, o[static_cast<long long>(s) * p.head_dim + d], acc);
      }
    }
    const float val = wsum > 0.f ? acc / wsum : 0.f;
    const long long idx = static_cast<long long>(row) * p.head_dim + d;
    if (p.out_dtype == kDtypeBf16)
      static_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16_rn(val);
    else
      static_cast<float*>(p.out)[idx] = val;
    if (d == 0 && p.lse_out != nullptr) p.lse_out[row] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
  }
}

}  // namespace

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.rows);
  cfg.blockDim = dim3(p.head_dim >= 128 ? 128 : 64);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  // resident while the decode grid finishes; griddepcontrol.wait holds it
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel, p);
}

}  // namespace mqa
