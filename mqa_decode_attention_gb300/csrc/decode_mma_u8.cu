// gqa_decode_attention on tensor cores over a uint8 cache (MQA_U8), the
// pages' QuantizedKVCache ("KV Cache 최적화 심층 분석", youngju.dev): each
// cached (token, kv head) row is codes c in [0, 255] with one (scale s,
// zero point z) pair, value (c - z) s.
//
// The codes go into fp16 MMAs without a dequantised copy:
//   * a byte permute turns codes into fp16 pairs 1024 + c (bit pattern
//     0x64cc), exact;
//   * S_t = s^k_t * sum_d q_d (c_td - z_t): the zero point comes off the fp32
//     score through the row sum of q, and the K scale multiplies it;
//   * O = sum_t (p_t s^v_t) (c_t - z_t): the V scale is folded into P, which
//     enters the second MMA as fp16 p * s^v * 64 (the factor 64 keeps small
//     scales out of fp16's subnormal range and is divided out at the end);
//     the zero-point term is one extra MMA column.
// Head dims are permuted consistently on both MMA operands so that each lane
// reads its codes as whole 16-byte words (see the fragment notes below), and
// the output's dims are put back in order when the block merges its warps.
//
// The same kernels read an fp8 e5m2 cache (template flag F8): an e5m2 value
// is an IEEE half with its low byte zero, so a byte permute makes the exact
// fp16 operand, and there is no scale, zero point or P' factor.
//
// Block = 4 consumer warps per head block of 16 query heads + 1 producer warp.
// The producer streams 64-token tiles of codes (TMA, 128- or 64-byte swizzle)
// and of the (scale, zero) rows, contiguous or page by page through the block
// table; two consumer warps share a tile, 32 tokens each, and the other two
// take the next tile.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>

#include "../../include/mqa_decode.h"
#include "launch.h"
#include "mma_warp.cuh"
#include "ptx.cuh"
#include "quant.cuh"
#include "rope.cuh"

namespace mqa {
namespace {

constexpr float kPScale = 64.0f;       // P' = p * s^v * kPScale in fp16
constexpr float kMaxVScale = 1023.0f;  // p * s^v * kPScale stays below fp16's 65504

template <int D>
struct U8Stages {
  static constexpr int value = D == 128 ? 6 : 8;  // even: a tile's parity fixes its stages
};

template <int D, int HB, int STAGES, bool F8 = false>
struct U8Cfg {
  static constexpr int kConsumerWarps = 4 * HB;
  static constexpr int kConsumerThreads = 32 * kConsumerWarps;
  static constexpr int kThreads = kConsumerThreads + 64;  // + producer warp + append warp (fused step)
  static constexpr int kCodeBytes = kTile * D;  // codes of a K (or V) tile
  static constexpr int kSzBytes = F8 ? 0 : kTile * 8;  // (scale, zero) pairs of a tile
  static constexpr int kStageBytes = 2 * kCodeBytes + 2 * kSzBytes;
  static constexpr int kPipeBytes = STAGES * kStageBytes;
  static constexpr int kMergeStride = D + 4;
  static constexpr int kMergeBytes = kConsumerWarps * 16 * (kMergeStride + 2) * 4;
  static constexpr int kBodyBytes = kPipeBytes > kMergeBytes ? kPipeBytes : kMergeBytes;
  static constexpr int kSmemBytes = kBodyBytes + 2 * STAGES * 8 + 1024;
  static_assert(kStageBytes % 1024 == 0, "stages stay 1 KB aligned (swizzle atoms)");
};

// Byte offset of 16-byte chunk `ch` of code row r, as TMA's swizzle wrote
// it. Rows come in blocks of 16 that start on 1 KB boundaries, `bs` bytes
// apart; inside a block, 128-byte rows (D = 128) sit under the 128-byte
// swizzle (chunk ch ^ (r mod 8)) and 64-byte rows (D = 64) under the 64-byte
// swizzle (chunk ch ^ ((r / 2) mod 4)).
template <int D, uint32_t BS>
__device__ __forceinline__ uint32_t code_off(int r, int ch) {
  const uint32_t row = BS == 16 * D ? r * D : (r >> 4) * BS + (r & 15) * D;  // rows back to back, or blocks
  if constexpr (D == 128) return row + ((ch ^ (r & 7)) << 4);
  return row + ((ch ^ ((r >> 1) & 3)) << 4);
}

// Byte offset of the (scale, zero) pair of row r: blocks of 16 rows BS apart.
template <uint32_t BS>
__device__ __forceinline__ uint32_t sz_off(int r) {
  return BS == 128 ? r * 8 : (r >> 4) * BS + (r & 15) * 8;
}

__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ float4 lds_f4(uint32_t a) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
  return v;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// D = A * B + D, m16n8k16, fp16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two codes of w (bytes 0, 1 with kSelLo; bytes 2, 3 with kSelHi) as the fp16
// pair (1024 + c_first, 1024 + c_second).
__device__ __forceinline__ uint32_t codes_f16(uint32_t w, uint32_t sel) { return __byte_perm(w, 0x64u, sel); }
constexpr uint32_t kSelLo = 0x4140u;
constexpr uint32_t kSelHi = 0x4342u;
// Two e5m2 codes of w (bytes 0, 1 / bytes 2, 3) as the fp16 pair whose high
// bytes they are: exact.
constexpr uint32_t kF8Lo = 0x1404u;
constexpr uint32_t kF8Hi = 0x3424u;

// One warp's share of the attention over a uint8 cache: up to 16 query heads
// (MMA rows) against 32 consecutive tokens per step.
//
// Fragment layout (mma m16n8k16, lane = 4 g + c): the A and B operands of a
// lane cover the same k positions {2c, 2c+1, 2c+8, 2c+9}.
//   S = Q K^T: k runs over head dims. At k-step ks, positions 2c + {0, 1} are
//     dims (D/4) c + 4 ks + {0, 1} and positions 2c + 8 + {0, 1} are dims
//     (D/4) c + 4 ks + {2, 3}: lane c's dims are one contiguous run of D/4
//     codes of its token row (B column g), read as 16-byte words. The four
//     n8 tiles of a step are tokens 8 nt .. 8 nt + 7.
//   O = P V: k runs over 16 tokens (position = token) for each half of the
//     step; output column g of dim tile dn is head dim g (D/8) + dn, so lane g
//     reads D/8 contiguous codes of each of its tokens 2c, 2c+1, 2c+8, 2c+9.
// Zero points never touch the elements: the MMAs see 1024 + c, and
//   S_t = s^k_t (sum_d q_d (1024 + c_td) - (1024 + z_t) sum_d q_d)
//   O   = sum_t p'_t (1024 + c_t) - sum_t p'_t (1024 + z_t),
// the last sum being one more n8 MMA tile whose B column is 1024 + z_t, so it
// sees exactly the fp16 P' the data columns see.
template <int D, bool F8 = false>
struct WarpAttnU8 {
  uint32_t qa[D / 16][4];  // Q (fp16, log2-domain scale folded in), permuted dims
  float o[D / 8][4];       // O + zero-point terms: rows g (regs 0,1) and g + 8 (regs 2,3)
  float cz[4];             // sum_t p'_t (1024 + z_t): rows g (reg 0) and g + 8 (reg 2)
  float qs0, qs1;          // sum_d of the fp16 Q rows g and g + 8
  float m0, m1, l0, l1;
  float vmax;  // largest V scale seen (range check)

  __device__ __forceinline__ void init(const float* q, int rows_valid, float scale_log2, int lane) {
    const int g = lane >> 2, c = lane & 3;
    init_from(
        [&](int ks, int hi) {
          const int row = g + 8 * hi;
          return row < rows_valid ? *reinterpret_cast<const float4*>(q + row * D + (D / 4) * c + 4 * ks)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
        },
        scale_log2);
  }

  // Rows g and g + 8 from two row pointers (several new tokens: the warp's 16
  // rows are (token, head) pairs, not consecutive heads); null = zeros.
  __device__ __forceinline__ void init_rows(const float* qa, const float* qb, float scale_log2, int lane) {
    const int c = lane & 3;
    init_from(
        [&](int ks, int hi) {
          const float* q = hi ? qb : qa;
          return q != nullptr ? *reinterpret_cast<const float4*>(q + (D / 4) * c + 4 * ks)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
        },
        scale_log2);
  }

  // This lane's raw bf16 q_new values (rows g, g + 8 of the warp's 16 heads;
  // dims (D/4) c + 4 ks .. + 3: two rotation pairs), rows >= rows_valid zero.
  // Kept apart from init_rope so the loads are in flight while the cos / sin
  // table is formed.
  __device__ __forceinline__ static void load_q(const __nv_bfloat16* q, int rows_valid, int lane,
                                                uint2 (&raw)[D / 16][2]) {
    const int g = lane >> 2, c = lane & 3;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
      for (int hi = 0; hi < 2; ++hi) {
        const int row = g + 8 * hi;
        raw[ks][hi] = row < rows_valid ? *reinterpret_cast<const uint2*>(q + row * D + (D / 4) * c + 4 * ks)
                                       : make_uint2(0u, 0u);
      }
    }
  }

  // Same as init, from the raw q_new of load_q rotated first: pair i turns by
  // the angle whose fp32 cosine / sine are cs[i] / cs[D/2 + i], as the other
  // fused kernels form q_rot (written to q_rot_out, [16][D] fp32, unless null).
  __device__ __forceinline__ void init_rope(const uint2 (&raw)[D / 16][2], int rows_valid, const float* cs,
                                            float scale_log2, int lane, float* q_rot_out) {
    const int g = lane >> 2, c = lane & 3;
    init_from(
        [&](int ks, int hi) {
          const int row = g + 8 * hi;
          const int col = (D / 4) * c + 4 * ks, i = col >> 1;
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
          if (row < rows_valid) {
            const uint2 w = raw[ks][hi];
            const float x0 = bf16lo_to_f32(w.x), y0 = bf16hi_to_f32(w.x);
            const float x1 = bf16lo_to_f32(w.y), y1 = bf16hi_to_f32(w.y);
            const float c0 = cs[i], s0 = cs[D / 2 + i], c1 = cs[i + 1], s1 = cs[D / 2 + i + 1];
            v = make_float4(x0 * c0 - y0 * s0, x0 * s0 + y0 * c0, x1 * c1 - y1 * s1, x1 * s1 + y1 * c1);
            if (q_rot_out != nullptr) *reinterpret_cast<float4*>(q_rot_out + row * D + col) = v;
          }
          return v;
        },
        scale_log2);
  }

  // Q fragments from q4(ks, hi) = the lane's four fp32 values of row g + 8 hi
  // (g = lane / 4), dims (D/4) c + 4 ks .. + 3; the other state reset.
  template <class F>
  __device__ __forceinline__ void init_from(F q4, float scale_log2) {
    qs0 = qs1 = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
      for (int hi = 0; hi < 2; ++hi) {
        const float4 v = q4(ks, hi);
        const __half2 h01 = __floats2half2_rn(v.x * scale_log2, v.y * scale_log2);
        const __half2 h23 = __floats2half2_rn(v.z * scale_log2, v.w * scale_log2);
        qa[ks][hi] = *reinterpret_cast<const uint32_t*>(&h01);
        qa[ks][2 + hi] = *reinterpret_cast<const uint32_t*>(&h23);
        const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
        const float part = (f01.x + f01.y) + (f23.x + f23.y);
        if (hi) qs1 += part; else qs0 += part;
      }
    }
    qs0 += __shfl_xor_sync(0xffffffffu, qs0, 1);
    qs0 += __shfl_xor_sync(0xffffffffu, qs0, 2);
    qs1 += __shfl_xor_sync(0xffffffffu, qs1, 1);
    qs1 += __shfl_xor_sync(0xffffffffu, qs1, 2);
#pragma unroll
    for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    cz[0] = cz[1] = cz[2] = cz[3] = 0.f;
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
    vmax = 0.f;
  }

  // Rows [trow0, trow0 + 32) of the code tiles at shared addresses kc / vc
  // (16-row blocks CBS bytes apart) and of the (scale, zero) rows at ksz / vsz
  // (16-row blocks SBS bytes apart); only rows lo .. hi-1 of the 32 are real
  // tokens. The others may hold anything (NaN scales included): their scores
  // are masked and their P' and zero points forced to 0. MULTI: row g sees
  // only tokens [lo0, hi0) and row g + 8 only [lo1, hi1) (within [lo, hi)),
  // and a row that has seen no token yet keeps a -inf maximum.
  template <uint32_t CBS, uint32_t SBS, bool MULTI = false>
  __device__ __forceinline__ void step(uint32_t kc, uint32_t vc, uint32_t ksz, uint32_t vsz, int trow0, int lo,
                                       int hi, int lane, int lo0 = 0, int hi0 = 32, int lo1 = 0, int hi1 = 32) {
    const int g = lane >> 2, c = lane & 3;
    auto lo2 = [](uint32_t x) { return F8 ? __byte_perm(x, 0u, kF8Lo) : codes_f16(x, kSelLo); };
    auto hi2 = [](uint32_t x) { return F8 ? __byte_perm(x, 0u, kF8Hi) : codes_f16(x, kSelHi); };
    // ---- raw scores sum_d q_d (1024 + c_td) (e5m2: sum_d q_d k_td): four n8
    // tiles, four independent MMA chains
    float s[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) s[nt][e] = 0.f;
    }
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int row = trow0 + nt * 8 + g;  // this lane's B column (token)
      uint32_t w[D / 16];
      if constexpr (D == 128) {
        const uint4 a = lds128(kc + code_off<D, CBS>(row, 2 * c));
        const uint4 b = lds128(kc + code_off<D, CBS>(row, 2 * c + 1));
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
        w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
      } else {
        const uint4 a = lds128(kc + code_off<D, CBS>(row, c));
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
      }
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        mma_f16_16816(s[nt], qa[ks], lo2(w[ks]), hi2(w[ks]));
    }
    // ---- scales and zero points of this lane's columns: tokens 8 nt + 2c + {0, 1}
    float sv[4][2], zv[4][2];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      if constexpr (F8) break;
      const float4 kq = lds_f4(ksz + sz_off<SBS>(trow0 + nt * 8 + 2 * c));
      const float4 vq = lds_f4(vsz + sz_off<SBS>(trow0 + nt * 8 + 2 * c));
      const float off0 = 1024.f + kq.y, off1 = 1024.f + kq.w;
      s[nt][0] = kq.x * fmaf(-off0, qs0, s[nt][0]);
      s[nt][1] = kq.z * fmaf(-off1, qs0, s[nt][1]);
      s[nt][2] = kq.x * fmaf(-off0, qs1, s[nt][2]);
      s[nt][3] = kq.z * fmaf(-off1, qs1, s[nt][3]);
      sv[nt][0] = vq.x;
      zv[nt][0] = vq.y;
      sv[nt][1] = vq.z;
      zv[nt][1] = vq.w;
    }
    const bool partial = lo > 0 || hi < 32;
    if (partial) {  // a partial step: mask the rows outside [lo, hi)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t = nt * 8 + 2 * c + e;
          if (t < lo || t >= hi) {
            s[nt][e] = -INFINITY;
            s[nt][2 + e] = -INFINITY;
            sv[nt][e] = 0.f;
            zv[nt][e] = 0.f;
          }
        }
      }
    }
    if constexpr (MULTI) {
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t = nt * 8 + 2 * c + e;
          if (t < lo0 || t >= hi0) s[nt][e] = -INFINITY;
          if (t < lo1 || t >= hi1) s[nt][2 + e] = -INFINITY;
        }
      }
    }
    if constexpr (!F8) {
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) vmax = fmaxf(vmax, fmaxf(sv[nt][0], sv[nt][1]));
    }
    // ---- online softmax (log2 domain), rows g and g + 8
    float mx0 = fmaxf(fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1])),
                      fmaxf(fmaxf(s[2][0], s[2][1]), fmaxf(s[3][0], s[3][1])));
    float mx1 = fmaxf(fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3])),
                      fmaxf(fmaxf(s[2][2], s[2][3]), fmaxf(s[3][2], s[3][3])));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const bool moved = (mn0 != m0) || (mn1 != m1);
    // (MULTI: a row with no token yet subtracts 0 instead of its -inf maximum)
    const float e0 = (MULTI && mn0 == -INFINITY) ? 0.f : mn0, e1 = (MULTI && mn1 == -INFINITY) ? 0.f : mn1;
    const float a0 = fast_exp2(m0 - e0), a1 = fast_exp2(m1 - e1);
    m0 = mn0;
    m1 = mn1;
    float pr[4][4];
    float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      pr[nt][0] = fast_exp2(s[nt][0] - e0);
      pr[nt][1] = fast_exp2(s[nt][1] - e0);
      pr[nt][2] = fast_exp2(s[nt][2] - e1);
      pr[nt][3] = fast_exp2(s[nt][3] - e1);
      sum0 += pr[nt][0] + pr[nt][1];
      sum1 += pr[nt][2] + pr[nt][3];
    }
    l0 = l0 * a0 + sum0;
    l1 = l1 * a1 + sum1;
    if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        o[n][0] *= a0;
        o[n][1] *= a0;
        o[n][2] *= a1;
        o[n][3] *= a1;
      }
      if constexpr (!F8) {
        cz[0] *= a0;
        cz[1] *= a0;
        cz[2] *= a1;
        cz[3] *= a1;
      }
    }
    // ---- P' = p s^v kPScale and the zero-point column 1024 + z, packed to fp16
    // for both 16-token halves before the V codes are read
    uint32_t pa[2][4], zb[2][2];
#pragma unroll
    for (int kh = 0; kh < 2; ++kh) {
      const int n0 = 2 * kh, n1 = 2 * kh + 1;
      if constexpr (F8) {  // P as it is
        pa[kh][0] = pack_f16x2(pr[n0][0], pr[n0][1]);
        pa[kh][1] = pack_f16x2(pr[n0][2], pr[n0][3]);
        pa[kh][2] = pack_f16x2(pr[n1][0], pr[n1][1]);
        pa[kh][3] = pack_f16x2(pr[n1][2], pr[n1][3]);
        continue;
      }
      const float w00 = sv[n0][0] * kPScale, w01 = sv[n0][1] * kPScale;
      const float w10 = sv[n1][0] * kPScale, w11 = sv[n1][1] * kPScale;
      pa[kh][0] = pack_f16x2(pr[n0][0] * w00, pr[n0][1] * w01);
      pa[kh][1] = pack_f16x2(pr[n0][2] * w00, pr[n0][3] * w01);
      pa[kh][2] = pack_f16x2(pr[n1][0] * w10, pr[n1][1] * w11);
      pa[kh][3] = pack_f16x2(pr[n1][2] * w10, pr[n1][3] * w11);
      zb[kh][0] = pack_f16x2(1024.f + zv[n0][0], 1024.f + zv[n0][1]);
      zb[kh][1] = pack_f16x2(1024.f + zv[n1][0], 1024.f + zv[n1][1]);
    }
    // ---- O += P' (1024 + V codes), cz += P' (1024 + z), per 16-token half
#pragma unroll
    for (int kh = 0; kh < 2; ++kh) {
      if constexpr (!F8) mma_f16_16816(cz, pa[kh], zb[kh][0], zb[kh][1]);
      const int r0 = trow0 + 16 * kh + 2 * c;
      // this lane's dims g (D/8) .. g (D/8) + D/8 - 1 of tokens 2c, 2c+1, 2c+8, 2c+9 of the half
      uint32_t ra[D / 32], rb[D / 32], rc[D / 32], rd[D / 32];
      if constexpr (D == 128) {
        const uint4 x0 = lds128(vc + code_off<D, CBS>(r0, g));
        const uint4 x1 = lds128(vc + code_off<D, CBS>(r0 + 1, g));
        const uint4 x2 = lds128(vc + code_off<D, CBS>(r0 + 8, g));
        const uint4 x3 = lds128(vc + code_off<D, CBS>(r0 + 9, g));
        ra[0] = x0.x; ra[1] = x0.y; ra[2] = x0.z; ra[3] = x0.w;
        rb[0] = x1.x; rb[1] = x1.y; rb[2] = x1.z; rb[3] = x1.w;
        rc[0] = x2.x; rc[1] = x2.y; rc[2] = x2.z; rc[3] = x2.w;
        rd[0] = x3.x; rd[1] = x3.y; rd[2] = x3.z; rd[3] = x3.w;
      } else {
        // 8 codes per row; odd c read row 2c+1 first so that the loads of a
        // half warp fall on distinct banks
        const int sw = c & 1;
        const uint32_t off = 8 * (g & 1);
        const uint2 y0 = lds64(vc + code_off<D, CBS>(r0 + sw, g >> 1) + off);
        const uint2 y1 = lds64(vc + code_off<D, CBS>(r0 + 1 - sw, g >> 1) + off);
        const uint2 y2 = lds64(vc + code_off<D, CBS>(r0 + 8 + sw, g >> 1) + off);
        const uint2 y3 = lds64(vc + code_off<D, CBS>(r0 + 9 - sw, g >> 1) + off);
        ra[0] = sw ? y1.x : y0.x; ra[1] = sw ? y1.y : y0.y;
        rb[0] = sw ? y0.x : y1.x; rb[1] = sw ? y0.y : y1.y;
        rc[0] = sw ? y3.x : y2.x; rc[1] = sw ? y3.y : y2.y;
        rd[0] = sw ? y2.x : y3.x; rd[1] = sw ? y2.y : y3.y;
      }
      if constexpr (F8) {
        // tokens outside [lo, hi) may hold any byte, NaN codes included: their
        // P is 0, and 0 * NaN would still poison O, so their codes become 0
        if (partial) {
          const int t0 = 16 * kh + 2 * c;
          const bool da = t0 < lo || t0 >= hi, db = t0 + 1 < lo || t0 + 1 >= hi;
          const bool dc = t0 + 8 < lo || t0 + 8 >= hi, dd = t0 + 9 < lo || t0 + 9 >= hi;
#pragma unroll
          for (int wi = 0; wi < D / 32; ++wi) {
            if (da) ra[wi] = 0u;
            if (db) rb[wi] = 0u;
            if (dc) rc[wi] = 0u;
            if (dd) rd[wi] = 0u;
          }
        }
      }
#pragma unroll
      for (int wi = 0; wi < D / 32; ++wi) {
        // interleave the codes of tokens (2c, 2c+1) and (2c+8, 2c+9) byte by byte
        const uint32_t x01 = __byte_perm(ra[wi], rb[wi], 0x5140u), y01 = __byte_perm(ra[wi], rb[wi], 0x7362u);
        const uint32_t x89 = __byte_perm(rc[wi], rd[wi], 0x5140u), y89 = __byte_perm(rc[wi], rd[wi], 0x7362u);
        mma_f16_16816(o[4 * wi + 0], pa[kh], lo2(x01), lo2(x89));
        mma_f16_16816(o[4 * wi + 1], pa[kh], hi2(x01), hi2(x89));
        mma_f16_16816(o[4 * wi + 2], pa[kh], lo2(y01), lo2(y89));
        mma_f16_16816(o[4 * wi + 3], pa[kh], hi2(y01), hi2(y89));
      }
    }
  }

  // Row sums over the 4 lanes of a row; the zero-point term subtracted and
  // the P' factor divided out of O.
  __device__ __forceinline__ void finish() {
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    if constexpr (F8) return;
    constexpr float inv = 1.0f / kPScale;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      o[n][0] = (o[n][0] - cz[0]) * inv;
      o[n][1] = (o[n][1] - cz[1]) * inv;
      o[n][2] = (o[n][2] - cz[2]) * inv;
      o[n][3] = (o[n][3] - cz[3]) * inv;
    }
  }
};

// MULTI: n_new > 1 new tokens per sequence (the verification of drafted
// tokens): the rows of a kv head are (new token i, query head h) pairs, row =
// i G + h, and row i sees the tokens up to L - n + i only (the bf16 warp-MMA
// kernel's scheme). The new rows come from a preceding append launch.
template <int D, int HB, int STAGES, bool F8, bool MULTI>
__global__ void __launch_bounds__(U8Cfg<D, HB, STAGES, F8>::kThreads, HB == 1 ? 2 : 1)
    decode_u8_kernel(const __grid_constant__ CUtensorMap tm_kc, const __grid_constant__ CUtensorMap tm_vc,
                     const __grid_constant__ CUtensorMap tm_ks, const __grid_constant__ CUtensorMap tm_vs,
                     const DecodeParams p) {
  using C = U8Cfg<D, HB, STAGES, F8>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBodyBytes);
  uint64_t* empty = full + STAGES;
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.num_splits;
  int cta = blockIdx.x;
  const int hsb = cta % p.head_blocks;
  cta /= p.head_blocks;
  const int split = cta % S;
  cta /= S;
  const int j = cta % p.h_kv;
  const int b = cta / p.h_kv;
  const int G = p.group;
  const int nq = MULTI ? p.n_new : 1;  // new tokens (query rows per head) of each sequence
  const int R = G * nq;                // query rows of this kv head

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), C::kConsumerWarps / 2);  // the warps of one tile parity
    }
    fence_mbar_init();
  }
  __syncthreads();
  // the combine (or the next step) may be scheduled now; it waits for this
  // whole grid before it reads anything this grid writes
  grid_dependents_launch();
  if (!p.early) grid_dependency_wait();
  long long limit = p.paged ? static_cast<long long>(p.max_pages) * p.page_size : p.capacity;
  if (limit > p.max_seq_len) limit = p.max_seq_len;
  int L = p.seq_lens[b];
  if (L < nq || L > limit) {
    if (threadIdx.x == 0 && split == 0 && hsb == 0) atomicOr(p.err, static_cast<int>(MQA_DEVERR_SEQ_LEN));
    L = L < nq ? (L < 0 ? 0 : L) : static_cast<int>(limit);
  }
  // sliding window: tokens [t_lo, L) (t_lo of the first new token, the lowest)
  const int t_lo = p.window > 0 ? max(0, L - nq + 1 - p.window) : 0;
  const int t_base = (t_lo / kTile) * kTile;
  const int t_begin = t_base + split * p.chunk;
  int t_end = min(L, t_begin + p.chunk);
  if (MULTI) {
    // keys past this block's last row are masked for all of its rows (a
    // prompt's early rows read only the early keys)
    const int last_row = min(R, (hsb + 1) * HB * 16) - 1;
    t_end = min(t_end, L - nq + last_row / G + 1);
  }
  const int n_tiles = t_end > t_begin ? (t_end - t_begin + kTile - 1) / kTile : 0;

  // the fused append (no append launch precedes this one): one block per
  // sequence and kv head quantises and writes the new token's rows
  const int apos = p.fuse_append ? p.pos[b] : 0;
  const bool awaits = p.fuse_append && hsb == 0 && split == append_split(apos - t_base, p.chunk, S);
  if (warp == C::kConsumerWarps + 1) {
    // --------------------------------------------------------- append warp
    // writes the rows, fences them for the async proxy and releases the
    // producer, which waits (named barrier 3) only before the tile holding them
    if (awaits) {
      append_row_q<D, F8>(p, b, j, apos, cache_row(p, b, j, apos, lane == 0), lane);
      named_bar_arrive(3, 64);
    }
    return;
  }
  if (warp == C::kConsumerWarps) {
    // ------------------------------------------------------------ producer
    const int ps = p.page_size;
    const int rpc = ps < kTile ? ps : kTile;  // rows per copy
    const int32_t* trow = p.block_table + static_cast<long long>(b) * p.max_pages;
    const int n_pages_seq = p.paged ? (L + ps - 1) / ps : 0;
    // table entries of 32 consecutive pages, one per lane, and of the next 32
    int wbase = p.paged ? t_begin / ps : 0;
    int wcur = -1, wnxt = -1;
    if (p.paged) {
      wcur = (wbase + lane < n_pages_seq) ? __ldg(trow + wbase + lane) : -1;
      wnxt = (wbase + 32 + lane < n_pages_seq) ? __ldg(trow + wbase + 32 + lane) : -1;
    }
    int issued = 0;
    bool waited = !p.early, appended = !awaits;
    for (int it = 0; it < n_tiles; ++it) {
      const int stage = it % STAGES;
      if (it >= STAGES) {
        if (!mbar_wait(smem_u32(&empty[stage]), ((it / STAGES) + 1) & 1, p.wait_ns)) {
          if (lane == 0) {
            s_abort = 1;
            atomicOr(p.err, static_cast<int>(MQA_DEVERR_TIMEOUT));
          }
          break;
        }
      }
      if (*reinterpret_cast<volatile int*>(&s_abort)) break;
      const int t0 = t_begin + it * kTile;
      if (!waited && L - nq < t0 + kTile) {  // this tile holds an appended token
        grid_dependency_wait();
        waited = true;
      }
      if (!appended && apos < t0 + kTile) {  // this tile holds the rows the append warp writes
        named_bar_sync(3, 64);
        appended = true;
      }
      const uint32_t base = smem_u32(smem + stage * C::kStageBytes);
      const uint32_t kc = base, vc = base + C::kCodeBytes;
      const uint32_t ksd = base + 2 * C::kCodeBytes, vsd = ksd + C::kSzBytes;
      const uint32_t fb = smem_u32(&full[stage]);
      if (!p.paged) {
        if (lane == 0) {
          mbar_arrive_expect_tx(fb, C::kStageBytes);
          const int row = b * p.h_kv + j;
          tma_load_3d(kc, &tm_kc, 0, t0, row, fb);
          tma_load_3d(vc, &tm_vc, 0, t0, row, fb);
          if constexpr (!F8) {
            tma_load_2d(ksd, &tm_ks, 2 * t0, row, fb);
            tma_load_2d(vsd, &tm_vs, 2 * t0, row, fb);
          }
        }
      } else {
        int pg[kTile / 16];
#pragma unroll
        for (int k = 0; k < kTile / 16; ++k) {
          pg[k] = -1;
          if (k * rpc < kTile) {
            int lp = (t0 + k * rpc) / ps;
            if (t0 + k * rpc + rpc <= t_lo) lp = t_lo / ps;  // wholly before the window: any live page
            if (lp >= n_pages_seq) lp = n_pages_seq - 1;
            while (lp >= wbase + 32) {
              wbase += 32;
              wcur = wnxt;
              wnxt = (wbase + 32 + lane < n_pages_seq) ? __ldg(trow + wbase + 32 + lane) : -1;
            }
            pg[k] = __shfl_sync(0xffffffffu, wcur, lp - wbase);
            if (pg[k] < 0 || pg[k] >= p.num_pages) {
              if (lane == 0) atomicOr(p.err, static_cast<int>(MQA_DEVERR_PAGE_RANGE));
              pg[k] = -1;
            }
          }
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(fb, C::kStageBytes);
#pragma unroll
          for (int k = 0; k < kTile / 16; ++k) {
            if (k * rpc >= kTile) break;
            const int r = (t0 + k * rpc) % ps;
            // a page outside the pool is read at a coordinate past the pool: TMA's zero fill
            const int page = pg[k] < 0 ? p.num_pages : pg[k];
            tma_load_4d(kc + k * rpc * D, &tm_kc, 0, r, j, page, fb);
            tma_load_4d(vc + k * rpc * D, &tm_vc, 0, r, j, page, fb);
            if constexpr (!F8) {
              tma_load_3d(ksd + k * rpc * 8, &tm_ks, 2 * r, j, page, fb);
              tma_load_3d(vsd + k * rpc * 8, &tm_vs, 2 * r, j, page, fb);
            }
          }
        }
      }
      __syncwarp();
      issued = it + 1;
    }
    if (!appended) named_bar_sync(3, 64);  // pair the append warp's arrival
    // every copy this warp issued lands before the block can exit: after a
    // timeout the consumers may have stopped waiting for them
    for (int it = (issued > STAGES ? issued - STAGES : 0); it < issued; ++it)
      (void)mbar_wait(smem_u32(&full[it % STAGES]), (it / STAGES) & 1, kWaitLimitNs);
    return;
  }

  // -------------------------------------------------------------- consumers
  const int hb = warp >> 2;
  const int ws = warp & 3;
  const int head0 = (hsb * HB + hb) * 16;
  WarpAttnU8<D, F8> wa;
  if (p.rope_q) {
    // fused step: q_new rotated here (its loads issued before the cos / sin
    // table is formed)
    __shared__ float s_cs[D];
    const long long qoff = (static_cast<long long>(b) * p.h_q + j * G + head0) * D;
    uint2 qraw[D / 16][2];
    WarpAttnU8<D, F8>::load_q(static_cast<const __nv_bfloat16*>(p.q_new) + qoff, G - head0, lane, qraw);
    rope_table<D>(s_cs, p, p.pos[b], threadIdx.x, 2, C::kConsumerThreads);
    wa.init_rope(qraw, G - head0, s_cs, p.scale_log2, lane,
                 (p.fuse_append && split == 0 && ws == 0) ? p.q_rot_out + qoff : nullptr);
  } else if (MULTI) {
    if (p.early) grid_dependency_wait();  // q_rot is written by the append kernel
    auto qrow = [&](int r) -> const float* {
      if (r >= R) return nullptr;
      const int i = r / G;
      return p.q_rot + ((static_cast<long long>(b) * nq + i) * p.h_q + j * G + (r - i * G)) * D;
    };
    wa.init_rows(qrow(head0 + (lane >> 2)), qrow(head0 + (lane >> 2) + 8), p.scale_log2, lane);
  } else {
    if (p.early) grid_dependency_wait();  // q_rot is written by the append kernel
    wa.init(p.q_rot + (static_cast<long long>(b) * p.h_q + j * G + head0) * D, G - head0, p.scale_log2, lane);
  }
  // MULTI: the key range [ka, ke) of this lane's rows g and g + 8 (row of new
  // token i: ends after position L - n + i; a window of W before that)
  int ka0 = 0, ke0 = L, ka1 = 0, ke1 = L;
  if (MULTI) {
    const int i0 = min(head0 + (lane >> 2), R - 1) / G, i1 = min(head0 + (lane >> 2) + 8, R - 1) / G;
    ke0 = L - nq + i0 + 1;
    ke1 = L - nq + i1 + 1;
    ka0 = p.window > 0 ? max(0, ke0 - p.window) : 0;
    ka1 = p.window > 0 ? max(0, ke1 - p.window) : 0;
  }

  // warps 0, 1 of a head block take the even tiles, warps 2, 3 the odd
  // ones; each warp 32 tokens of its tiles
  const int trow0 = (ws & 1) * 32;
  bool ok = true;
  for (int it = ws >> 1; it < n_tiles; it += 2) {
    const int stage = it % STAGES;
    if (!mbar_wait(smem_u32(&full[stage]), (it / STAGES) & 1, p.wait_ns)) {
      if (lane == 0) {
        s_abort = 1;
        atomicOr(p.err, static_cast<int>(MQA_DEVERR_TIMEOUT));
      }
      ok = false;
      break;
    }
    const uint32_t st = smem_u32(smem + stage * C::kStageBytes);
    const int tt = t_begin + it * kTile + trow0;
    const int lo = max(0, t_lo - tt), hi = min(32, t_end - tt);
    if (lo < hi) {
      if constexpr (MULTI)
        wa.template step<16 * D, 128, true>(st, st + C::kCodeBytes, st + 2 * C::kCodeBytes,
                                            st + 2 * C::kCodeBytes + C::kSzBytes, trow0, lo, hi, lane,
                                            max(0, ka0 - tt), min(32, min(ke0, t_end) - tt), max(0, ka1 - tt),
                                            min(32, min(ke1, t_end) - tt));
      else
        wa.template step<16 * D, 128>(st, st + C::kCodeBytes, st + 2 * C::kCodeBytes,
                                      st + 2 * C::kCodeBytes + C::kSzBytes, trow0, lo, hi, lane);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[stage]));
  }
  wa.finish();
  if (!F8 && __any_sync(0xffffffffu, wa.vmax > kMaxVScale) && lane == 0)
    atomicOr(p.err, static_cast<int>(MQA_DEVERR_U8_SCALE));

  // ------------------------------------------- merge the 4 token slices
  // one decision for every consumer warp (the producer may time out and set
  // s_abort at any moment); the barrier also ends their reads of the stages
  if (bar_any(4, C::kConsumerThreads, *reinterpret_cast<volatile int*>(&s_abort) || !ok)) return;
  float* mo = reinterpret_cast<float*>(smem);  // [warp][16][kMergeStride], columns in fragment order
  float* mm = mo + C::kConsumerWarps * 16 * C::kMergeStride;
  float* ml = mm + C::kConsumerWarps * 16;
  {
    const int g = lane >> 2, c2 = (lane & 3) * 2;
    float* mine = mo + warp * 16 * C::kMergeStride;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      *reinterpret_cast<float2*>(mine + g * C::kMergeStride + n * 8 + c2) = make_float2(wa.o[n][0], wa.o[n][1]);
      *reinterpret_cast<float2*>(mine + (g + 8) * C::kMergeStride + n * 8 + c2) =
          make_float2(wa.o[n][2], wa.o[n][3]);
    }
    if ((lane & 3) == 0) {
      mm[warp * 16 + g] = wa.m0;
      mm[warp * 16 + g + 8] = wa.m1;
      ml[warp * 16 + g] = wa.l0;
      ml[warp * 16 + g + 8] = wa.l1;
    }
  }
  named_bar_sync(1, C::kConsumerThreads);

  const bool split_out = S > 1;
  const int tid = threadIdx.x;
  for (int hbi = 0; hbi < HB; ++hbi) {
    const int hh0 = (hsb * HB + hbi) * 16;
    const int n_rows = min(16, R - hh0);
    for (int idx = tid; idx < n_rows * D; idx += C::kConsumerThreads) {
      const int r = idx / D, d = idx - r * D;
      const int pc = (d % (D / 8)) * 8 + d / (D / 8);  // head dim d = column (D/8) + dim tile
      float mx = -INFINITY;
#pragma unroll
      for (int w = 0; w < 4; ++w) mx = fmaxf(mx, mm[(hbi * 4 + w) * 16 + r]);
      float num = 0.f, den = 0.f;
      if (mx != -INFINITY) {
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const int ww = hbi * 4 + w;
          const float wt = exp2f(mm[ww * 16 + r] - mx);
          num = fmaf(wt, mo[(ww * 16 + r) * C::kMergeStride + pc], num);
          den = fmaf(wt, ml[ww * 16 + r], den);
        }
      }
      const float ov = den > 0.f ? num / den : 0.f;
      const float lse = den > 0.f ? (mx + log2f(den)) * 0.69314718055994530942f : -INFINITY;
      long long grow = static_cast<long long>(b) * p.h_q + j * G + hh0 + r;  // output row [B, (n,) H_q]
      if (MULTI) {
        const int i = (hh0 + r) / G;
        grow = (static_cast<long long>(b) * nq + i) * p.h_q + j * G + (hh0 + r - i * G);
      }
      if (split_out) {
        p.o_part[(grow * S + split) * D + d] = ov;
        if (d == 0) p.lse_part[grow * S + split] = lse;
      } else {
        if (p.out_dtype == kDtypeBf16)
          static_cast<__nv_bfloat16*>(p.out)[grow * D + d] = __float2bfloat16_rn(ov);
        else
          static_cast<float*>(p.out)[grow * D + d] = ov;
        if (d == 0 && p.lse_out != nullptr) p.lse_out[grow] = lse;
      }
    }
  }
}

template <int D, int HB, bool F8, bool MULTI>
cudaError_t launch_u8_t(const DecodeParams& p, const CUtensorMap* maps, cudaStream_t stream) {
  constexpr int ST = U8Stages<D>::value;
  using C = U8Cfg<D, HB, ST, F8>;
  auto kern = decode_u8_kernel<D, HB, ST, F8, MULTI>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.batch) * p.h_kv * p.head_blocks * p.num_splits);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], maps[3], p);
}

// Blocks per SM as the occupancy calculator sees them (registers bound the
// 288-thread blocks to one); 0 if there is no device to ask.
template <int D, int HB, bool F8>
KernelShape shape_t() {
  using C = U8Cfg<D, HB, U8Stages<D>::value, F8>;
  static std::atomic<int> occ{-1};
  int n = occ.load(std::memory_order_relaxed);
  if (n < 0) {
    auto kern = decode_u8_kernel<D, HB, U8Stages<D>::value, F8, false>;
    n = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, C::kThreads, C::kSmemBytes) != cudaSuccess) {
      n = 0;
      cudaGetLastError();  // the failed query's own error, not left for the next launch check
    }
    occ.store(n, std::memory_order_relaxed);
  }
  return {C::kThreads, C::kSmemBytes, 16 * HB, n};
}

// ---------------------------------------------------------------------------
// Paged uint8 pools of 16- or 32-token pages, G <= 16: one block per
// (sequence, group of HG kv heads, split). In the pool [num_pages, h_kv, PS,
// D] the slices of HG consecutive kv heads of one page are one contiguous run
// of HG x PS x D bytes (and HG x PS x 8 bytes of scale / zero pairs), which
// one TMA box fetches; a single head's page would be a 2 or 4 KB run.
// Block = HG consumer warps + 1 producer warp; a stage holds 32 tokens (two
// 16-token pages or one 32-token page) of the HG heads. Consumer warp w owns
// kv head jg HG + w and its G <= 16 query heads, runs its own online softmax
// over the block's token range and writes its rows itself.
template <int D, int HG, int PS, int STAGES, bool F8 = false>
struct U8HeadsCfg {
  static constexpr int kTokens = 32;                 // per stage
  static constexpr int kRows = PS < 32 ? PS : 32;    // rows of one box
  static constexpr int kBoxes = kTokens / kRows;     // pages per stage
  static constexpr int kThreads = 32 * (HG + 1);
  static constexpr int kCodeBytes = HG * kTokens * D;
  static constexpr int kSzBytes = F8 ? 0 : HG * kTokens * 8;
  static constexpr int kStageBytes = 2 * kCodeBytes + 2 * kSzBytes;
  static constexpr int kSmemBytes = STAGES * kStageBytes + 2 * STAGES * 8 + 1024;
  // byte strides in a stage: between heads, and between 16-row blocks of a head
  static constexpr uint32_t kHeadCode = kRows * D;
  static constexpr uint32_t kBlockCode = PS == 16 ? HG * 16 * D : 16 * D;
  static constexpr uint32_t kHeadSz = kRows * 8;
  static constexpr uint32_t kBlockSz = PS == 16 ? HG * 128 : 128;
  static_assert(PS == 16 || PS == 32, "16- or 32-token pages");
  static_assert(kStageBytes % 1024 == 0, "stages stay 1 KB aligned (swizzle atoms)");
};

template <int D, int HG, int PS, int STAGES, bool F8>
__global__ void __launch_bounds__(U8HeadsCfg<D, HG, PS, STAGES, F8>::kThreads, HG <= 4 ? 2 : 1)
    decode_u8_heads_kernel(const __grid_constant__ CUtensorMap tm_kc, const __grid_constant__ CUtensorMap tm_vc,
                           const __grid_constant__ CUtensorMap tm_ks, const __grid_constant__ CUtensorMap tm_vs,
                           const DecodeParams p) {
  using C = U8HeadsCfg<D, HG, PS, STAGES, F8>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * C::kStageBytes);
  uint64_t* empty = full + STAGES;
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.num_splits;
  const int n_groups = p.h_kv / HG;
  int cta = blockIdx.x;
  const int split = cta % S;
  cta /= S;
  const int jg = cta % n_groups;
  const int b = cta / n_groups;
  const int G = p.group;

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), HG);
    }
    fence_mbar_init();
  }
  __syncthreads();
  // the combine (or the next step) may be scheduled now; it waits for this
  // whole grid before it reads anything this grid writes
  grid_dependents_launch();
  if (!p.early) grid_dependency_wait();
  long long limit = static_cast<long long>(p.max_pages) * PS;
  if (limit > p.max_seq_len) limit = p.max_seq_len;
  int L = p.seq_lens[b];
  if (L < 1 || L > limit) {
    if (threadIdx.x == 0 && split == 0 && jg == 0) atomicOr(p.err, static_cast<int>(MQA_DEVERR_SEQ_LEN));
    L = L < 0 ? 0 : static_cast<int>(L > limit ? limit : L);
  }
  const int t_lo = p.window > 0 ? max(0, L - p.window) : 0;
  const int t_base = (t_lo / kTile) * kTile;
  const int t_begin = t_base + split * p.chunk;
  const int t_end = min(L, t_begin + p.chunk);
  const int n_steps = t_end > t_begin ? (t_end - t_begin + C::kTokens - 1) / C::kTokens : 0;

  if (warp == HG) {
    // ------------------------------------------------------------ producer
    const int32_t* trow = p.block_table + static_cast<long long>(b) * p.max_pages;
    const int n_pages_seq = (L + PS - 1) / PS;
    int wbase = t_begin / PS;
    int wcur = (wbase + lane < n_pages_seq) ? __ldg(trow + wbase + lane) : -1;
    int wnxt = (wbase + 32 + lane < n_pages_seq) ? __ldg(trow + wbase + 32 + lane) : -1;
    int issued = 0;
    bool waited = !p.early;
    // the fused append of the group's HG rows (no append launch precedes this
    // one), by this warp: once the first stages are in flight, or before the
    // stage that holds the rows if that comes sooner
    const int apos = p.fuse_append ? p.pos[b] : 0;
    bool appended = !(p.fuse_append && split == append_split(apos - t_base, p.chunk, S));
    auto append = [&]() {
      for (int h = 0; h < HG; ++h) {
        const int jj = jg * HG + h;
        append_row_q<D, F8>(p, b, jj, apos, cache_row(p, b, jj, apos, lane == 0 && h == 0), lane);
      }
      appended = true;
    };
    for (int it = 0; it < n_steps; ++it) {
      const int stage = it % STAGES;
      if (!appended && it == STAGES) append();
      if (it >= STAGES) {
        if (!mbar_wait(smem_u32(&empty[stage]), ((it / STAGES) + 1) & 1, p.wait_ns)) {
          if (lane == 0) {
            s_abort = 1;
            atomicOr(p.err, static_cast<int>(MQA_DEVERR_TIMEOUT));
          }
          break;
        }
      }
      if (*reinterpret_cast<volatile int*>(&s_abort)) break;
      const int t0 = t_begin + it * C::kTokens;
      if (!waited && L - 1 < t0 + C::kTokens) {  // this stage holds the appended token
        grid_dependency_wait();
        waited = true;
      }
      if (!appended && apos < t0 + C::kTokens) append();  // this stage holds the rows this block appends
      int pg[C::kBoxes];
#pragma unroll
      for (int k = 0; k < C::kBoxes; ++k) {
        int lp = (t0 + k * C::kRows) / PS;
        if (t0 + (k + 1) * C::kRows <= t_lo) lp = t_lo / PS;  // wholly before the window: any live page
        if (lp >= n_pages_seq) lp = n_pages_seq - 1;
        while (lp >= wbase + 32) {
          wbase += 32;
          wcur = wnxt;
          wnxt = (wbase + 32 + lane < n_pages_seq) ? __ldg(trow + wbase + 32 + lane) : -1;
        }
        pg[k] = __shfl_sync(0xffffffffu, wcur, lp - wbase);
        if (pg[k] < 0 || pg[k] >= p.num_pages) {
          if (lane == 0) atomicOr(p.err, static_cast<int>(MQA_DEVERR_PAGE_RANGE));
          pg[k] = p.num_pages;  // past the pool: TMA's zero fill
        }
      }
      if (lane == 0) {
        const uint32_t base = smem_u32(smem + stage * C::kStageBytes);
        const uint32_t kc = base, vc = base + C::kCodeBytes;
        const uint32_t ksd = base + 2 * C::kCodeBytes, vsd = ksd + C::kSzBytes;
        const uint32_t fb = smem_u32(&full[stage]);
        mbar_arrive_expect_tx(fb, C::kStageBytes);
        // t0 is a multiple of 32: every box starts at row 0 of its page
#pragma unroll
        for (int k = 0; k < C::kBoxes; ++k) {
          tma_load_4d(kc + k * HG * C::kRows * D, &tm_kc, 0, 0, jg * HG, pg[k], fb);
          tma_load_4d(vc + k * HG * C::kRows * D, &tm_vc, 0, 0, jg * HG, pg[k], fb);
          if constexpr (!F8) {
            tma_load_3d(ksd + k * HG * C::kRows * 8, &tm_ks, 0, jg * HG, pg[k], fb);
            tma_load_3d(vsd + k * HG * C::kRows * 8, &tm_vs, 0, jg * HG, pg[k], fb);
          }
        }
      }
      __syncwarp();
      issued = it + 1;
    }
    if (!appended) append();  // rows this block never reads
    // every copy this warp issued lands before the block can exit: after a
    // timeout the consumers may have stopped waiting for them
    for (int it = (issued > STAGES ? issued - STAGES : 0); it < issued; ++it)
      (void)mbar_wait(smem_u32(&full[it % STAGES]), (it / STAGES) & 1, kWaitLimitNs);
    return;
  }

  // -------------------------------------------------------------- consumers
  const int j = jg * HG + warp;  // this warp's kv head
  WarpAttnU8<D, F8> wa;
  if (p.rope_q) {
    // fused step: q_new rotated here (its loads issued before the cos / sin
    // table is formed)
    __shared__ float s_cs[D];
    const long long qoff = (static_cast<long long>(b) * p.h_q + j * G) * D;
    uint2 qraw[D / 16][2];
    WarpAttnU8<D, F8>::load_q(static_cast<const __nv_bfloat16*>(p.q_new) + qoff, G, lane, qraw);
    rope_table<D>(s_cs, p, p.pos[b], threadIdx.x, 2, HG * 32);
    wa.init_rope(qraw, G, s_cs, p.scale_log2, lane, (p.fuse_append && split == 0) ? p.q_rot_out + qoff : nullptr);
  } else {
    if (p.early) grid_dependency_wait();  // q_rot is written by the append kernel
    wa.init(p.q_rot + (static_cast<long long>(b) * p.h_q + j * G) * D, G, p.scale_log2, lane);
  }
  bool ok = true;
  for (int it = 0; it < n_steps; ++it) {
    const int stage = it % STAGES;
    if (!mbar_wait(smem_u32(&full[stage]), (it / STAGES) & 1, p.wait_ns)) {
      if (lane == 0) {
        s_abort = 1;
        atomicOr(p.err, static_cast<int>(MQA_DEVERR_TIMEOUT));
      }
      ok = false;
      break;
    }
    const uint32_t st = smem_u32(smem + stage * C::kStageBytes);
    const int tt = t_begin + it * C::kTokens;
    const int lo = max(0, t_lo - tt), hi = min(C::kTokens, t_end - tt);
    if (lo < hi)
      wa.template step<C::kBlockCode, C::kBlockSz>(
          st + warp * C::kHeadCode, st + C::kCodeBytes + warp * C::kHeadCode, st + 2 * C::kCodeBytes + warp * C::kHeadSz,
          st + 2 * C::kCodeBytes + C::kSzBytes + warp * C::kHeadSz, 0, lo, hi, lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[stage]));
  }
  wa.finish();
  if (!F8 && __any_sync(0xffffffffu, wa.vmax > kMaxVScale) && lane == 0)
    atomicOr(p.err, static_cast<int>(MQA_DEVERR_U8_SCALE));
  if (!ok) return;

  // ---- rows g, g + 8: O / l (or the split's partial) and the log-sum-exp.
  // Lane (g, c) holds head dims (2c + e) D/8 .. (2c + e) D/8 + D/8 - 1 of each
  // row in o[0 .. D/8)[e] (row g) and o[..][2 + e] (row g + 8).
  const int g = lane >> 2, c = lane & 3;
  const bool split_out = S > 1;
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int row = g + 8 * hr;
    if (row >= G) continue;
    const float l = hr ? wa.l1 : wa.l0, m = hr ? wa.m1 : wa.m0;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float lse = l > 0.f ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
    const long long grow = static_cast<long long>(b) * p.h_q + j * G + row;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int d0 = (2 * c + e) * (D / 8);
      if (split_out) {
        float* dst = p.o_part + (grow * S + split) * D + d0;
#pragma unroll
        for (int q4 = 0; q4 < D / 32; ++q4)
          *reinterpret_cast<float4*>(dst + 4 * q4) =
              make_float4(wa.o[4 * q4][2 * hr + e] * inv, wa.o[4 * q4 + 1][2 * hr + e] * inv,
                          wa.o[4 * q4 + 2][2 * hr + e] * inv, wa.o[4 * q4 + 3][2 * hr + e] * inv);
      } else if (p.out_dtype == kDtypeBf16) {
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + grow * D + d0;
#pragma unroll
        for (int q8 = 0; q8 < D / 64; ++q8) {
          uint4 v;
          v.x = pack_bf16x2(wa.o[8 * q8][2 * hr + e] * inv, wa.o[8 * q8 + 1][2 * hr + e] * inv);
          v.y = pack_bf16x2(wa.o[8 * q8 + 2][2 * hr + e] * inv, wa.o[8 * q8 + 3][2 * hr + e] * inv);
          v.z = pack_bf16x2(wa.o[8 * q8 + 4][2 * hr + e] * inv, wa.o[8 * q8 + 5][2 * hr + e] * inv);
          v.w = pack_bf16x2(wa.o[8 * q8 + 6][2 * hr + e] * inv, wa.o[8 * q8 + 7][2 * hr + e] * inv);
          *reinterpret_cast<uint4*>(dst + 8 * q8) = v;
        }
      } else {
        float* dst = static_cast<float*>(p.out) + grow * D + d0;
#pragma unroll
        for (int q4 = 0; q4 < D / 32; ++q4)
          *reinterpret_cast<float4*>(dst + 4 * q4) =
              make_float4(wa.o[4 * q4][2 * hr + e] * inv, wa.o[4 * q4 + 1][2 * hr + e] * inv,
                          wa.o[4 * q4 + 2][2 * hr + e] * inv, wa.o[4 * q4 + 3][2 * hr + e] * inv);
      }
    }
    if (c == 0) {
      if (split_out)
        p.lse_part[grow * S + split] = lse;
      else if (p.lse_out != nullptr)
        p.lse_out[grow] = lse;
    }
  }
}

template <int D, int HG, int PS, bool F8>
cudaError_t launch_u8_heads_t(const DecodeParams& p, const CUtensorMap* maps, cudaStream_t stream) {
  constexpr int ST = 3;
  using C = U8HeadsCfg<D, HG, PS, ST, F8>;
  auto kern = decode_u8_heads_kernel<D, HG, PS, ST, F8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.batch) * (p.h_kv / HG) * p.num_splits);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], maps[3], p);
}

int u8_hb(int group) { return group > 16 ? 2 : 1; }

}  // namespace

template <bool F8>
KernelShape u8_shape(int head_dim, int group) {
  const bool two = u8_hb(group) == 2;
  if (head_dim == 128) return two ? shape_t<128, 2, F8>() : shape_t<128, 1, F8>();
  return two ? shape_t<64, 2, F8>() : shape_t<64, 1, F8>();
}

KernelShape decode_u8_shape(int head_dim, int group, bool f8) {
  return f8 ? u8_shape<true>(head_dim, group) : u8_shape<false>(head_dim, group);
}

int decode_u8_heads_group(const DecodeParams& p) {
  if (!p.paged || (p.page_size != 16 && p.page_size != 32) || p.group > 16 || p.n_new > 1) return 0;
  if (p.h_kv % 4 == 0) return 4;
  if (p.h_kv % 2 == 0) return 2;
  return 0;
}

template <bool F8>
cudaError_t u8_heads(const DecodeParams& p, int hg, const CUtensorMap* maps, cudaStream_t stream) {
  if (p.head_dim == 128) {
    if (p.page_size == 16) return hg == 4 ? launch_u8_heads_t<128, 4, 16, F8>(p, maps, stream)
                                          : launch_u8_heads_t<128, 2, 16, F8>(p, maps, stream);
    return hg == 4 ? launch_u8_heads_t<128, 4, 32, F8>(p, maps, stream)
                   : launch_u8_heads_t<128, 2, 32, F8>(p, maps, stream);
  }
  if (p.page_size == 16) return hg == 4 ? launch_u8_heads_t<64, 4, 16, F8>(p, maps, stream)
                                        : launch_u8_heads_t<64, 2, 16, F8>(p, maps, stream);
  return hg == 4 ? launch_u8_heads_t<64, 4, 32, F8>(p, maps, stream) : launch_u8_heads_t<64, 2, 32, F8>(p, maps, stream);
}

template <bool F8, bool MULTI>
cudaError_t u8_slices_m(const DecodeParams& p, const CUtensorMap* maps, cudaStream_t stream) {
  const bool two = u8_hb(p.group * (MULTI ? p.n_new : 1)) == 2;
  if (p.head_dim == 128)
    return two ? launch_u8_t<128, 2, F8, MULTI>(p, maps, stream) : launch_u8_t<128, 1, F8, MULTI>(p, maps, stream);
  return two ? launch_u8_t<64, 2, F8, MULTI>(p, maps, stream) : launch_u8_t<64, 1, F8, MULTI>(p, maps, stream);
}

template <bool F8>
cudaError_t u8_slices(const DecodeParams& p, const CUtensorMap* maps, cudaStream_t stream) {
  return p.n_new > 1 ? u8_slices_m<F8, true>(p, maps, stream) : u8_slices_m<F8, false>(p, maps, stream);
}

cudaError_t launch_decode_u8_heads(const DecodeParams& p, int hg, const CUtensorMap* maps, cudaStream_t stream) {
  return p.cache_dtype == kDtypeF8 ? u8_heads<true>(p, hg, maps, stream) : u8_heads<false>(p, hg, maps, stream);
}

cudaError_t launch_decode_u8(const DecodeParams& p, const CUtensorMap* maps, cudaStream_t stream) {
  return p.cache_dtype == kDtypeF8 ? u8_slices<true>(p, maps, stream) : u8_slices<false>(p, maps, stream);
}

}  // namespace mqa
