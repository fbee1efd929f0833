// One warp's share of decode attention on bf16 tensor cores: up to 16 query
// heads of one kv head (the rows of the MMA A operand) against 16 tokens at a
// time, with an online softmax in registers.
//
//   S = Q K^T    m16 x n8 x k16 MMAs over head_dim (two n8 tiles of tokens)
//   running max / sum per row ("Arsitektur Inferensi LLM", section 5)
//   O += P V     P taken from the S fragments, rounded to bf16
//
// K and V rows sit in shared memory in the 128-byte-swizzled layout TMA
// writes (see swz).
#pragma once

#include <cuda_bf16.h>

#include "launch.h"
#include "ptx.cuh"

namespace mqa {

// Shared-memory byte offset of 16-byte chunk c (0 .. D/8-1) of row r. Rows are
// stored as blocks of `1 << lg_rpb` rows (one TMA box: a page, or a whole
// 64-row tile); inside a block each 64-column half is a span of 128-byte rows,
// and TMA's 128-byte swizzle put chunk (c mod 8) of row r at position
// (c mod 8) xor (r mod 8). Blocks and spans start on 1 KB boundaries, so the 8
// rows an ldmatrix reads land in 8 distinct bank groups.
template <int D>
__device__ __forceinline__ uint32_t swz(int r, int c, int lg_rpb) {
  const int blk = r >> lg_rpb, rin = r & ((1 << lg_rpb) - 1);
  return ((blk * (D / 64) + (c >> 3)) << (lg_rpb + 7)) + rin * 128 + (((c & 7) ^ (r & 7)) << 4);
}

template <int D>
struct WarpAttn {
  uint32_t qa[D / 16][4];  // Q as the A operand, pre-scaled into the log2 domain
  float o[D / 8][4];       // O accumulators: rows r0 (regs 0,1) and r0 + 8 (regs 2,3)
  float m0, m1, l0, l1;    // running max / (lane-partial) sum of rows r0, r0 + 8

  // q points at row 0 of this warp's 16 query heads ([16][D] fp32, row stride D);
  // rows >= rows_valid are padding and read as zero.
  __device__ __forceinline__ void init(const float* q, int rows_valid, float scale_log2, int lane) {
    const int r0 = lane >> 2, c2 = (lane & 3) * 2;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
      for (int part = 0; part < 4; ++part) {
        const int row = r0 + ((part & 1) ? 8 : 0);
        const int col = ks * 16 + c2 + ((part & 2) ? 8 : 0);
        float2 v = make_float2(0.f, 0.f);
        if (row < rows_valid) v = *reinterpret_cast<const float2*>(q + row * D + col);
        qa[ks][part] = pack_bf16x2(v.x * scale_log2, v.y * scale_log2);
      }
    }
#pragma unroll
    for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
  }

  // Rows [trow0, trow0 + 16) of the K / V tiles at shared addresses kb / vb;
  // only the first n_valid of them are real tokens (1 <= n_valid). vtile is the
  // generic pointer of the V tile: rows past n_valid may hold anything (even
  // NaN bit patterns) and are zeroed so that P = 0 contributes exactly nothing.
  __device__ __forceinline__ void step(uint32_t kb, uint32_t vb, unsigned char* vtile, int trow0, int n_valid,
                                       int lg_rpb, int lane) {
    const int c2 = (lane & 3) * 2;
    if (n_valid < 16) {
      for (int idx = lane; idx < (16 - n_valid) * (D / 8); idx += 32) {
        const int r = trow0 + n_valid + idx / (D / 8);
        const int c = idx % (D / 8);
        *reinterpret_cast<uint4*>(vtile + swz<D>(r, c, lg_rpb)) = make_uint4(0u, 0u, 0u, 0u);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
    }
    // ---- S = Q K^T over 16 tokens (two n8 tiles)
    float s[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 32; ++kk) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int row = trow0 + nt * 8 + (lane & 7);
        const int c = kk * 4 + (lane >> 3);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kb + swz<D>(row, c, lg_rpb), b0, b1, b2, b3);
        mma_bf16_16816(s[nt], qa[2 * kk], b0, b1);
        mma_bf16_16816(s[nt], qa[2 * kk + 1], b2, b3);
      }
    }
    // ---- mask, online softmax (rows r0 and r0 + 8)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        if (nt * 8 + c2 + e >= n_valid) {
          s[nt][e] = -INFINITY;
          s[nt][2 + e] = -INFINITY;
        }
      }
    }
    float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
    float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    // mn is finite: at least one of the 16 tokens is valid
    const float a0 = exp2f(m0 - mn0), a1 = exp2f(m1 - mn1);
    m0 = mn0;
    m1 = mn1;
    float pr[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      pr[nt][0] = exp2f(s[nt][0] - mn0);
      pr[nt][1] = exp2f(s[nt][1] - mn0);
      pr[nt][2] = exp2f(s[nt][2] - mn1);
      pr[nt][3] = exp2f(s[nt][3] - mn1);
    }
    l0 = l0 * a0 + (pr[0][0] + pr[0][1] + pr[1][0] + pr[1][1]);
    l1 = l1 * a1 + (pr[0][2] + pr[0][3] + pr[1][2] + pr[1][3]);
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      o[n][0] *= a0;
      o[n][1] *= a0;
      o[n][2] *= a1;
      o[n][3] *= a1;
    }
    // ---- O += P V
    uint32_t pa[4];
    pa[0] = pack_bf16x2(pr[0][0], pr[0][1]);
    pa[1] = pack_bf16x2(pr[0][2], pr[0][3]);
    pa[2] = pack_bf16x2(pr[1][0], pr[1][1]);
    pa[3] = pack_bf16x2(pr[1][2], pr[1][3]);
#pragma unroll
    for (int dn = 0; dn < D / 16; ++dn) {
      const int row = trow0 + ((lane >> 3) & 1) * 8 + (lane & 7);
      const int c = dn * 2 + (lane >> 4);
      uint32_t v0, v1, v2, v3;
      ldsm_x4_trans(vb + swz<D>(row, c, lg_rpb), v0, v1, v2, v3);
      mma_bf16_16816(o[2 * dn], pa, v0, v1);
      mma_bf16_16816(o[2 * dn + 1], pa, v2, v3);
    }
  }

  // Sum the lane-partial row sums over the 4 lanes that share a row.
  __device__ __forceinline__ void finish_sums() {
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  }
};

}  // namespace mqa
