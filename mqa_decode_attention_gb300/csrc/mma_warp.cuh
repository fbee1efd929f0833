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
#include "rope.cuh"

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

// Element offset of the cache row (sequence b, kv head j, token pos), or -1
// (with the matching error bit when `report`) if pos or its page is out of
// range. Same checks as the append kernel.
__device__ __forceinline__ long long cache_row(const DecodeParams& p, int b, int j, int pos, bool report) {
  if (!p.paged) {
    if (pos < 0 || pos >= p.capacity) {
      if (report) atomicOr(p.err, 0x1);  // MQA_DEVERR_POS_RANGE
      return -1;
    }
    return ((static_cast<long long>(b) * p.h_kv + j) * p.capacity + pos) * p.head_dim;
  }
  const int lp = pos >= 0 ? pos / p.page_size : -1;
  if (pos < 0 || lp >= p.max_pages) {
    if (report) atomicOr(p.err, 0x1);  // MQA_DEVERR_POS_RANGE
    return -1;
  }
  const int page = p.block_table[static_cast<long long>(b) * p.max_pages + lp];
  if (page < 0 || page >= p.num_pages) {
    if (report) atomicOr(p.err, 0x2);  // MQA_DEVERR_PAGE_RANGE
    return -1;
  }
  return ((static_cast<long long>(page) * p.h_kv + j) * p.page_size + pos % p.page_size) * p.head_dim;
}

// Split whose block performs the fused append of sequence b's new token:
// the one whose token range holds pos, else split 0.
__device__ __forceinline__ int append_split(int pos, int chunk, int splits) {
  return (pos >= 0 && pos / chunk < splits) ? pos / chunk : 0;
}

// Fill cs[0 .. D/2) with cos and cs[D/2 .. D) with sin of pos * theta_i for
// rotating the query in fp32: the angle is formed and reduced in fp64, then
// its fp32 sine/cosine taken. Called by all `count` consumer threads (named
// barrier `bar`); the first D/2 compute.
template <int D>
__device__ __forceinline__ void rope_table(float* cs, const DecodeParams& p, int pos, int tid, int bar, int count) {
  if (tid < D / 2) {
    const double ang = reduce_two_pi(static_cast<double>(pos) * p.theta[tid]);
    float sf, cf;
    sincosf(static_cast<float>(ang), &sf, &cf);
    cs[tid] = cf;
    cs[D / 2 + tid] = sf;
  }
  named_bar_sync(bar, count);
}

// The fused append of sequence b's new token for kv heads j0 .. j0 + H - 1,
// by one whole warp (lane i owns rotation pairs i, i + 32, ...), with the
// append kernel's result: k turned by the angle formed and reduced in fp64
// and rounded once to bf16 (rope_k_bf16, equal to the fp64 rotation), v
// copied. It comes in three parts so that its memory latencies overlap the
// producer's other work: load() issues every global read, write() turns k and
// stores both rows, publish() fences them for TMA loads (async proxy) that
// this warp issues afterwards.
template <int D, int H>
struct AppendRows {
  static constexpr int kPer = D / 64;  // rotation pairs per lane
  uint32_t k[H][kPer], v[H][kPer];
  double theta[kPer];
  long long row[H];

  // tok / n_tok: the new token's index among the sequence's n_tok new tokens
  // (k_new / v_new [B, n_tok, H_kv, D])
  __device__ __forceinline__ void load(const DecodeParams& p, int b, int j0, int pos, int lane, int tok = 0,
                                       int n_tok = 1) {
#pragma unroll
    for (int i = 0; i < kPer; ++i) theta[i] = p.theta[lane + 32 * i];
#pragma unroll
    for (int h = 0; h < H; ++h) {
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const long long src =
            ((static_cast<long long>(b) * n_tok + tok) * p.h_kv + j0 + h) * D + 2 * (lane + 32 * i);
        k[h][i] = *reinterpret_cast<const uint32_t*>(static_cast<const __nv_bfloat16*>(p.k_new) + src);
        v[h][i] = *reinterpret_cast<const uint32_t*>(static_cast<const __nv_bfloat16*>(p.v_new) + src);
      }
    }
#pragma unroll
    for (int h = 0; h < H; ++h) row[h] = cache_row(p, b, j0 + h, pos, lane == 0 && h == 0);
  }

  __device__ __forceinline__ void write(const DecodeParams& p, int pos, int lane) const {
    double ang[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) ang[i] = reduce_two_pi(static_cast<double>(pos) * theta[i]);
#pragma unroll
    for (int h = 0; h < H; ++h) {
      if (row[h] < 0) continue;  // the same for every lane
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const long long e = row[h] + 2 * (lane + 32 * i);
        __nv_bfloat16* kc = static_cast<__nv_bfloat16*>(const_cast<void*>(p.k_cache)) + e;
        __nv_bfloat16* vc = static_cast<__nv_bfloat16*>(const_cast<void*>(p.v_cache)) + e;
        *reinterpret_cast<__nv_bfloat162*>(kc) = rope_k_bf16(bf16lo_to_f32(k[h][i]), bf16hi_to_f32(k[h][i]), ang[i]);
        *reinterpret_cast<uint32_t*>(vc) = v[h][i];
      }
    }
  }

  __device__ __forceinline__ static void publish() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __syncwarp();
  }
};

template <int D>
struct WarpAttn {
  uint32_t qa[D / 16][4];  // Q as the A operand, pre-scaled into the log2 domain
  float o[D / 8][4];       // O accumulators: rows r0 (regs 0,1) and r0 + 8 (regs 2,3)
  float m0, m1, l0, l1;    // running max / (lane-partial) sum of rows r0, r0 + 8

  // q points at row 0 of this warp's 16 query heads ([16][D] fp32, row stride D);
  // rows >= rows_valid are padding and read as zero.
  __device__ __forceinline__ void init(const float* q, int rows_valid, float scale_log2, int lane) {
    const int r0 = lane >> 2;
    init2(r0 < rows_valid ? q + r0 * D : nullptr, r0 + 8 < rows_valid ? q + (r0 + 8) * D : nullptr, scale_log2,
          lane);
  }

  // The same with the lane's two rows given directly: q0 is row r0 = lane / 4
  // of the warp's 16, q1 row r0 + 8 (each fp32 [D], or null for padding).
  __device__ __forceinline__ void init2(const float* q0, const float* q1, float scale_log2, int lane) {
    const int c2 = (lane & 3) * 2;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
      for (int part = 0; part < 4; ++part) {
        const float* q = (part & 1) ? q1 : q0;
        const int col = ks * 16 + c2 + ((part & 2) ? 8 : 0);
        float2 v = make_float2(0.f, 0.f);
        if (q != nullptr) v = *reinterpret_cast<const float2*>(q + col);
        qa[ks][part] = pack_bf16x2(v.x * scale_log2, v.y * scale_log2);
      }
    }
#pragma unroll
    for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
  }

  // Rows [trow0, trow0 + 16) of the K / V tiles at shared addresses kb / vb;
  // only rows lo .. hi-1 of these 16 are real tokens (0 <= lo < hi <= 16).
  // vtile is the generic pointer of the V tile: the other rows may hold
  // anything (even NaN bit patterns) and are zeroed so that P = 0 contributes
  // exactly nothing. With PER_ROW, the query rows r0 and r0 + 8 of this lane
  // see only tokens [lo0, hi0) and [lo1, hi1) of the 16 (inside [lo, hi));
  // a row may then see none of them, and the softmax update stays finite.
  template <bool PER_ROW = false>
  __device__ __forceinline__ void step(uint32_t kb, uint32_t vb, unsigned char* vtile, int trow0, int lo, int hi,
                                       int lg_rpb, int lane, int lo0 = 0, int hi0 = 0, int lo1 = 0, int hi1 = 0) {
    if constexpr (!PER_ROW) {
      lo0 = lo1 = lo;
      hi0 = hi1 = hi;
    }
    const int c2 = (lane & 3) * 2;
    if (lo > 0 || hi < 16) {
      const int n_bad = 16 - (hi - lo);
      for (int idx = lane; idx < n_bad * (D / 8); idx += 32) {
        int r = idx / (D / 8);
        r = r < lo ? r : r + (hi - lo);  // rows [0, lo) then [hi, 16)
        const int c = idx % (D / 8);
        *reinterpret_cast<uint4*>(vtile + swz<D>(trow0 + r, c, lg_rpb)) = make_uint4(0u, 0u, 0u, 0u);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
    }
    // ---- S = Q K^T over 16 tokens (two n8 tiles); even and odd k-steps
    // accumulate separately so four independent MMA chains are in flight
    float s[2][4], s2[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
      s2[nt][0] = s2[nt][1] = s2[nt][2] = s2[nt][3] = 0.f;
    }
#pragma unroll
    for (int kk = 0; kk < D / 32; ++kk) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int row = trow0 + nt * 8 + (lane & 7);
        const int c = kk * 4 + (lane >> 3);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kb + swz<D>(row, c, lg_rpb), b0, b1, b2, b3);
        mma_bf16_16816(s[nt], qa[2 * kk], b0, b1);
        mma_bf16_16816(s2[nt], qa[2 * kk + 1], b2, b3);
      }
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) s[nt][e] += s2[nt][e];
    }
    // ---- mask, online softmax (rows r0 and r0 + 8)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int r = nt * 8 + c2 + e;
        if (r < lo0 || r >= hi0) s[nt][e] = -INFINITY;
        if (r < lo1 || r >= hi1) s[nt][2 + e] = -INFINITY;
      }
    }
    float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
    float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    // Without PER_ROW, mn is finite: at least one of the 16 tokens is valid
    // (lo < hi). With it, a row that has seen no token yet keeps -inf, and
    // its exponentials use 0 in place of the max (2^-inf = 0, no inf - inf).
    const bool moved = (mn0 != m0) || (mn1 != m1);
    const float e0 = (PER_ROW && mn0 == -INFINITY) ? 0.f : mn0;
    const float e1 = (PER_ROW && mn1 == -INFINITY) ? 0.f : mn1;
    const float a0 = fast_exp2(m0 - e0), a1 = fast_exp2(m1 - e1);
    m0 = mn0;
    m1 = mn1;
    float pr[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      pr[nt][0] = fast_exp2(s[nt][0] - e0);
      pr[nt][1] = fast_exp2(s[nt][1] - e0);
      pr[nt][2] = fast_exp2(s[nt][2] - e1);
      pr[nt][3] = fast_exp2(s[nt][3] - e1);
    }
    l0 = l0 * a0 + (pr[0][0] + pr[0][1] + pr[1][0] + pr[1][1]);
    l1 = l1 * a1 + (pr[0][2] + pr[0][3] + pr[1][2] + pr[1][3]);
    // rescale the accumulators only when some row's running max moved
    if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        o[n][0] *= a0;
        o[n][1] *= a0;
        o[n][2] *= a1;
        o[n][3] *= a1;
      }
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

  // Load this lane's fragment of the raw bf16 query q_new (q points at row 0
  // of the warp's 16 query heads, [16][D], rows >= rows_valid read as zero).
  // Kept apart from init_rope so the loads are in flight while the cos / sin
  // table is formed.
  __device__ __forceinline__ static void load_q(const __nv_bfloat16* q, int rows_valid, int lane,
                                                uint32_t (&raw)[D / 16][4]) {
    const int r0 = lane >> 2, c2 = (lane & 3) * 2;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
      for (int part = 0; part < 4; ++part) {
        const int row = r0 + ((part & 1) ? 8 : 0);
        const int col = ks * 16 + c2 + ((part & 2) ? 8 : 0);
        raw[ks][part] = row < rows_valid ? *reinterpret_cast<const uint32_t*>(q + row * D + col) : 0u;
      }
    }
  }

  // Same as init, but from the raw bf16 query loaded by load_q, rotated first:
  // pair i of a row turns by the angle whose fp32 cosine / sine are cs[i] /
  // cs[D/2 + i], as the append kernel does for q_rot (written to q_rot_out, a
  // [16][D] fp32 block like q, unless null).
  __device__ __forceinline__ void init_rope(const uint32_t (&raw)[D / 16][4], int rows_valid, const float* cs,
                                            float scale_log2, int lane, float* q_rot_out) {
    const int r0 = lane >> 2, c2 = (lane & 3) * 2;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
      for (int part = 0; part < 4; ++part) {
        const int row = r0 + ((part & 1) ? 8 : 0);
        const int col = ks * 16 + c2 + ((part & 2) ? 8 : 0);
        float2 v = make_float2(0.f, 0.f);
        if (row < rows_valid) {
          const float x = bf16lo_to_f32(raw[ks][part]), y = bf16hi_to_f32(raw[ks][part]);
          const float c = cs[col >> 1], s = cs[D / 2 + (col >> 1)];
          v = make_float2(x * c - y * s, x * s + y * c);
          if (q_rot_out != nullptr) *reinterpret_cast<float2*>(q_rot_out + row * D + col) = v;
        }
        qa[ks][part] = pack_bf16x2(v.x * scale_log2, v.y * scale_log2);
      }
    }
#pragma unroll
    for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
  }

  // Two rows of raw bf16 q_new for init2_rope: q0 is row r0 = lane / 4 of the
  // warp's 16, q1 row r0 + 8 (each bf16 [D], or null for padding); this
  // lane's columns of both.
  __device__ __forceinline__ static void load_q2(const __nv_bfloat16* q0, const __nv_bfloat16* q1, int lane,
                                                 uint32_t (&raw)[D / 16][4]) {
    const int c2 = (lane & 3) * 2;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
      for (int part = 0; part < 4; ++part) {
        const __nv_bfloat16* q = (part & 1) ? q1 : q0;
        const int col = ks * 16 + c2 + ((part & 2) ? 8 : 0);
        raw[ks][part] = q != nullptr ? *reinterpret_cast<const uint32_t*>(q + col) : 0u;
      }
    }
  }

  // Same as init2, from the raw rows of load_q2 rotated first, row r0 by the
  // fp32 cos / sin table cs0 (cs[i], cs[D/2 + i] for pair i) and row r0 + 8 by
  // cs1 (rows of different new tokens turn by different positions); the
  // rotated rows also go to out0 / out1 (fp32 [D]) unless null.
  __device__ __forceinline__ void init2_rope(const uint32_t (&raw)[D / 16][4], bool valid0, bool valid1,
                                             const float* cs0, const float* cs1, float scale_log2, int lane,
                                             float* out0, float* out1) {
    const int c2 = (lane & 3) * 2;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
      for (int part = 0; part < 4; ++part) {
        const bool hi = (part & 1) != 0;
        const int col = ks * 16 + c2 + ((part & 2) ? 8 : 0);
        const float* cs = hi ? cs1 : cs0;
        float* out = hi ? out1 : out0;
        float2 v = make_float2(0.f, 0.f);
        if (hi ? valid1 : valid0) {
          const float x = bf16lo_to_f32(raw[ks][part]), y = bf16hi_to_f32(raw[ks][part]);
          const float c = cs[col >> 1], sn = cs[D / 2 + (col >> 1)];
          v = make_float2(x * c - y * sn, x * sn + y * c);
          if (out != nullptr) *reinterpret_cast<float2*>(out + col) = v;
        }
        qa[ks][part] = pack_bf16x2(v.x * scale_log2, v.y * scale_log2);
      }
    }
#pragma unroll
    for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
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
