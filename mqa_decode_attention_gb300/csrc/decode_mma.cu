// gqa_decode_attention on tensor cores, bf16 cache.
//
// Same result as the CUDA-core kernel, O_h = softmax(scale * q_h K_j^T) V_j
// for the query heads h of kv head j ("Grouped-query attention" page,
// equations for A_h and O_h), with an online softmax ("Arsitektur Inferensi
// LLM", section 5: running max and sum, no score matrix in HBM).
//
// The G query heads of a group are the rows of the MMA A operand (padded to
// 16 per head block), so one K/V tile in shared memory serves every head of
// the group:  S = Q K^T  (m16 x n8 x k16 steps over head_dim), then
// O += P V with P rounded to bf16 (the fp32 softmax state stays in registers).
//
// Block = 4 consumer warps per head block of 16 heads + 1 producer warp + 1
// warp for the fused append (idle in other launches). The
// producer streams 64-token K and V tiles with TMA tensor copies
// (cp.async.bulk.tensor, 128-byte swizzle, one mbarrier pair per stage);
// a paged cache is gathered page by page through the block table. Consumer
// warp w reads tokens [16 (w % 4), 16 (w % 4) + 16) of every tile with
// ldmatrix (the swizzle keeps the 8 rows of each 8x8 matrix in distinct
// banks), runs its own online softmax over its tokens, and the 4 warps of a
// head block merge once at the end.
#include <cuda_bf16.h>

#include "../../include/mqa_decode.h"
#include "launch.h"
#include "mma_warp.cuh"
#include "ptx.cuh"

#ifndef MQA_MMA_STAGES_D128
#define MQA_MMA_STAGES_D128 3
#endif
#ifndef MQA_MMA_STAGES_D64
#define MQA_MMA_STAGES_D64 4
#endif


namespace mqa {
namespace {

template <int D, int HB, int STAGES>
struct MmaCfg {
  static constexpr int kConsumerWarps = 4 * HB;
  static constexpr int kConsumerThreads = 32 * kConsumerWarps;
  static constexpr int kThreads = kConsumerThreads + 64;     // + producer warp + append warp
  // one head block: as many blocks per SM as their stages fit in shared
  // memory (two for d = 128, three for d = 64), so their registers must fit
  // the SM's 64 K as well
  static constexpr int kMinBlocks = HB == 1 ? (D == 128 ? 2 : 3) : 1;
  static constexpr int kHalfBytes = kTile * 128;             // 64 rows x 64 bf16 (one swizzle span)
  static constexpr int kTileBytes = (D / 64) * kHalfBytes;    // a K (or V) tile
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kMergeStride = D + 8;                  // floats per merged row
  static constexpr int kMergeBytes = kConsumerWarps * 16 * (kMergeStride + 2) * 4;
  static constexpr int kBodyBytes = (STAGES * kStageBytes > kMergeBytes) ? STAGES * kStageBytes : kMergeBytes;
  static constexpr int kSmemBytes = kBodyBytes + 2 * STAGES * 8 + 1024;  // + alignment slack
  // the fused multi-token step's cos / sin tables (one per new token), placed
  // after the barriers and requested only by that launch
  static constexpr int kMultiTableBytes = kMaxFusedNewTokens * D * 4;
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
};

// MULTI: n_new > 1 query tokens per sequence (the verification pass of
// speculative decoding): the rows of a kv head are (new token i, query head
// h) pairs, row = i G + h, and row i sees tokens [.., L - n + i] only.
template <int D, int HB, int STAGES, bool MULTI>
__global__ void __launch_bounds__(MmaCfg<D, HB, STAGES>::kThreads, MmaCfg<D, HB, STAGES>::kMinBlocks)
    decode_mma_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                      const DecodeParams p) {
  using C = MmaCfg<D, HB, STAGES>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBodyBytes);
  uint64_t* empty = full + STAGES;
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.num_splits;
  // head blocks of one (sequence, kv head, split) are adjacent, so blocks that
  // read the same K/V tiles run together and share them through L2
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
      mbar_init(smem_u32(&empty[s]), C::kConsumerWarps);
    }
    fence_mbar_init();
  }
  if (warp == C::kConsumerWarps && lane == 0) {
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
  }
  __syncthreads();
  // Unless the preceding launch is known to be the append kernel, wait for it
  // before reading anything. After the append kernel, the lengths, the block
  // table and every cached row except the new token's are already final, so
  // the producer streams them early and only the tile holding the new token
  // (and the consumers, which need q_rot) wait.
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
  // sliding window: tokens [t_lo, L) (t_lo of the first new token, the lowest);
  // splits start at t_lo rounded down to a tile
  const int t_lo = p.window > 0 ? max(0, L - nq + 1 - p.window) : 0;
  const int t_base = (t_lo / kTile) * kTile;
  const int t_begin = t_base + split * p.chunk;
  const int t_end = min(L, t_begin + p.chunk);
  const int n_tiles = t_end > t_begin ? (t_end - t_begin + kTile - 1) / kTile : 0;


  // the fused append (no append launch precedes this one): new token i
  // (at apos + i) is written by the head-block-0 block of the split whose
  // token range holds it (else split 0), so that no block reads a row that
  // another block writes; a_first is this block's first such row
  const int apos = p.fuse_append ? p.pos[b] : 0;
  int a_first = -1;
  if (p.fuse_append && hsb == 0) {
    for (int i = nq - 1; i >= 0; --i)
      if (split == append_split(apos + i - t_base, p.chunk, S)) a_first = i;
  }
  const bool awaits = a_first >= 0;
  if (warp == C::kConsumerWarps + 1) {
    // --------------------------------------------------------- append warp
    // writes the rows, fences them for the async proxy and releases the
    // producer, which waits (named barrier 3) only before the first tile
    // holding one of them
    if (awaits) {
      for (int i = a_first; i < nq; ++i) {
        if (split != append_split(apos + i - t_base, p.chunk, S)) continue;
        AppendRows<D, 1> ar;
        ar.load(p, b, j, apos + i, lane, i, nq);
        ar.write(p, apos + i, lane);
      }
      AppendRows<D, 1>::publish();
      named_bar_arrive(3, 64);
    }
    return;
  }
  if (warp == C::kConsumerWarps) {
    // ------------------------------------------------------------ producer
    const int ps = p.page_size;
    const int rpc = ps < kTile ? ps : kTile;  // tile rows per paged copy
    const int32_t* trow = p.block_table + static_cast<long long>(b) * p.max_pages;
    const int n_pages_seq = p.paged ? (L + ps - 1) / ps : 0;
    int wbase = p.paged ? t_begin / ps : 0;  // logical page window [wbase, wbase + 32)
    int wcur = -1, wnxt = -1;
    if (p.paged) {
      wcur = (wbase + lane < n_pages_seq) ? __ldg(trow + wbase + lane) : -1;
      wnxt = (wbase + 32 + lane < n_pages_seq) ? __ldg(trow + wbase + 32 + lane) : -1;
    }
    int issued = 0;
    bool waited = !p.early;
    bool appended = !awaits;
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
      if (!appended && apos + a_first < t0 + kTile) {  // this tile holds a row the append warp writes
        named_bar_sync(3, 64);
        appended = true;
      }
      const uint32_t kdst = smem_u32(smem + stage * C::kStageBytes);
      const uint32_t vdst = kdst + C::kTileBytes;
      const uint32_t fb = smem_u32(&full[stage]);
      if (!p.paged) {
        if (lane == 0) {
          mbar_arrive_expect_tx(fb, C::kStageBytes);
          const int row = b * p.h_kv + j;
          if (p.merged_halves) {  // one box: both halves of 64 rows
            tma_load_4d(kdst, &tmap_k, 0, t0, 0, row, fb);
            tma_load_4d(vdst, &tmap_v, 0, t0, 0, row, fb);
          } else {
#pragma unroll
            for (int hf = 0; hf < D / 64; ++hf) {
              tma_load_3d(kdst + hf * C::kHalfBytes, &tmap_k, 64 * hf, t0, row, fb);
              tma_load_3d(vdst + hf * C::kHalfBytes, &tmap_v, 64 * hf, t0, row, fb);
            }
          }
        }
      } else {
        // Every copy is issued whole: rows past the sequence read a page that
        // is still in bounds (or, for a bad table entry, the TMA fill value),
        // and the consumers mask those rows.
        int pg[kTile / 16];
#pragma unroll
        for (int k = 0; k < kTile / 16; ++k) {
          pg[k] = -1;
          if (k * rpc < kTile) {
            int lp = (t0 + k * rpc) / ps;
            if (t0 + k * rpc + rpc <= t_lo) lp = t_lo / ps;  // wholly before the window: never read a released page
            if (lp >= n_pages_seq) lp = n_pages_seq - 1;
            while (lp >= wbase + 32) {  // warp-uniform window advance
              wbase += 32;
              wcur = wnxt;
              wnxt = (wbase + 32 + lane < n_pages_seq) ? __ldg(trow + wbase + 32 + lane) : -1;
            }
            pg[k] = __shfl_sync(0xffffffffu, wcur, lp - wbase);
            if ((pg[k] < 0 || pg[k] >= p.num_pages) && lane == 0)
              atomicOr(p.err, static_cast<int>(MQA_DEVERR_PAGE_RANGE));
          }
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(fb, C::kStageBytes);
#pragma unroll
          for (int k = 0; k < kTile / 16; ++k) {
            if (k * rpc >= kTile) break;
            const int r = (t0 + k * rpc) % ps;
            if (p.merged_halves) {  // one box per page: both halves of rpc rows
              const uint32_t off = k * rpc * 128 * (D / 64);
              tma_load_5d(kdst + off, &tmap_k, 0, r, 0, j, pg[k], fb);
              tma_load_5d(vdst + off, &tmap_v, 0, r, 0, j, pg[k], fb);
            } else {
#pragma unroll
              for (int hf = 0; hf < D / 64; ++hf) {
                tma_load_4d(kdst + hf * C::kHalfBytes + k * rpc * 128, &tmap_k, 64 * hf, r, j, pg[k], fb);
                tma_load_4d(vdst + hf * C::kHalfBytes + k * rpc * 128, &tmap_v, 64 * hf, r, j, pg[k], fb);
              }
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
  const int hb = warp >> 2;           // head block within this CTA
  const int ws = warp & 3;            // token slice of each tile
  const int head0 = (hsb * HB + hb) * 16;  // first head (within the group) of this warp's rows
  const int r0 = lane >> 2;           // fragment rows r0 and r0 + 8
  const int c2 = (lane & 3) * 2;      // fragment column pair

  WarpAttn<D> wa;
  if (p.rope_q && !MULTI) {
    // rotate q_new here: nothing the consumers read comes from the append kernel
    // (the q loads are issued before the cos / sin table is formed)
    __shared__ float s_cs[D];
    const long long qoff = (static_cast<long long>(b) * p.h_q + j * G + head0) * D;
    uint32_t qraw[D / 16][4];
    WarpAttn<D>::load_q(static_cast<const __nv_bfloat16*>(p.q_new) + qoff, G - head0, lane, qraw);
    rope_table<D>(s_cs, p, p.pos[b], threadIdx.x, 2, C::kConsumerThreads);
    wa.init_rope(qraw, G - head0, s_cs, p.scale_log2, lane,
                 (p.fuse_append && split == 0 && ws == 0) ? p.q_rot_out + qoff : nullptr);
  } else if (MULTI && p.fuse_append) {
    // fused multi-token step: q_new [B, n, H_q, D] rotated here, row (i, h)
    // by the table of position pos + i (fp32 cos / sin of the fp64-reduced
    // angle, one table per new token); the rows' loads are issued first
    float(*s_csm)[D] = reinterpret_cast<float(*)[D]>(smem + C::kBodyBytes + 2 * STAGES * 8);
    auto qnew = [&](int r) -> const __nv_bfloat16* {
      if (r >= R) return nullptr;
      const int i = r / G;
      return static_cast<const __nv_bfloat16*>(p.q_new) +
             ((static_cast<long long>(b) * nq + i) * p.h_q + j * G + (r - i * G)) * D;
    };
    auto qout = [&](int r) -> float* {
      if (r >= R || split != 0 || ws != 0) return nullptr;
      const int i = r / G;
      return p.q_rot_out + ((static_cast<long long>(b) * nq + i) * p.h_q + j * G + (r - i * G)) * D;
    };
    const int ra = head0 + (lane >> 2), rb = ra + 8;
    uint32_t qraw[D / 16][4];
    WarpAttn<D>::load_q2(qnew(ra), qnew(rb), lane, qraw);
    for (int idx = threadIdx.x; idx < nq * (D / 2); idx += C::kConsumerThreads) {
      const int i = idx / (D / 2), t = idx - i * (D / 2);
      const double ang = reduce_two_pi(static_cast<double>(apos + i) * p.theta[t]);
      float sf, cf;
      sincosf(static_cast<float>(ang), &sf, &cf);
      s_csm[i][t] = cf;
      s_csm[i][D / 2 + t] = sf;
    }
    named_bar_sync(2, C::kConsumerThreads);
    wa.init2_rope(qraw, ra < R, rb < R, s_csm[min(ra, R - 1) / G], s_csm[min(rb, R - 1) / G], p.scale_log2, lane,
                  qout(ra), qout(rb));
  } else if (MULTI) {
    if (p.early) grid_dependency_wait();  // q_rot comes from the append kernel
    auto qrow = [&](int r) -> const float* {
      if (r >= R) return nullptr;
      const int i = r / G;
      return p.q_rot + ((static_cast<long long>(b) * nq + i) * p.h_q + j * G + (r - i * G)) * D;
    };
    wa.init2(qrow(head0 + r0), qrow(head0 + r0 + 8), p.scale_log2, lane);
  } else {
    if (p.early) grid_dependency_wait();  // q_rot comes from the append kernel
    wa.init(p.q_rot + (static_cast<long long>(b) * p.h_q + j * G + head0) * D, G - head0, p.scale_log2, lane);
  }
  // MULTI: the key range [ka, ke) of this lane's rows r0 and r0 + 8 (row of
  // new token i: ends after position L - nq + i; a window of W before that)
  int ka0 = 0, ke0 = L, ka1 = 0, ke1 = L;
  if (MULTI) {
    const int i0 = min(head0 + r0, R - 1) / G, i1 = min(head0 + r0 + 8, R - 1) / G;
    ke0 = L - nq + i0 + 1;
    ke1 = L - nq + i1 + 1;
    ka0 = p.window > 0 ? max(0, ke0 - p.window) : 0;
    ka1 = p.window > 0 ? max(0, ke1 - p.window) : 0;
  }

  bool ok = true;
  const int trow0 = ws * 16;  // first tile row of this warp
  // rows per TMA box in shared memory: a page when each box holds one page's
  // two halves, else the whole tile
  const int rpb = (p.paged && p.merged_halves && p.page_size < kTile) ? p.page_size : kTile;
  const int lg_rpb = 31 - __clz(rpb);
  for (int it = 0; it < n_tiles; ++it) {
    const int stage = it % STAGES;
    if (!mbar_wait(smem_u32(&full[stage]), (it / STAGES) & 1, p.wait_ns)) {
      if (lane == 0) {
        s_abort = 1;
        atomicOr(p.err, static_cast<int>(MQA_DEVERR_TIMEOUT));
      }
      ok = false;
      break;
    }
    const int tt = t_begin + it * kTile + trow0;  // token of this warp's first row
    const int lo = max(0, t_lo - tt), hi = min(16, t_end - tt);
    if (lo < hi) {
      unsigned char* ktile = smem + stage * C::kStageBytes;
      if constexpr (MULTI) {
        wa.template step<true>(smem_u32(ktile), smem_u32(ktile + C::kTileBytes), ktile + C::kTileBytes, trow0, lo,
                               hi, lg_rpb, lane, max(0, ka0 - tt), min(16, min(ke0, t_end) - tt), max(0, ka1 - tt),
                               min(16, min(ke1, t_end) - tt));
      } else {
        wa.step(smem_u32(ktile), smem_u32(ktile + C::kTileBytes), ktile + C::kTileBytes, trow0, lo, hi, lg_rpb,
                lane);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[stage]));
  }
  wa.finish_sums();
  // ------------------------------------------- merge the 4 token slices
  // one decision for every consumer warp (the producer may time out and set
  // s_abort at any moment); the barrier also ends their reads of the stages
  if (bar_any(4, C::kConsumerThreads, *reinterpret_cast<volatile int*>(&s_abort) || !ok)) return;
  float* mo = reinterpret_cast<float*>(smem);            // [warps][16][stride]
  float* mm = mo + C::kConsumerWarps * 16 * C::kMergeStride;  // [warps][16]
  float* ml = mm + C::kConsumerWarps * 16;                     // [warps][16]
  {
    float* mine = mo + warp * 16 * C::kMergeStride;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      *reinterpret_cast<float2*>(mine + r0 * C::kMergeStride + n * 8 + c2) = make_float2(wa.o[n][0], wa.o[n][1]);
      *reinterpret_cast<float2*>(mine + (r0 + 8) * C::kMergeStride + n * 8 + c2) =
          make_float2(wa.o[n][2], wa.o[n][3]);
    }
    if ((lane & 3) == 0) {
      mm[warp * 16 + r0] = wa.m0;
      mm[warp * 16 + r0 + 8] = wa.m1;
      ml[warp * 16 + r0] = wa.l0;
      ml[warp * 16 + r0 + 8] = wa.l1;
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
      float mx = -INFINITY;
#pragma unroll
      for (int w = 0; w < 4; ++w) mx = fmaxf(mx, mm[(hbi * 4 + w) * 16 + r]);
      float num = 0.f, den = 0.f;
      if (mx != -INFINITY) {
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const int ww = hbi * 4 + w;
          const float wt = exp2f(mm[ww * 16 + r] - mx);
          num = fmaf(wt, mo[(ww * 16 + r) * C::kMergeStride + d], num);
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

template <int D, int HB>
constexpr int mma_stages() {
  return D == 128 ? MQA_MMA_STAGES_D128 : MQA_MMA_STAGES_D64;
}

template <int D, int HB, bool MULTI>
cudaError_t launch_mma_t(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream) {
  constexpr int ST = mma_stages<D, HB>();
  using C = MmaCfg<D, HB, ST>;
  auto kern = decode_mma_kernel<D, HB, ST, MULTI>;
  const int smem = C::kSmemBytes + ((MULTI && p.fuse_append) ? C::kMultiTableBytes : 0);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmemBytes + (MULTI ? C::kMultiTableBytes : 0));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.batch) * p.h_kv * p.head_blocks * p.num_splits);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tk, tv, p);
}

#ifndef MQA_MMA_MAX_HB
#define MQA_MMA_MAX_HB 2
#endif
int mma_hb(int rows) { return (rows > 16 && MQA_MMA_MAX_HB >= 2) ? 2 : 1; }

template <bool MULTI>
cudaError_t launch_mma_m(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream) {
  const int hb = mma_hb(p.group * (MULTI ? p.n_new : 1));
  if (p.head_dim == 128)
    return hb == 2 ? launch_mma_t<128, 2, MULTI>(p, tk, tv, stream) : launch_mma_t<128, 1, MULTI>(p, tk, tv, stream);
  return hb == 2 ? launch_mma_t<64, 2, MULTI>(p, tk, tv, stream) : launch_mma_t<64, 1, MULTI>(p, tk, tv, stream);
}

}  // namespace

KernelShape decode_mma_shape(int head_dim, int rows) {
  const int hb = mma_hb(rows);
  if (head_dim == 128) {
    if (hb == 2) {
      using C = MmaCfg<128, 2, mma_stages<128, 2>()>;
      return {C::kThreads, C::kSmemBytes, 32, 1};
    }
    using C = MmaCfg<128, 1, mma_stages<128, 1>()>;
    return {C::kThreads, C::kSmemBytes, 16, 0};
  }
  if (hb == 2) {
    using C = MmaCfg<64, 2, mma_stages<64, 2>()>;
    return {C::kThreads, C::kSmemBytes, 32, 1};
  }
  using C = MmaCfg<64, 1, mma_stages<64, 1>()>;
  return {C::kThreads, C::kSmemBytes, 16, 0};
}

cudaError_t launch_decode_mma(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                              cudaStream_t stream) {
  return p.n_new > 1 ? launch_mma_m<true>(p, tk, tv, stream) : launch_mma_m<false>(p, tk, tv, stream);
}

}  // namespace mqa
