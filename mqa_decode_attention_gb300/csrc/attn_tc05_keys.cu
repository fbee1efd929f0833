// One decode step of multi-query attention over a one-byte cache (one new
// token per sequence, 32 query heads per kv head: "Arsitektur Inferensi LLM",
// the MQA / GQA section; uint8 codes with a float32 (scale, zero point) per
// cached row as in the QuantizedKVCache of "KV Cache 최적화 심층 분석", or fp8
// e5m2 values) on the 5th-generation tensor cores, with the KEYS on the MMA's
// row dimension. Launched for uint8 only: an e5m2 cache takes
// attn_tc05_widen.cu (heads on the rows), measured faster for it.
//
// A decode step has only G = 32 query rows per kv head, a quarter of the 128
// rows a tcgen05 MMA computes, so the products are taken transposed and a
// tile's 128 keys fill the rows:
//   widen           four converter warps turn the landed code tile into exact
//                   fp16: uint8 code c of a row with zero point z becomes
//                   c - z (a byte permute gives 1024 + c, one half2 subtract
//                   removes 1024 + z); an e5m2 byte is the high byte of an
//                   IEEE half. K goes to tensor memory (the A operand of S^T),
//                   V to shared memory (the A operand of O^T).
//   S^T = K Q^T     tcgen05.mma M=128 (keys) N=32 (heads) K=128 (head dim),
//                   A = widened K from tensor memory, B = Q (fp16, K-major)
//   softmax         thread t of warps 0-3 owns key t of the tile: one
//                   tcgen05.ld brings its 32 scores; uint8: times the key's
//                   scale. The 32 reference maxima are shared (shared
//                   memory); each thread keeps its own 32 partial sums.
//   O^T += V^T P^T  tcgen05.mma M=128 (head dim) N=32 (heads) K=128 (keys),
//                   A = widened V read MN-major, B = P^T (fp16) written by the
//                   softmax threads into shared memory (64-byte swizzle);
//                   uint8: P^T carries p * s^v / 4, so O^T sums p (c - z) s^v
//   epilogue        O^T / l (uint8: times 4), thread = head dim
// The reference maximum of a head moves only when one of its scores exceeds
// it by more than 2^8 (P stays below 256, O / l is unchanged): each thread
// tests its 32 scores and one barrier reduction (bar.red.or) over the four
// softmax warps tells whether any did. Only then -- the first tile, and
// rarely later -- are the tile's per-head maxima reduced (a butterfly leaving
// head h on lane h, then the four warps through shared memory) and O^T's
// columns rescaled.
//
// Warps: 0-3 softmax and epilogue, 4 K loader, 5 V loader (TMA: codes and,
// uint8, the (scale, zero point) rows; 3 stages each), 6 MMA issue (one
// thread) and tensor-memory allocation, 7-10 converters (warp w widens the
// rows of tensor-memory lane quarter w mod 4).
// In a one-token step the kernel is the only launch (FUSE): the softmax warps
// rotate q_new and write q_rot, warp 11 quantises the new row with the append
// kernel's encoder (append_row_q) and the loaders wait for it only before the
// tile that holds it.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "../../include/mqa_decode.h"
#include "launch.h"
#include "ptx.cuh"
#include "quant.cuh"
#include "rope.cuh"
#include "tc05.cuh"

namespace mqa {
namespace {

constexpr int kD = 128;      // head_dim
constexpr int kNP = 32;      // query heads of a kv head (MMA N)
constexpr int kBN = 128;     // keys per tile (MMA M of S^T)
constexpr int kStages = 3;   // code tiles in flight
constexpr int kPB = 3;       // S^T buffers (tensor memory), P^T and scale buffers (shared memory)
constexpr int kOpB = 2;      // widened K (tensor memory) and V (shared memory) buffers
constexpr int kThreads = 384;
constexpr int kCodeBytes = kBN * kD;                     // 16 KB: [128 rows][128 B], 128-byte swizzle
constexpr int kSzBytes = kBN * 8;                        // 1 KB: (scale, zero point) per row
constexpr int kCodeStage = kCodeBytes + kSzBytes;        // 17 KB (1 KB multiple)
constexpr int kOpBytes = kBN * kD * 2;                   // 32 KB: [2 halves][128 rows][128 B]
constexpr int kQHalf = kNP * 128;                        // one 64-dim half of the Q tile
constexpr int kPBytes = kBN * kNP * 2;                   // 8 KB: [128 keys][64 B]
constexpr int kKCOff = 0;
constexpr int kVCOff = kKCOff + kStages * kCodeStage;
constexpr int kVOpOff = kVCOff + kStages * kCodeStage;
constexpr int kQOff = kVOpOff + kOpB * kOpBytes;
constexpr int kPOff = kQOff + 2 * kQHalf;
constexpr int kSclOff = kPOff + kPB * kPBytes;           // [kPB][128] (s^k, s^v)
constexpr int kBarOff = kSclOff + kPB * kBN * 8;
constexpr int kSmemBytes = kBarOff + 512 + 1024;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0;                  // S^T buffers, 32 columns each
constexpr uint32_t kColO = kPB * kNP;          // O^T
constexpr uint32_t kColK = 128;                // widened K buffers, 64 columns each (fp16 pairs)
static_assert(kColO + kNP <= kColK && kColK + kOpB * 64 <= kTmemCols, "tensor memory");
constexpr float kRescaleLog2 = 8.0f;
// initial reference maximum: below every finite score, so the first valid key
// of a head moves it, yet finite, so that exp2(score - m) needs no test (a
// block's first tile always holds a valid key: the range starts at most 63
// keys before the window)
constexpr float kNoMax = -1e30f;
// uint8: P^T = p * s^v * kPScale in fp16; p < 256, so a V scale up to 1023
// stays below fp16's 65504
constexpr float kPScale = 0.25f;
constexpr float kMaxVScale = 1023.0f;

// mbarriers (8 bytes each) at kBarOff
constexpr int kQReady = 0;
constexpr int kKFull = 1;                    // [kStages] K codes (and rows' scales) landed
constexpr int kKEmpty = kKFull + kStages;    // [kStages] ... read by the converters
constexpr int kVFull = kKEmpty + kStages;    // [kStages]
constexpr int kVEmpty = kVFull + kStages;    // [kStages]
constexpr int kKOpFull = kVEmpty + kStages;  // [kOpB] widened K in tensor memory
constexpr int kKOpEmpty = kKOpFull + kOpB;   // [kOpB] ... read by its S^T
constexpr int kVOpFull = kKOpEmpty + kOpB;   // [kOpB] widened V in shared memory
constexpr int kVOpEmpty = kVOpFull + kOpB;   // [kOpB] ... read by its PV
constexpr int kSFull = kVOpEmpty + kOpB;     // [kPB]
constexpr int kPFull = kSFull + kPB;         // [kPB]
constexpr int kODone = kPFull + kPB;         // [kPB]
constexpr int kSclFull = kODone + kPB;       // [kPB] uint8: the tile's row scales for the softmax
constexpr int kSclEmpty = kSclFull + kPB;    // [kPB]
constexpr int kDrain = kSclEmpty + kPB;
constexpr int kAppended = kDrain + 1;        // fused step: the new row's codes and scales are in the cache
constexpr int kNBars = kAppended + 1;
static_assert(kNBars * 8 + 4 <= 512, "barrier area");

// named barriers: 1 the softmax warps (bar.sync), 2 Q rows requested
// (softmax + loaders), 3 the softmax warps' votes (bar.red; never mixed with
// bar.sync on one barrier), 4 the fused step's cos / sin table
constexpr int kBarSoftmax = 1, kBarQ = 2, kBarVote = 3, kBarTable = 4;

__device__ __forceinline__ bool aborted(const Tc05Params& p) {
  return (*reinterpret_cast<volatile int32_t*>(p.err) & static_cast<int>(MQA_DEVERR_TIMEOUT)) != 0;
}

// Butterfly over the warp: on return v[0] of lane h is op over the 32 lanes of
// the values they held for head h (the other entries are spent).
template <bool MAX>
__device__ __forceinline__ float warp_reduce_heads(float (&v)[32], int lane) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool up = (lane & w) != 0;  // this lane keeps the upper w heads of its current 2w
#pragma unroll
    for (int k = 0; k < w; ++k) {
      const float keep = up ? v[k + w] : v[k];
      const float send = up ? v[k] : v[k + w];
      const float got = __shfl_xor_sync(0xffffffffu, send, w);
      v[k] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
  return v[0];
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Four codes (bytes 0-3 of w, dims 0-3) as two fp16 pairs, dims (0, 1) and
// (2, 3), the lower dim in the low half. uint8: c - z exactly (1024 + c is the
// half 0x64cc; zz holds 1024 + z twice). e5m2: the byte as the high byte of a
// half, which is the e5m2 value exactly.
template <bool U8>
__device__ __forceinline__ void widen4(uint32_t w, uint32_t zz, uint32_t& lo, uint32_t& hi) {
  if constexpr (U8) {
    const uint32_t a = prmt(w, 0x64646464u, 0x4140u), b = prmt(w, 0x64646464u, 0x4342u);
    __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&zz));
    __half2 hb = __hsub2(*reinterpret_cast<const __half2*>(&b), *reinterpret_cast<const __half2*>(&zz));
    lo = *reinterpret_cast<uint32_t*>(&ha);
    hi = *reinterpret_cast<uint32_t*>(&hb);
  } else {
    lo = prmt(w, 0u, 0x1404u);
    hi = prmt(w, 0u, 0x3424u);
  }
}

template <bool U8, bool FUSE>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc05_keys_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                          const __grid_constant__ CUtensorMap tmap_ksz, const __grid_constant__ CUtensorMap tmap_vsz,
                          const Tc05Params p) {
  extern __shared__ unsigned char smem_raw[];
  // 1 KB aligned (128-byte swizzle atoms); offsetting the __shared__ array
  // itself keeps accesses through `smem` in the shared state space
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + kBarOff + kNBars * 8);
  __shared__ int s_abort, s_skip;
  __shared__ float s_red[4][kNP];  // per-warp partial maxima / sums of each head
  __shared__ __align__(16) float s_mref[kNP];   // reference maxima of the heads
  __shared__ __align__(16) float s_alpha[kNP];  // their rescale factors when they move
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.group, S = p.num_splits;
  int cta = blockIdx.x;
  const int b = cta % p.batch;
  cta /= p.batch;
  const int j = cta % p.h_kv;
  const int split = cta / p.h_kv;

  long long limit = p.capacity < p.max_seq_len ? p.capacity : p.max_seq_len;
  int L = p.seq_lens[b];
  const int apos = FUSE ? p.pos[b] : 0;  // fused step: the new token's position
  if (L < 1 || L > limit) {
    // reported; the rows are then unspecified
    if (tid == 0 && split == 0 && j == 0) atomicOr(p.err, static_cast<int>(MQA_DEVERR_SEQ_LEN));
    L = L < 1 ? 1 : static_cast<int>(limit);
  }
  if (tid == 0) s_skip = aborted(p) ? 1 : 0;  // an earlier block timed out: the result is invalid already
  __syncthreads();
  if (s_skip) return;
  const int Lp = L - 1;  // the new token's position: keys [ka, Lp]
  const int ka = p.window > 0 ? max(0, Lp + 1 - p.window) : 0;
  // the split's token range (as the other decode kernels cut it)
  const int kstart = (ka / 64) * 64 + split * p.chunk;
  const int t_end = min(L, kstart + p.chunk);
  const int T = t_end > kstart ? (t_end - kstart + kBN - 1) / kBN : 0;  // key tiles of this block
  const bool split_out = S > 1;
  const long long row0 = static_cast<long long>(b) * p.h_q + j * G;  // output row of head 0 of the group
  // fused step: the split whose token range holds the new token's position
  // (else split 0) appends its row
  const int tbase = (ka / 64) * 64;
  const bool writer =
      FUSE && split == ((apos - tbase >= 0 && (apos - tbase) / p.chunk < S) ? (apos - tbase) / p.chunk : 0);
  if (T == 0) {
    // no key of this split: an empty partial (weight 0 in the combine)
    grid_dependency_wait();
    if (split_out) {
      for (int idx = tid; idx < G * kD; idx += kThreads) {
        const long long grow = row0 + idx / kD;
        p.o_part[(grow * S + split) * kD + idx % kD] = 0.f;
        if (idx % kD == 0) p.lse_part[grow * S + split] = -INFINITY;
      }
    }
    return;
  }

  if (tid == 0) {
    s_abort = 0;
    mbar_init(bar(kQReady), 4);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kKFull + s), 1);
      mbar_init(bar(kKEmpty + s), 4);
      mbar_init(bar(kVFull + s), 1);
      mbar_init(bar(kVEmpty + s), 4);
    }
    for (int s = 0; s < kOpB; ++s) {
      mbar_init(bar(kKOpFull + s), 4);
      mbar_init(bar(kKOpEmpty + s), 1);
      mbar_init(bar(kVOpFull + s), 4);
      mbar_init(bar(kVOpEmpty + s), 1);
    }
    for (int s = 0; s < kPB; ++s) {
      mbar_init(bar(kSFull + s), 1);
      mbar_init(bar(kPFull + s), 4);
      mbar_init(bar(kODone + s), 1);
      mbar_init(bar(kSclFull + s), 4);
      mbar_init(bar(kSclEmpty + s), 4);
    }
    mbar_init(bar(kDrain), 1);
    mbar_init(bar(kAppended), 1);  // the append warp
    fence_mbar_init();
  }
  if (warp == 6) {
    tc05::tmem_alloc(smem_u32(tslot), kTmemCols);
    tc05::tmem_relinquish();
  }
  tc05::fence_before_sync();
  __syncthreads();
  tc05::fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tslot);
  const uint32_t sbase = smem_u32(smem);
  // q_rot and the new token's cache row come from the preceding launch. After
  // the append kernel (early) every other cached row is final already: the
  // loaders stream those while it runs and wait only before the tile that
  // holds the new token; the softmax threads wait before reading q_rot.
  // The combine (or the next step) may be scheduled now; it waits for this
  // whole grid before it reads anything this grid writes.
  grid_dependents_launch();
  if (!p.early) grid_dependency_wait();

  auto fail = [&](int role_lane0) {
    if (role_lane0) {
      s_abort = 1;
      atomicOr(p.err, static_cast<int>(MQA_DEVERR_TIMEOUT));
    }
  };
  auto stop = [&]() { return *reinterpret_cast<volatile int*>(&s_abort) != 0; };

  if (warp == 4 || warp == 5) {
    // ------------------------------------------------- K (warp 4) / V (warp 5) loaders
    const bool is_k = warp == 4;
    const CUtensorMap* map = is_k ? &tmap_k : &tmap_v;
    const CUtensorMap* map_sz = is_k ? &tmap_ksz : &tmap_vsz;
    const int full = is_k ? kKFull : kVFull, empty = is_k ? kKEmpty : kVEmpty;
    const uint32_t dst0 = sbase + (is_k ? kKCOff : kVCOff);
    const int row = b * p.h_kv + j;
    auto issue = [&](int it) {
      const int s = it % kStages, tok = kstart + it * kBN;
      const uint32_t dst = dst0 + s * kCodeStage;
      mbar_arrive_expect_tx(bar(full + s), kCodeBytes + (U8 ? kSzBytes : 0));
      tma_load_3d(dst, map, 0, tok, row, bar(full + s));
      if (U8) tma_load_2d(dst + kCodeBytes, map_sz, 2 * tok, row, bar(full + s));
    };
    int it = 0;
    if (p.early) {
      // while the append kernel runs: the ring's first fill, tiles wholly
      // before the new token
      for (; it < T && it < kStages && kstart + (it + 1) * kBN <= Lp; ++it)
        if (lane == 0) issue(it);
    }
    // the rest only once the Q rows have been requested: behind a burst of
    // tile loads the Q reads would wait microseconds
    named_bar_sync(kBarQ, 128 + 64);
    if (lane == 0) {
      bool waited = !p.early, appended = !writer;
      for (; it < T; ++it) {
        const int s = it % kStages;
        if (it >= kStages && !mbar_wait(bar(empty + s), ((it - kStages) / kStages) & 1)) {
          fail(1);
          break;
        }
        if (stop()) break;
        if (!waited && Lp < kstart + (it + 1) * kBN) {  // this tile holds the new token's row
          grid_dependency_wait();
          waited = true;
        }
        if (!appended && apos < kstart + (it + 1) * kBN) {  // ... written by this block's append warp
          if (!mbar_wait(bar(kAppended), 0)) {
            fail(1);
            break;
          }
          appended = true;
        }
        issue(it);
      }
    }
    __syncwarp();
  } else if (warp == 6) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      const uint32_t id_s = tc05::idesc_f16_f32(kBN, kNP, false, false);  // K (tensor memory) x Q (K-major)
      // V^T (MN-major) x P^T (MN-major; its 32 heads are one 64-byte swizzle
      // atom wide, so the leading offset between atoms is unused)
      const uint32_t id_o = tc05::idesc_f16_f32(kD, kNP, true, true);
      const uint32_t q_s = sbase + kQOff;
      bool ok = mbar_wait(bar(kQReady), 0);
      // S^T of tile it into buffer it % kPB. That buffer was last read by the
      // softmax of tile it - kPB, which arrived on its P barrier afterwards.
      auto issue_s = [&](int it) {
        const int sb = it % kPB, kb = it % kOpB;
        tc05::fence_after_sync();
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks)
          tc05::mma_bf16_ta(tmem + kColS + sb * kNP, tmem + kColK + kb * 64 + ks * 8,
                            tc05::smem_desc_sw128(q_s + (ks >> 2) * kQHalf + (ks & 3) * 32, 16, 1024), id_s,
                            ks > 0);
        tc05::commit(bar(kSFull + sb));
        tc05::commit(bar(kKOpEmpty + kb));
      };
      auto issue_pv = [&](int it) {
        const int pb = it % kPB, vb = it % kOpB;
        tc05::fence_after_sync();
        const uint32_t v_s = sbase + kVOpOff + vb * kOpBytes;
        const uint32_t p_s = sbase + kPOff + pb * kPBytes;
#pragma unroll
        for (int ks = 0; ks < kBN / 16; ++ks)
          tc05::mma_bf16(tmem + kColO, tc05::smem_desc_sw128(v_s + ks * 2048, 16384, 1024),
                         tc05::smem_desc_sw64(p_s + ks * 1024, 16, 512), id_o, it > 0 || ks > 0);
        tc05::commit(bar(kODone + pb));
        tc05::commit(bar(kVOpEmpty + vb));
      };
      int ns = 0, np = 0;
      unsigned long long t_idle = global_timer_ns();
      while (ok && np < T) {
        bool progress = false;
        if (ns < T && ns <= np + (kPB - 1) && mbar_test(bar(kKOpFull + ns % kOpB), (ns / kOpB) & 1)) {
          issue_s(ns++);
          progress = true;
        }
        if (np < ns && mbar_test(bar(kPFull + np % kPB), (np / kPB) & 1) &&
            mbar_test(bar(kVOpFull + np % kOpB), (np / kOpB) & 1)) {
          issue_pv(np++);
          progress = true;
        }
        if (progress) {
          t_idle = global_timer_ns();
        } else if (stop() || global_timer_ns() - t_idle > kWaitLimitNs) {
          ok = false;
        } else {
          __nanosleep(32);
        }
      }
      if (!ok) fail(1);
    }
    __syncwarp();
  } else if (warp == 11) {
    // ------------------------------------------------------ append (fused step)
    // the new token's codes and (scale, zero point) rows exactly as the append
    // kernel writes them (append_row_q); a position outside the cache is
    // reported and nothing is written. Fenced for the loaders' TMA reads, which
    // wait for it only before the tile that holds the row.
    if (writer) {
      long long row = -1;
      if (apos >= 0 && apos < p.capacity)
        row = ((static_cast<long long>(b) * p.h_kv + j) * p.capacity + apos) * kD;
      else if (lane == 0)
        atomicOr(p.err, static_cast<int>(MQA_DEVERR_POS_RANGE));
      append_row_q<kD, !U8>(p, b, j, apos, row, lane);
      if (lane == 0) mbar_arrive(bar(kAppended));
    }
  } else if (warp >= 7) {
    // ----------------------------------------------------- converters (row = key)
    const int ct = 32 * (warp & 3) + lane;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t sw = static_cast<uint32_t>(ct & 7);
    for (int it = 0; it < T; ++it) {
      const int s = it % kStages, ob = it % kOpB, sb = it % kPB;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(bar(kKFull + s), (it / kStages) & 1) &&
                                                  mbar_wait(bar(kVFull + s), (it / kStages) & 1) && !stop());
      if (!ok) {
        if (lane == 0) fail(1);
        break;
      }
      const unsigned char* kc = smem + kKCOff + s * kCodeStage;
      const unsigned char* vc = smem + kVCOff + s * kCodeStage;
      uint4 kr[8], vr[8];  // codes of dims 16 c .. 16 c + 15
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        kr[c] = *reinterpret_cast<const uint4*>(kc + ct * 128 + ((c ^ sw) << 4));
        vr[c] = *reinterpret_cast<const uint4*>(vc + ct * 128 + ((c ^ sw) << 4));
      }
      float2 ksz = make_float2(1.f, 0.f), vsz = make_float2(1.f, 0.f);
      if constexpr (U8) {
        ksz = *reinterpret_cast<const float2*>(kc + kCodeBytes + ct * 8);
        vsz = *reinterpret_cast<const float2*>(vc + kCodeBytes + ct * 8);
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(kKEmpty + s));
        mbar_arrive(bar(kVEmpty + s));
      }
      const bool past = kstart + it * kBN + ct >= t_end;  // past the split: V row of zeros
      if constexpr (U8) {
        // the row's scales for the softmax thread of this key
        const bool free_slot = it < kPB || mbar_wait(bar(kSclEmpty + sb), ((it - kPB) / kPB) & 1);
        if (!__all_sync(0xffffffffu, free_slot)) {
          if (lane == 0) fail(1);
          break;
        }
        *reinterpret_cast<float2*>(smem + kSclOff + (sb * kBN + ct) * 8) = make_float2(ksz.x, vsz.x);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kSclFull + sb));
      }
      // ---- K: widened into tensor memory (lane = key, column pair = dims)
      if (it >= kOpB && !__all_sync(0xffffffffu, mbar_wait(bar(kKOpEmpty + ob), ((it - kOpB) / kOpB) & 1))) {
        if (lane == 0) fail(1);
        break;
      }
      tc05::fence_after_sync();
      {
        __half2 zh = __float2half2_rn(1024.f + ksz.y);
        const uint32_t zz = *reinterpret_cast<uint32_t*>(&zh);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {  // dims 64 hh .. + 63: 32 columns of fp16 pairs
          uint32_t ko[32];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint4 w = kr[4 * hh + i];
            widen4<U8>(w.x, zz, ko[8 * i + 0], ko[8 * i + 1]);
            widen4<U8>(w.y, zz, ko[8 * i + 2], ko[8 * i + 3]);
            widen4<U8>(w.z, zz, ko[8 * i + 4], ko[8 * i + 5]);
            widen4<U8>(w.w, zz, ko[8 * i + 6], ko[8 * i + 7]);
          }
          tc05::st_32x32b_x32_u(tmem + lane_base + kColK + ob * 64 + 32 * hh, ko);
        }
      }
      tc05::wait_st();
      tc05::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kKOpFull + ob));
      // ---- V: widened into the swizzled operand tile (row = key)
      if (it >= kOpB && !__all_sync(0xffffffffu, mbar_wait(bar(kVOpEmpty + ob), ((it - kOpB) / kOpB) & 1))) {
        if (lane == 0) fail(1);
        break;
      }
      {
        __half2 zh = __float2half2_rn(1024.f + vsz.y);
        const uint32_t zz = *reinterpret_cast<uint32_t*>(&zh);
        unsigned char* vrow = smem + kVOpOff + ob * kOpBytes + ct * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {  // codes of dims 16c .. 16c + 15: two 16-byte chunks of fp16
          uint4 o0 = make_uint4(0u, 0u, 0u, 0u), o1 = make_uint4(0u, 0u, 0u, 0u);
          if (!past) {
            widen4<U8>(vr[c].x, zz, o0.x, o0.y);
            widen4<U8>(vr[c].y, zz, o0.z, o0.w);
            widen4<U8>(vr[c].z, zz, o1.x, o1.y);
            widen4<U8>(vr[c].w, zz, o1.z, o1.w);
          }
          const int half = c >> 2, cc = 2 * (c & 3);
          *reinterpret_cast<uint4*>(vrow + half * 16384 + ((cc ^ sw) << 4)) = o0;
          *reinterpret_cast<uint4*>(vrow + half * 16384 + (((cc + 1) ^ sw) << 4)) = o1;
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kVOpFull + ob));
    }
  } else {
    // ------------------------------------------- softmax (key = thread) and epilogue
    const int t = tid;
    {
      // Q: thread t brings dims 32 (t % 4) .. + 32 of head t / 4, pre-scaled
      // into the log2 domain, as fp16 into the swizzled tile (rows past G are
      // zero). The loads are issued before the loaders are released: behind
      // their burst of tile requests they would wait microseconds.
      const int r = t >> 2, qd = t & 3;
      const bool live = r < G;
      const long long grow = row0 + r;
      float qv[32];
      if constexpr (FUSE) {
        // fused step: q_new (bf16) rotated here, pair i by the fp32 cosine /
        // sine of the fp64-reduced angle pos * theta_i, as the other fused
        // kernels form q_rot
        __shared__ float s_cs[kD];
        const uint4* qn = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.q_new) + grow * kD + 32 * qd);
        uint4 raw[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) raw[c] = live ? qn[c] : make_uint4(0u, 0u, 0u, 0u);
        named_bar_arrive(kBarQ, 128 + 64);
        if (t < kD / 2) {
          const double ang = reduce_two_pi(static_cast<double>(apos) * p.theta[t]);
          float sf, cf;
          sincosf(static_cast<float>(ang), &sf, &cf);
          s_cs[t] = cf;
          s_cs[kD / 2 + t] = sf;
        }
        named_bar_sync(kBarTable, 128);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t w4[4] = {raw[c].x, raw[c].y, raw[c].z, raw[c].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int pi = 16 * qd + 4 * c + e;  // pair (2 pi, 2 pi + 1)
            const float x = bf16lo_to_f32(w4[e]), y = bf16hi_to_f32(w4[e]);
            const float cs = s_cs[pi], sn = s_cs[kD / 2 + pi];
            qv[8 * c + 2 * e] = x * cs - y * sn;
            qv[8 * c + 2 * e + 1] = x * sn + y * cs;
          }
        }
        if (live && split == 0) {  // one copy of each row to q_rot
          float4* qo = reinterpret_cast<float4*>(p.q_rot_out + grow * kD + 32 * qd);
#pragma unroll
          for (int c = 0; c < 8; ++c) qo[c] = make_float4(qv[4 * c], qv[4 * c + 1], qv[4 * c + 2], qv[4 * c + 3]);
        }
      } else {
        if (p.early) grid_dependency_wait();
        const float4* q = reinterpret_cast<const float4*>(p.q_rot + grow * kD + 32 * qd);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float4 v = live ? q[c] : make_float4(0.f, 0.f, 0.f, 0.f);
          qv[4 * c] = v.x;
          qv[4 * c + 1] = v.y;
          qv[4 * c + 2] = v.z;
          qv[4 * c + 3] = v.w;
        }
        named_bar_arrive(kBarQ, 128 + 64);
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {  // 8 dims = one 16-byte chunk of the 128-byte row
        const int col = 32 * qd + 8 * c, half = col >> 6, chunk = (col & 63) >> 3;
        __half2 h0 = __floats2half2_rn(qv[8 * c] * p.scale_log2, qv[8 * c + 1] * p.scale_log2);
        __half2 h1 = __floats2half2_rn(qv[8 * c + 2] * p.scale_log2, qv[8 * c + 3] * p.scale_log2);
        __half2 h2 = __floats2half2_rn(qv[8 * c + 4] * p.scale_log2, qv[8 * c + 5] * p.scale_log2);
        __half2 h3 = __floats2half2_rn(qv[8 * c + 6] * p.scale_log2, qv[8 * c + 7] * p.scale_log2);
        uint4 v;
        v.x = *reinterpret_cast<uint32_t*>(&h0);
        v.y = *reinterpret_cast<uint32_t*>(&h1);
        v.z = *reinterpret_cast<uint32_t*>(&h2);
        v.w = *reinterpret_cast<uint32_t*>(&h3);
        *reinterpret_cast<uint4*>(smem + kQOff + half * kQHalf + r * 128 + ((chunk ^ (r & 7)) << 4)) = v;
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kQReady));
    }
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    // the reference maxima are the same for every thread: they live in shared
    // memory (read as broadcast 16-byte loads), which keeps the softmax within
    // the registers of a 480-thread block
    const float4* mref4 = reinterpret_cast<const float4*>(s_mref);
    const float4* alpha4 = reinterpret_cast<const float4*>(s_alpha);
    if (t < kNP) s_mref[t] = kNoMax;
    float l_part[kNP];  // this key's partial sums of each head
#pragma unroll
    for (int h = 0; h < kNP; ++h) l_part[h] = 0.f;
    named_bar_sync(kBarSoftmax, 128);
    bool ok = true, big_scale = false;
    for (int it = 0; it < T; ++it) {
      const int sb = it % kPB;
      const int kk = kstart + it * kBN + t;
      // every wait of the tile first, so that a timeout anywhere ends all four
      // warps at the same barrier below
      bool mine = mbar_wait(bar(kSFull + sb), (it / kPB) & 1);
      // P^T buffer sb was last read by the PV of tile it - kPB
      if (it >= kPB) mine = mine && mbar_wait(bar(kODone + sb), ((it - kPB) / kPB) & 1);
      if (U8) mine = mine && mbar_wait(bar(kSclFull + sb), (it / kPB) & 1);
      mine = mine && !stop();
      tc05::fence_after_sync();
      float s[kNP];
      tc05::ld_32x32b_x32(tmem + lane_base + kColS + sb * kNP, s);
      float2 sc = make_float2(1.f, 1.f);  // this key's (K scale, V scale)
      if constexpr (U8) {
        sc = *reinterpret_cast<const float2*>(smem + kSclOff + (sb * kBN + t) * 8);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kSclEmpty + sb));
      }
      tc05::wait_ld();
      tc05::reg_fence(s);
      const bool valid = kk >= ka && kk < t_end;
      if (valid) {
        if constexpr (U8) {
#pragma unroll
          for (int h = 0; h < kNP; ++h) s[h] *= sc.x;
          big_scale |= sc.y > kMaxVScale;
        }
      } else {
#pragma unroll
        for (int h = 0; h < kNP; ++h) s[h] = -INFINITY;
      }
      bool grow = false;
#pragma unroll
      for (int c = 0; c < kNP / 4; ++c) {
        const float4 m4 = mref4[c];
        grow |= (s[4 * c] > m4.x + kRescaleLog2) | (s[4 * c + 1] > m4.y + kRescaleLog2) |
                (s[4 * c + 2] > m4.z + kRescaleLog2) | (s[4 * c + 3] > m4.w + kRescaleLog2);
      }
      if (bar_any(kBarVote, 128, grow || !mine)) {
        // a timeout, or a head's maximum grew by more than 2^8: the tile's
        // per-head maxima over its 128 keys
        if (bar_any(kBarVote, 128, !mine)) {
          ok = false;
          break;
        }
        float v[kNP];
#pragma unroll
        for (int h = 0; h < kNP; ++h) v[h] = s[h];
        s_red[warp][lane] = warp_reduce_heads<true>(v, lane);
        named_bar_sync(kBarSoftmax, 128);
        bool g = false;
        if (t < kNP) {  // thread h decides head h
          const float mt = fmaxf(fmaxf(s_red[0][t], s_red[1][t]), fmaxf(s_red[2][t], s_red[3][t]));
          const float mo = s_mref[t];
          g = mt > mo + kRescaleLog2;  // the same test the threads took, on the maximum
          const float m_new = g ? mt : mo;
          s_alpha[t] = g ? fast_exp2(mo - m_new) : 1.f;  // 0 from kNoMax: nothing to keep
          s_mref[t] = m_new;
        }
        const bool rescale = bar_any(kBarVote, 128, g);  // also publishes s_mref / s_alpha
        if (it > 0 && rescale) {
          // O^T is rescaled (thread = head dim, column = head): PV of the
          // previous tile must be done first
          const bool done = mbar_wait(bar(kODone + (it - 1) % kPB), ((it - 1) / kPB) & 1) && !stop();
          if (bar_any(kBarVote, 128, !done)) {
            ok = false;
            break;
          }
          tc05::fence_after_sync();
          float o[kNP];
          tc05::ld_32x32b_x32(tmem + lane_base + kColO, o);
          tc05::wait_ld();
          tc05::reg_fence(o);
#pragma unroll
          for (int c = 0; c < kNP / 4; ++c) {
            const float4 a4 = alpha4[c];
            o[4 * c] *= a4.x;
            o[4 * c + 1] *= a4.y;
            o[4 * c + 2] *= a4.z;
            o[4 * c + 3] *= a4.w;
          }
          tc05::st_32x32b_x32(tmem + lane_base + kColO, o);
          tc05::wait_st();
        }
        if (rescale) {
#pragma unroll
          for (int c = 0; c < kNP / 4; ++c) {
            const float4 a4 = alpha4[c];
            l_part[4 * c] *= a4.x;
            l_part[4 * c + 1] *= a4.y;
            l_part[4 * c + 2] *= a4.z;
            l_part[4 * c + 3] *= a4.w;
          }
        }
        named_bar_sync(kBarSoftmax, 128);  // s_red and s_alpha are read by all before their next use
      }
      // P^T row of this key: 32 heads as fp16, 64 bytes in four 16-byte
      // chunks, chunk c at c ^ ((t / 2) mod 4) (64-byte swizzle); a masked
      // key gives 0 (uint8: also when its V scale is not a number)
      const float pv = U8 ? (valid ? sc.y * kPScale : 0.f) : 1.f;
      unsigned char* prow = smem + kPOff + sb * kPBytes + t * 64;
#pragma unroll
      for (int c = 0; c < 4; ++c) {  // heads 8c .. 8c + 7
        const float4 ma = mref4[2 * c], mb = mref4[2 * c + 1];
        const float m8[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int h = 8 * c + 2 * e;
          const float p0 = fast_exp2(s[h] - m8[2 * e]);
          const float p1 = fast_exp2(s[h + 1] - m8[2 * e + 1]);
          l_part[h] += p0;
          l_part[h + 1] += p1;
          __half2 hp = __floats2half2_rn(p0 * pv, p1 * pv);
          pk[e] = *reinterpret_cast<uint32_t*>(&hp);
        }
        *reinterpret_cast<uint4*>(prow + ((c ^ ((t >> 1) & 3)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc05::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kPFull + sb));
    }
    if (U8 && big_scale) atomicOr(p.err, static_cast<int>(MQA_DEVERR_U8_SCALE));
    if (ok) ok = mbar_wait(bar(kODone + (T - 1) % kPB), ((T - 1) / kPB) & 1);
    // every softmax thread reaches the barriers below (a timeout ends the loop
    // of all four warps at the same tile)
    const bool all_ok = !bar_any(kBarVote, 128, !ok || stop());
    if (!all_ok && lane == 0) fail(1);
    if (all_ok) {
      tc05::fence_after_sync();
      // ---- epilogue: l of each head over the block's keys; O^T / l, thread = head dim
      s_red[warp][lane] = warp_reduce_heads<false>(l_part, lane);
      named_bar_sync(kBarSoftmax, 128);
      if (t < G) {
        const float lh = (s_red[0][t] + s_red[1][t]) + (s_red[2][t] + s_red[3][t]);
        const float lse = lh > 0.f ? (s_mref[t] + log2f(lh)) * 0.69314718055994530942f : -INFINITY;
        if (split_out)
          p.lse_part[(row0 + t) * S + split] = lse;
        else if (p.lse_out != nullptr)
          p.lse_out[row0 + t] = lse;
      }
      float o[kNP];
      tc05::ld_32x32b_x32(tmem + lane_base + kColO, o);
      tc05::wait_ld();
      tc05::reg_fence(o);
      const int d = t;
#pragma unroll
      for (int h = 0; h < kNP; ++h) {
        if (h < G) {
          const float lh = (s_red[0][h] + s_red[1][h]) + (s_red[2][h] + s_red[3][h]);
          const float ov = lh > 0.f ? o[h] * ((U8 ? 1.f / kPScale : 1.f) / lh) : 0.f;
          const long long grow = row0 + h;
          if (split_out)
            p.o_part[(grow * S + split) * kD + d] = ov;
          else if (p.out_dtype == kDtypeBf16)
            static_cast<__nv_bfloat16*>(p.out)[grow * kD + d] = __float2bfloat16_rn(ov);
          else
            static_cast<float*>(p.out)[grow * kD + d] = ov;
        }
      }
    }
  }

  // ---- teardown: every role is done with tensor memory
  tc05::fence_before_sync();
  __syncthreads();
  if (warp == 6) {
    if (*reinterpret_cast<volatile int*>(&s_abort)) {
      // MMAs may still be in flight after a timeout: wait (bounded) for them
      // before the columns are released
      if (lane == 0) {
        tc05::commit(bar(kDrain));
        (void)mbar_wait(bar(kDrain), 0);
      }
      __syncwarp();
    }
    tc05::fence_after_sync();
    tc05::tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool U8, bool FUSE>
cudaError_t launch_keys(const Tc05Params& p, const CUtensorMap* maps, cudaStream_t stream) {
  auto kern = attn_tc05_keys_kernel<U8, FUSE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.batch) * p.h_kv * p.num_splits);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], maps[3], p);
}

}  // namespace

KernelShape tc05_keys_shape() { return {kThreads, kSmemBytes, kNP, 1}; }

bool tc05_keys_applies(int group, int n_new, int head_dim, bool paged) {
  return n_new == 1 && group > 16 && group <= kNP && head_dim == kD && !paged;
}

cudaError_t launch_tc05_keys_attention(const Tc05Params& p, int cache_dtype, const CUtensorMap* maps,
                                       cudaStream_t stream) {
  // an e5m2 cache takes attn_tc05_widen.cu (measured faster there); the
  // kernel's e5m2 form (U8 = false) is kept compiled out
  if (cache_dtype != kDtypeU8) return cudaErrorInvalidValue;
  return p.fuse ? launch_keys<true, true>(p, maps, stream) : launch_keys<true, false>(p, maps, stream);
}

}  // namespace mqa
