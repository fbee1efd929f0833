// One decode step of multi-query attention over an fp8 e5m2 cache (one new
// token per sequence, 17 to 32 query heads per kv head: "Arsitektur Inferensi
// LLM", the MQA / GQA section; the one-byte e5m2 values of the pages' vLLM
// cache flag) on the 5th-generation tensor cores, with the query heads on the
// MMA rows and 128 keys per MMA: the layout of the bf16 kernel
// (attn_tc05.cu), fed by converter warps that widen the code tiles.
//
//   widen           converter warps (two for K, two for V) turn each landed
//                   code tile into an exact fp16 operand tile in shared
//                   memory, two key rows per thread: an e5m2 byte is the high
//                   byte of an IEEE half. Rows past the split are written as
//                   zeros.
//   S = Q K^T       tcgen05.mma M=128 N=128 K=128: Q (fp16, the G <= 32 heads
//                   replicated four times over the 128 rows) and the widened
//                   K tile, both from shared memory; S into tensor memory
//   softmax         thread r keeps the online softmax of head r mod 32 over
//                   its quarter (32 keys) of every tile; P as fp16 over its
//                   own S columns, zeros over the other parts'
//   O += P V        tcgen05.mma, A = P from tensor memory, B = the widened V
//                   tile (MN-major); O stays in tensor memory
//   epilogue        the four replicas of a head merged by their lse (shared
//                   memory), O / l; with two splits the two blocks of a kv
//                   head are a cluster and block 0 merges them (distributed
//                   shared memory), else split partials for the combine
// The reference maximum of a row moves only when its maximum grows by more
// than 2^8 (P stays below 256, O / l is unchanged). A uint8 cache takes the
// keys-on-rows kernel (attn_tc05_keys.cu), measured faster there: its
// per-key scales lengthen this layout's softmax chain.
//
// A one-token step is one launch (FUSE): the softmax warps rotate q_new and
// write q_rot, warp 11 encodes the new k / v row to e5m2 with the append
// kernel's encoder and the loaders wait for it only before the tile that holds
// that row.
//
// Warps: 0-3 softmax and epilogue, 4 K loader, 5 V loader (TMA, 3 stages
// each), 6 MMA issue (one thread) and tensor-memory allocation, 7-8 K
// converters, 9-10 V converters, 11 the fused step's append.
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
constexpr int kBM = 128;     // MMA rows: 32 head rows x 4 replicas
constexpr int kBN = 128;     // keys per tile
constexpr int kParts = 4;    // replicas of each head row; each takes a quarter of every tile
constexpr int kRPad = kBM / kParts;  // head rows per replica (32)
constexpr int kKW = kBN / kParts;    // keys of a tile per softmax thread (32)
constexpr int kStages = 3;   // code tiles in flight (K and V each)
// widened K tiles (measured: a second one, at the cost of a code stage, was
// slower: the three code stages keep more bytes in flight)
constexpr int kKOpB = 1;
constexpr int kSBuf = 3;     // S / P buffers in tensor memory
constexpr int kThreads = 384;
constexpr int kCodeStage = kBN * kD;                 // 16 KB: [128 rows][128 B], 128-byte swizzle
constexpr int kOpBytes = kBN * kD * 2;               // 32 KB fp16 tile: [2 halves][128 rows][128 B]
constexpr int kQOff = 0;
constexpr int kKCOff = kQOff + kOpBytes;             // K code stages
constexpr int kVCOff = kKCOff + kStages * kCodeStage;
constexpr int kKOpOff = kVCOff + kStages * kCodeStage;  // widened K [kKOpB]
constexpr int kVOpOff = kKOpOff + kKOpB * kOpBytes;     // widened V
constexpr int kBarOff = kVOpOff + kOpBytes;
constexpr int kSmemBytes = kBarOff + 512 + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColO = kSBuf * 128;
static_assert(kColO + kD <= kTmemCols, "S buffers and O exceed tensor memory");
static_assert(kKCOff % 1024 == 0 && kVCOff % 1024 == 0 && kKOpOff % 1024 == 0 && kVOpOff % 1024 == 0,
              "swizzled tiles start on 1 KB");
constexpr float kRescaleLog2 = 8.0f;
// epilogue: the replicas' merge area (the code stages and the widened K
// tiles: every tile has been widened and multiplied by then) and the
// two-block cluster exchange (the widened V tile)
constexpr int kMergeStride = kD + 4;
static_assert((kBM * kMergeStride + 3 * kBM) * 4 <= 2 * kStages * kCodeStage + kKOpB * kOpBytes, "merge area");
constexpr int kXRows = kRPad;
constexpr int kXOff = kVOpOff;
static_assert((kXRows * (kD + 3)) * 4 <= kOpBytes, "cluster exchange area");

// mbarriers (8 bytes each) at kBarOff
constexpr int kQReady = 0;
constexpr int kKFull = 1;                    // [kStages] K codes landed
constexpr int kKEmpty = kKFull + kStages;    // [kStages] ... read by the converters
constexpr int kVFull = kKEmpty + kStages;    // [kStages]
constexpr int kVEmpty = kVFull + kStages;    // [kStages]
constexpr int kKOpFull = kVEmpty + kStages;  // [kKOpB] widened K in shared memory
constexpr int kKOpEmpty = kKOpFull + kKOpB;  // [kKOpB] ... read by its S
constexpr int kVOpFull = kKOpEmpty + kKOpB;  // widened V
constexpr int kVOpEmpty = kVOpFull + 1;      // ... read by its PV
constexpr int kSFull = kVOpEmpty + 1;        // [kSBuf]
constexpr int kPFull = kSFull + kSBuf;       // [kSBuf]
constexpr int kODone = kPFull + kSBuf;       // [kSBuf]
constexpr int kDrain = kODone + kSBuf;
constexpr int kAppended = kDrain + 1;        // fused step: the new k / v codes are in the cache
constexpr int kNBars = kAppended + 1;
static_assert(kNBars * 8 + 4 <= 512, "barrier area");

// named barriers: 1 the softmax warps, 2 Q rows requested (softmax + loaders),
// 3 the fused step's cos / sin table (softmax warps)
constexpr int kBarSoftmax = 1, kBarQ = 2, kBarTable = 3;

__device__ __forceinline__ uint32_t sw128(int r, int col) {  // byte offset of 16-bit element (r, col) of a tile
  const int half = col >> 6, chunk = (col & 63) >> 3;
  return half * 16384 + r * 128 + ((chunk ^ (r & 7)) << 4) + (col & 7) * 2;
}

__device__ __forceinline__ bool aborted(const Tc05Params& p) {
  return (*reinterpret_cast<volatile int32_t*>(p.err) & static_cast<int>(MQA_DEVERR_TIMEOUT)) != 0;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Four e5m2 codes (bytes 0-3 of w, dims 0-3) as two fp16 pairs, dims (0, 1)
// and (2, 3), the lower dim in the low half: each byte as the high byte of a
// half, which is the e5m2 value exactly.
__device__ __forceinline__ void widen4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  lo = prmt(w, 0u, 0x1404u);
  hi = prmt(w, 0u, 0x3424u);
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// CL: the two splits of a (sequence, kv head) are one cluster of two blocks
// that merge their results through distributed shared memory; block 0 writes
// the output (no combine launch, no partials in global memory).
template <bool FUSE, bool CL>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc05_widen_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                           const Tc05Params p) {
  extern __shared__ unsigned char smem_raw[];
  // 1 KB aligned (128-byte swizzle atoms); offsetting the __shared__ array
  // itself keeps accesses through `smem` in the shared state space
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + kBarOff + kNBars * 8);
  __shared__ int s_abort, s_skip;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.group, S = p.num_splits;
  // block order: sequence fastest, then kv head, split; CL: the split (the
  // block's rank in its cluster) fastest
  int cta = blockIdx.x;
  int cl_rank = 0;
  if constexpr (CL) {
    cl_rank = cta & 1;
    cta >>= 1;
  }
  const int b = cta % p.batch;
  cta /= p.batch;
  const int j = cta % p.h_kv;
  const int split = CL ? cl_rank : cta / p.h_kv;
  const int rows = G;  // <= 32 head rows
  const long long row0 = static_cast<long long>(b) * p.h_q + j * G;  // output row of head 0 of the group

  long long limit = p.capacity < p.max_seq_len ? p.capacity : p.max_seq_len;
  int L = p.seq_lens[b];
  const int apos = FUSE ? p.pos[b] : 0;  // fused step: the new token's position
  if (L < 1 || L > limit) {
    // reported; the rows are then unspecified
    if (tid == 0 && split == 0 && j == 0) atomicOr(p.err, static_cast<int>(MQA_DEVERR_SEQ_LEN));
    L = L < 1 ? 1 : static_cast<int>(limit);
  }

  // CL: the exchange between the two blocks of the cluster. Every thread of
  // both blocks runs it exactly once, on every path through the kernel (the
  // cluster barriers have no timeout). Block 1 leaves (xo, xl) of its split
  // in its shared memory; block 0 reads them, merges them with its own by
  // their lse (as the combine does) and writes out and lse_out.
  float* xo = reinterpret_cast<float*>(smem + kXOff);  // [kXRows][kD]
  float* xl = xo + kXRows * kD;                         // [kXRows]
  float* xw = xl + kXRows;                              // [2][kXRows] (block 0)
  auto cl_exchange = [&]() {
    grid_dependency_wait();  // out may still be read by the preceding launch
    cluster_sync_all();
    if (cl_rank == 0) {
      const uint32_t peer = dsmem_map(smem_u32(xo), 1);
      if (tid < rows) {
        const float l0 = xl[tid], l1 = dsmem_ld_f32(peer + (kXRows * kD + tid) * 4);
        const float m = fmaxf(l0, l1);
        float w0 = 0.f, w1 = 0.f, lse = -INFINITY;
        if (m != -INFINITY) {
          w0 = expf(l0 - m);  // exp(-inf) = 0 for an empty split
          w1 = expf(l1 - m);
          lse = m + logf(w0 + w1);
          const float inv = 1.f / (w0 + w1);
          w0 *= inv;
          w1 *= inv;
        }
        xw[tid] = w0;
        xw[kXRows + tid] = w1;
        if (p.lse_out != nullptr) p.lse_out[row0 + tid] = lse;
      }
      __syncthreads();
      // four elements per item; the peer's loads of a batch in flight together
      constexpr int kBatch = 4;
      const int items = rows * (kD / 4);
      for (int i0 = tid; i0 < items; i0 += kBatch * kThreads) {
        float4 pv[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int it = i0 + u * kThreads;
          pv[u] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (it < items) pv[u] = dsmem_ld_f32x4(peer + it * 16);
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int it = i0 + u * kThreads;
          if (it >= items) break;
          const int r = it / (kD / 4), d = (it % (kD / 4)) * 4;
          const float wa = xw[r], wb = xw[kXRows + r];
          const float4 a = *reinterpret_cast<const float4*>(xo + r * kD + d);
          float v[4] = {0.f, 0.f, 0.f, 0.f};
          if (wa > 0.f) {  // an empty or skipped split's rows are never read
            v[0] = wa * a.x, v[1] = wa * a.y, v[2] = wa * a.z, v[3] = wa * a.w;
          }
          if (wb > 0.f) {
            v[0] = fmaf(wb, pv[u].x, v[0]), v[1] = fmaf(wb, pv[u].y, v[1]);
            v[2] = fmaf(wb, pv[u].z, v[2]), v[3] = fmaf(wb, pv[u].w, v[3]);
          }
          const long long o = (row0 + r) * kD + d;
          if (p.out_dtype == kDtypeBf16) {
            uint2 w;
            w.x = pack_bf16x2(v[0], v[1]);
            w.y = pack_bf16x2(v[2], v[3]);
            *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + o) = w;
          } else {
            *reinterpret_cast<float4*>(static_cast<float*>(p.out) + o) = make_float4(v[0], v[1], v[2], v[3]);
          }
        }
      }
    }
    cluster_sync_all();  // block 1's shared memory is kept until block 0 has read it
  };
  auto cl_empty = [&]() {  // a split with no result: weight 0 in the merge
    for (int r = tid; r < rows; r += kThreads) xl[r] = -INFINITY;
  };

  if (tid == 0) s_skip = aborted(p) ? 1 : 0;  // an earlier block timed out: the result is invalid already
  __syncthreads();
  if (s_skip) {
    if constexpr (CL) {
      cl_empty();
      cl_exchange();
    }
    return;
  }
  const int Lp = L - 1;  // the new token's position: keys [ka, Lp]
  const int ka = p.window > 0 ? max(0, Lp + 1 - p.window) : 0;
  // the split's token range (as the other decode kernels cut it)
  const int kstart = (ka / 64) * 64 + split * p.chunk;
  const int t_end = min(L, kstart + p.chunk);
  const int T = t_end > kstart ? (t_end - kstart + kBN - 1) / kBN : 0;  // key tiles of this block
  const bool split_out = S > 1 && !CL;
  // fused step: the split whose token range holds the new token's position
  // (else split 0) appends its k / v row
  const int tbase = (ka / 64) * 64;
  const bool writer =
      FUSE && split == ((apos - tbase >= 0 && (apos - tbase) / p.chunk < S) ? (apos - tbase) / p.chunk : 0);
  if (T == 0) {
    // no key of this split: an empty partial (weight 0 in the combine)
    grid_dependency_wait();
    if constexpr (CL) {
      cl_empty();
      cl_exchange();
      return;
    }
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
      mbar_init(bar(kKEmpty + s), 2);  // the two K converter warps
      mbar_init(bar(kVFull + s), 1);
      mbar_init(bar(kVEmpty + s), 2);  // the two V converter warps
    }
    for (int s = 0; s < kKOpB; ++s) {
      mbar_init(bar(kKOpFull + s), 2);
      mbar_init(bar(kKOpEmpty + s), 1);
    }
    mbar_init(bar(kVOpFull), 2);
    mbar_init(bar(kVOpEmpty), 1);
    for (int s = 0; s < kSBuf; ++s) {
      mbar_init(bar(kSFull + s), 1);
      mbar_init(bar(kPFull + s), 4);
      mbar_init(bar(kODone + s), 1);
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
    const int full = is_k ? kKFull : kVFull, empty = is_k ? kKEmpty : kVEmpty;
    const uint32_t dst0 = sbase + (is_k ? kKCOff : kVCOff);
    const int row = b * p.h_kv + j;
    auto issue = [&](int it) {
      const int s = it % kStages, tok = kstart + it * kBN;
      const uint32_t dst = dst0 + s * kCodeStage;
      mbar_arrive_expect_tx(bar(full + s), kCodeStage);
      tma_load_3d(dst, map, 0, tok, row, bar(full + s));
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
    named_bar_sync(kBarQ, kBM + 64);
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
      const uint32_t id_s = tc05::idesc_f16_f32(kBM, kBN, false, false);  // Q x K, both K-major
      const uint32_t id_o = tc05::idesc_f16_f32(kBM, kD, false, true);    // P (tensor memory) x V (MN-major)
      const uint32_t q_s = sbase + kQOff, v_s = sbase + kVOpOff;
      bool ok = mbar_wait(bar(kQReady), 0);
      // S of tile it into buffer it % kSBuf. That buffer last held P of tile
      // it - kSBuf, whose PV was issued before: MMAs of this thread execute in order.
      auto issue_s = [&](int it) {
        const int sb = it % kSBuf, kb = it % kKOpB;
        const uint32_t k_s = sbase + kKOpOff + kb * kOpBytes;
        tc05::fence_after_sync();
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
          const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
          tc05::mma_bf16(tmem + kColS + sb * 128, tc05::smem_desc_sw128(q_s + off, 16, 1024),
                         tc05::smem_desc_sw128(k_s + off, 16, 1024), id_s, ks > 0);
        }
        tc05::commit(bar(kSFull + sb));
        tc05::commit(bar(kKOpEmpty + kb));
      };
      auto issue_pv = [&](int it) {
        const int pb = it % kSBuf;
        tc05::fence_after_sync();
#pragma unroll
        for (int ks = 0; ks < kBN / 16; ++ks)
          tc05::mma_bf16_ta(tmem + kColO, tmem + kColS + pb * 128 + ks * 8,
                            tc05::smem_desc_sw128(v_s + ks * 2048, 16384, 1024), id_o, it > 0 || ks > 0);
        tc05::commit(bar(kODone + pb));
        tc05::commit(bar(kVOpEmpty));
      };
      // Issue S and PV as their inputs land: S of tile ns needs its widened K
      // tile and (buffer reuse) the PV of tile ns - kSBuf issued; PV of tile
      // np needs its P and widened V tile. Neither waits behind the other.
      int ns = 0, np = 0;
      unsigned long long t_idle = global_timer_ns();
      while (ok && np < T) {
        bool progress = false;
        if (ns < T && ns <= np + (kSBuf - 1) && mbar_test(bar(kKOpFull + ns % kKOpB), (ns / kKOpB) & 1)) {
          issue_s(ns++);
          progress = true;
        }
        if (np < ns && mbar_test(bar(kPFull + np % kSBuf), (np / kSBuf) & 1) && mbar_test(bar(kVOpFull), np & 1)) {
          issue_pv(np++);
          progress = true;
        }
        if (progress) {
          t_idle = global_timer_ns();
        } else if (stop() || global_timer_ns() - t_idle > kWaitLimitNs) {
          ok = false;
        } else {
          __nanosleep(32);  // leave the issue slots to the softmax warp sharing this scheduler
        }
      }
      if (!ok) fail(1);
    }
    __syncwarp();
  } else if (warp == 11) {
    // ------------------------------------------------------ append (fused step)
    // the new token's cache row exactly as the append kernel writes it: k pair
    // i turned in fp64 (fp64 sine and cosine of the reduced angle,
    // round-to-nearest products) and v, each rounded once to e5m2; a position
    // outside the cache is reported and nothing is written. Fenced for the
    // loaders' TMA reads (async proxy), which wait for it only before the tile
    // that holds the row.
    if (writer) {
      long long row = -1;
      if (apos >= 0 && apos < p.capacity)
        row = ((static_cast<long long>(b) * p.h_kv + j) * p.capacity + apos) * kD;
      else if (lane == 0)
        atomicOr(p.err, static_cast<int>(MQA_DEVERR_POS_RANGE));
      append_row_q<kD, true>(p, b, j, apos, row, lane);
      if (lane == 0) mbar_arrive(bar(kAppended));
    }
  } else if (warp >= 7) {
    // ------------------------------------------- converters: warps 7-8 K, 9-10 V
    // Each widens rows ct and ct + 64 of its tiles. K and V have their own
    // warps, so that the widening of K tile it + 1 (which S of tile it frees)
    // never waits behind the PV of tile it - 1 (which frees the V tile).
    const bool is_k = warp < 9;
    const int ct0 = 32 * ((warp - 7) & 1) + lane;
    const int code_full = is_k ? kKFull : kVFull, code_empty = is_k ? kKEmpty : kVEmpty;
    const int code_off = is_k ? kKCOff : kVCOff;
    const int n_op = is_k ? kKOpB : 1;  // widened tiles of this side
    for (int it = 0; it < T; ++it) {
      const int s = it % kStages;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(code_full + s), (it / kStages) & 1) && !stop())) {
        if (lane == 0) fail(1);
        break;
      }
      const unsigned char* cs = smem + code_off + s * kCodeStage;
      uint4 cr[2][8];  // codes of dims 16 c .. 16 c + 15 of the two rows
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int ct = ct0 + 64 * h;
#pragma unroll
        for (int c = 0; c < 8; ++c) cr[h][c] = *reinterpret_cast<const uint4*>(cs + ct * 128 + ((c ^ (ct & 7)) << 4));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(code_empty + s));
      // rows past the split may hold anything (past the sequence any bit
      // pattern, NaN and infinity codes included): they become zero rows
      bool past[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) past[h] = kstart + it * kBN + ct0 + 64 * h >= t_end;
      // widened into the swizzled operand tile (row = key)
      const int ob = it % n_op;
      const int op_full = (is_k ? kKOpFull : kVOpFull) + ob, op_empty = (is_k ? kKOpEmpty : kVOpEmpty) + ob;
      unsigned char* op = smem + (is_k ? kKOpOff : kVOpOff) + ob * kOpBytes;
      if (it >= n_op && !__all_sync(0xffffffffu, mbar_wait(bar(op_empty), ((it - n_op) / n_op) & 1))) {
        if (lane == 0) fail(1);
        break;
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int ct = ct0 + 64 * h, sw = ct & 7;
        unsigned char* orow = op + ct * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {  // codes of dims 16c .. 16c + 15: two 16-byte chunks of fp16
          const uint4 w = cr[h][c];
          uint4 o0 = make_uint4(0u, 0u, 0u, 0u), o1 = make_uint4(0u, 0u, 0u, 0u);
          if (!past[h]) {
            widen4(w.x, o0.x, o0.y);
            widen4(w.y, o0.z, o0.w);
            widen4(w.z, o1.x, o1.y);
            widen4(w.w, o1.z, o1.w);
          }
          const int half = c >> 2, cc = 2 * (c & 3);
          *reinterpret_cast<uint4*>(orow + half * 16384 + ((cc ^ sw) << 4)) = o0;
          *reinterpret_cast<uint4*>(orow + half * 16384 + (((cc + 1) ^ sw) << 4)) = o1;
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(op_full));
    }
  } else {
    // --------------------------------------------------- softmax (row = tid)
    const int r = tid;
    const int part = r / kRPad, gr = r - part * kRPad;  // key quarter and head row of this thread
    const bool live = gr < rows;
    {
      // Q row (head gr, replica `part`), pre-scaled into the log2 domain, as
      // fp16 in the swizzled tile. The whole row is requested at once, and
      // the loaders are released only then: behind their burst of tile
      // requests these loads would wait microseconds.
      float4 qv[kD / 4];
      if constexpr (FUSE) {
        // fused step: q_new (bf16) rotated here, pair i by the fp32 cosine /
        // sine of the fp64-reduced angle pos * theta_i, as the other fused
        // kernels form q_rot
        __shared__ float s_cs[kD];
        const uint4* qn = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.q_new) + (row0 + gr) * kD);
        uint4 raw[kD / 8];
#pragma unroll
        for (int c = 0; c < kD / 8; ++c) raw[c] = live ? qn[c] : make_uint4(0u, 0u, 0u, 0u);
        named_bar_arrive(kBarQ, kBM + 64);
        if (tid < kD / 2) {
          const double ang = reduce_two_pi(static_cast<double>(apos) * p.theta[tid]);
          float sf, cf;
          sincosf(static_cast<float>(ang), &sf, &cf);
          s_cs[tid] = cf;
          s_cs[kD / 2 + tid] = sf;
        }
        named_bar_sync(kBarTable, kBM);
#pragma unroll
        for (int c = 0; c < kD / 8; ++c) {
          const uint32_t w4[4] = {raw[c].x, raw[c].y, raw[c].z, raw[c].w};
          float rv[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int pi = 4 * c + e;  // pair (2 pi, 2 pi + 1)
            const float x = bf16lo_to_f32(w4[e]), y = bf16hi_to_f32(w4[e]);
            const float cs = s_cs[pi], sn = s_cs[kD / 2 + pi];
            rv[2 * e] = x * cs - y * sn;
            rv[2 * e + 1] = x * sn + y * cs;
          }
          qv[2 * c] = make_float4(rv[0], rv[1], rv[2], rv[3]);
          qv[2 * c + 1] = make_float4(rv[4], rv[5], rv[6], rv[7]);
        }
        if (live && part == 0 && split == 0) {  // one copy of each row to q_rot
          float4* qo = reinterpret_cast<float4*>(p.q_rot_out + (row0 + gr) * kD);
#pragma unroll
          for (int c = 0; c < kD / 4; ++c) qo[c] = qv[c];
        }
      } else {
        if (p.early) grid_dependency_wait();  // q_rot comes from the append kernel
        const float4* q = reinterpret_cast<const float4*>(p.q_rot + (row0 + gr) * kD);
#pragma unroll
        for (int c = 0; c < kD / 4; ++c) qv[c] = live ? q[c] : make_float4(0.f, 0.f, 0.f, 0.f);
        named_bar_arrive(kBarQ, kBM + 64);
      }
#pragma unroll
      for (int c = 0; c < kD; c += 8) {
        const float4 a = qv[c / 4], bq = qv[c / 4 + 1];
        uint4 v;
        v.x = pack_half2(a.x * p.scale_log2, a.y * p.scale_log2);
        v.y = pack_half2(a.z * p.scale_log2, a.w * p.scale_log2);
        v.z = pack_half2(bq.x * p.scale_log2, bq.y * p.scale_log2);
        v.w = pack_half2(bq.z * p.scale_log2, bq.w * p.scale_log2);
        *reinterpret_cast<uint4*>(smem + kQOff + sw128(r, c)) = v;
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kQReady));
    }
    const int pos = live ? min(Lp, t_end - 1) : -1;  // last key of this row in the split (none: padding)
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int it = 0; it < T; ++it) {
      const int sb = it % kSBuf;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(kSFull + sb), (it / kSBuf) & 1) && !stop());
      if (!ok) break;
      tc05::fence_after_sync();
      float s[kKW];
      tc05::ld_32x32b_x32(tmem + lane_base + kColS + sb * 128 + part * kKW, s);
      tc05::wait_ld();
      tc05::reg_fence(s);
      // keys of this tile outside [ka, pos] are masked
      const int kk0 = kstart + it * kBN + part * kKW;  // first key of this thread's slice
      if (kk0 < ka || kk0 + kKW - 1 > pos) {
#pragma unroll
        for (int c = 0; c < kKW; ++c)
          if (kk0 + c < ka || kk0 + c > pos) s[c] = -INFINITY;
      }
      float mx8[8];  // eight independent chains
#pragma unroll
      for (int i = 0; i < 8; ++i) mx8[i] = s[i];
#pragma unroll
      for (int c = 8; c < kKW; c += 8) {
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(mx8[i], s[c + i]);
      }
      const float mt = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      // a new reference maximum only when the row's maximum grew by more than 2^8
      const bool grow = mt > m_ref + kRescaleLog2 || (m_ref == -INFINITY && mt != -INFINITY);
      const float m_new = grow ? mt : m_ref;
      if (it > 0 && __any_sync(0xffffffffu, grow && m_ref != -INFINITY)) {
        // O is rescaled: PV of the previous tile must be done first
        ok = __all_sync(0xffffffffu, mbar_wait(bar(kODone + (it - 1) % kSBuf), ((it - 1) / kSBuf) & 1) && !stop());
        if (!ok) break;
        tc05::fence_after_sync();
        const float alpha = (grow && m_ref != -INFINITY) ? fast_exp2(m_ref - m_new) : 1.f;
#pragma unroll
        for (int c = 0; c < kD / 32; ++c) {
          float v[32];
          tc05::ld_32x32b_x32(tmem + lane_base + kColO + c * 32, v);
          tc05::wait_ld();
          tc05::reg_fence(v);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= alpha;
          tc05::st_32x32b_x32(tmem + lane_base + kColO + c * 32, v);
        }
        l *= alpha;
      }
      m_ref = m_new;
      const float e = m_ref == -INFINITY ? 0.f : m_ref;
      float sm8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      // P of this thread's keys as fp16 pairs over its own S columns; the
      // other parts' columns of this row carry zeros
      uint32_t pk[kKW / 2];
#pragma unroll
      for (int i = 0; i < kKW / 2; ++i) {
        const float p0 = fast_exp2(s[2 * i] - e), p1 = fast_exp2(s[2 * i + 1] - e);
        sm8[(2 * i) & 7] += p0;
        sm8[(2 * i + 1) & 7] += p1;
        pk[i] = pack_half2(p0, p1);
      }
      const uint32_t prow = tmem + lane_base + kColS + sb * 128;
      uint32_t z[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) z[i] = 0u;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        if (q4 == part)
          tc05::st_32x32b_x16_u(prow + 16 * q4, pk);
        else
          tc05::st_32x32b_x16_u(prow + 16 * q4, z);
      }
      l += ((sm8[0] + sm8[1]) + (sm8[2] + sm8[3])) + ((sm8[4] + sm8[5]) + (sm8[6] + sm8[7]));
      tc05::wait_st();
      tc05::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kPFull + sb));
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(kODone + (T - 1) % kSBuf), ((T - 1) / kSBuf) & 1));
    if (!ok && lane == 0) fail(1);
    if (ok) tc05::fence_after_sync();
    // ---- merge the four replicas of each head row through shared memory
    // (the code stages and widened K tiles: every tile is done by now)
    float* mo = reinterpret_cast<float*>(smem + kKCOff);  // [128][kMergeStride] unnormalised O
    float* mm = mo + kBM * kMergeStride;                   // [128] reference maxima
    float* ml = mm + kBM;                                  // [128] sums
    if (ok) {
#pragma unroll
      for (int c = 0; c < kD / 32; ++c) {
        float v[32];
        tc05::ld_32x32b_x32(tmem + lane_base + kColO + c * 32, v);
        tc05::wait_ld();
        tc05::reg_fence(v);
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          *reinterpret_cast<float4*>(mo + r * kMergeStride + c * 32 + i) =
              make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
      }
      mm[r] = m_ref;
      ml[r] = l;
    }
    // every softmax warp arrives, also after a timeout (which set s_abort first)
    named_bar_sync(kBarSoftmax, kBM);
    // thread r < rows: the weight of each replica in row r (its partial
    // softmax renormalised to the row's maximum and divided by the row's
    // total) and the row's lse
    float* mw = ml + kBM;  // [kParts][kRPad]
    if (r < rows && !stop()) {
      float mx = -INFINITY;
#pragma unroll
      for (int q = 0; q < kParts; ++q) mx = fmaxf(mx, mm[q * kRPad + r]);
      float w[kParts], den = 0.f;
#pragma unroll
      for (int q = 0; q < kParts; ++q) {
        w[q] = mx == -INFINITY ? 0.f : exp2f(mm[q * kRPad + r] - mx);
        den = fmaf(w[q], ml[q * kRPad + r], den);
      }
      const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
      for (int q = 0; q < kParts; ++q) mw[q * kRPad + r] = w[q] * inv;
      const float lse = den > 0.f ? (mx + log2f(den)) * 0.69314718055994530942f : -INFINITY;
      if constexpr (CL)
        xl[r] = lse;
      else if (split_out)
        p.lse_part[(row0 + r) * S + split] = lse;
      else if (p.lse_out != nullptr)
        p.lse_out[row0 + r] = lse;
    }
    named_bar_sync(kBarSoftmax, kBM);
    // thread = head dim: every row's output element, rows independent
    const int d = r;
    if (!stop()) {
#pragma unroll 4
      for (int row = 0; row < rows; ++row) {
        float ov = 0.f;
#pragma unroll
        for (int q = 0; q < kParts; ++q) ov = fmaf(mw[q * kRPad + row], mo[(q * kRPad + row) * kMergeStride + d], ov);
        const long long orow = row0 + row;
        if constexpr (CL) {
          xo[row * kD + d] = ov;
        } else if (split_out) {
          p.o_part[(orow * S + split) * kD + d] = ov;
        } else if (p.out_dtype == kDtypeBf16) {
          static_cast<__nv_bfloat16*>(p.out)[orow * kD + d] = __float2bfloat16_rn(ov);
        } else {
          static_cast<float*>(p.out)[orow * kD + d] = ov;
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
  if constexpr (CL) cl_exchange();
}

template <bool FUSE, bool CL>
cudaError_t launch_widen(const Tc05Params& p, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream) {
  auto kern = attn_tc05_widen_kernel<FUSE, CL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.batch) * p.h_kv * p.num_splits);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (CL) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  return cudaLaunchKernelEx(&cfg, kern, tk, tv, p);
}

}  // namespace

KernelShape tc05_widen_shape() { return {kThreads, kSmemBytes, kRPad, 1}; }

bool tc05_widen_merges_splits(const Tc05Params& p) { return p.num_splits == 2; }

cudaError_t launch_tc05_widen_attention(const Tc05Params& p, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                                        cudaStream_t stream) {
  const bool cl = tc05_widen_merges_splits(p);
  if (p.fuse) return cl ? launch_widen<true, true>(p, tmap_k, tmap_v, stream) : launch_widen<true, false>(p, tmap_k, tmap_v, stream);
  return cl ? launch_widen<false, true>(p, tmap_k, tmap_v, stream) : launch_widen<false, false>(p, tmap_k, tmap_v, stream);
}

}  // namespace mqa
