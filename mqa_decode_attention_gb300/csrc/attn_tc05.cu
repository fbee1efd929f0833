// Attention of the last n_new tokens of every sequence on the 5th-generation
// tensor cores: prefill ("KV Cache" explainer, Langkah 1 and 4: the prompt's
// keys and values are computed in one pass and stored, and the work is
// compute-bound), and decode steps with many query rows per kv head (MQA,
// G = 32; several new tokens per sequence).
//
// The rows of kv head j are its (new token i, query head h = j G + hl) pairs,
// row = i G + hl, in blocks of 128. Block = (sequence b, kv head j, token-axis
// split, row block). Row (i, hl), at position p = L - n_new + i, attends to the
// keys [max(0, p + 1 - W) if windowed else 0, p] that fall in the split's
// range. For each 128-key tile of the block's range:
//   S = Q K^T      tcgen05.mma M=128 N=128 K=128, Q and K from shared memory,
//                  S (f32) into tensor memory
//   online softmax one row per thread of warps 0-3 (tcgen05.ld of the row);
//                  P (bf16) written back over its own S columns (tcgen05.st)
//   O += P V       tcgen05.mma with A = P read from tensor memory, V from
//                  shared memory; O stays in tensor memory
// with the running maximum of FlashAttention ("Arsitektur Inferensi LLM",
// section 5). S is double-buffered in tensor memory so the tensor core
// computes S of the next tile while the softmax works on this one; O is only
// rescaled when a row's maximum grows by more than 2^8 (the exponentials are
// taken against a reference at most 8 below the true maximum, so P stays
// below 256 and the final O / l is unchanged).
//
// With few rows per kv head (R <= 64: MQA's 32 query heads; a few new tokens
// of a GQA group) the R rows are replicated PARTS = 128 / R_pad times over the
// MMA's 128 rows and the softmax warps split every key tile: thread r (part
// r / R_pad) keeps the online softmax of row r % R_pad over its 128 / PARTS
// keys of each tile, its P row holds zeros over the other keys, and the
// partial results of a row are merged (log-sum-exp weights) at the end.
//
// Warps: 0-3 softmax and epilogue (row = thread), 4 K loader, 5 V loader
// (TMA, 3 stages each; a K stage is released when its S is computed, a V
// stage when its PV is), 6 MMA issue (one thread) and tensor-memory
// allocation, 7 the fused step's append (its own warp, so that the block
// that writes the new rows publishes Q as early as the others).
#include <cuda_bf16.h>

#include "../../include/mqa_decode.h"
#include "launch.h"
#include "ptx.cuh"
#include "rope.cuh"
#include "tc05.cuh"

namespace mqa {
namespace {

constexpr int kD = 128;       // head_dim
constexpr int kBM = 128;      // query rows (tokens of one head) per block
constexpr int kBN = 128;      // keys per tile
constexpr int kThreads = 256;
constexpr int kSBuf = 3;                                 // S / P buffers in tensor memory
constexpr uint32_t kTmemCols = 512;                      // S0 .. S{kSBuf-1}, O
constexpr uint32_t kColS = 0, kColO = kSBuf * 128;
static_assert(kColO + kD <= kTmemCols, "S buffers and O exceed tensor memory");
constexpr float kRescaleLog2 = 8.0f;
// In the fused step the loaders request this many tiles before the Q rows
// have landed, the rest after (other steps: before the Q rows are requested): a full ring of tile requests ahead of the Q reads delays them by
// microseconds, none at all leaves the memory idle meanwhile (mqa8k, same-box
// A/B: 2 tiles then Q 53.3 / 48.0 us isolated / back to back, 3 tiles with Q
// requested 53.3 / 48.1, no tile 55.5 / 49.4).
constexpr int kPreTiles = 2;
// two-split cluster (CL): each block's normalised output rows (fp32) and their
// lse, left in its V stages once its last PV is done
constexpr int kXRows = 64;
// F8 (fp8 e5m2 cache): Q and P enter the MMAs as e4m3 pairs hi + lo, Q scaled
// by 2^6 first (its values then sit in e4m3's normal range); the scores come
// out 2^6 too large and are scaled back exactly
constexpr float kQScaleF8 = 64.f;

// Shared memory and mbarriers. bf16 cache: Q [2 halves][128 rows][128 B], K
// and V tiles of 32 KB, three stages each. fp8 e5m2 cache (F8): Q as two
// 16 KB e4m3 tiles (hi, lo) [128 rows][128 B], K and V code tiles of 16 KB
// (128 keys x 128 one-byte values, as TMA lands them), six stages each: the
// same bytes in flight.
template <bool F8>
struct Lay {
  static constexpr int kStages = F8 ? 6 : 3;
  static constexpr int kTileBytes = F8 ? kBN * kD : kBN * kD * 2;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = 32768;
  static constexpr int kVOff = kKOff + kStages * kTileBytes;
  static constexpr int kBarOff = kVOff + kStages * kTileBytes;
  static constexpr int kSmemBytes = kBarOff + 512 + 1024;
  static constexpr int kXOff = kVOff;
  // mbarriers (8 bytes each) at kBarOff
  static constexpr int kQReady = 0;
  static constexpr int kKFull = 1;                   // [kStages]
  static constexpr int kKEmpty = kKFull + kStages;   // [kStages]
  static constexpr int kVFull = kKEmpty + kStages;   // [kStages]
  static constexpr int kVEmpty = kVFull + kStages;   // [kStages]
  static constexpr int kSFull = kVEmpty + kStages;   // [kSBuf]
  static constexpr int kPFull = kSFull + kSBuf;      // [kSBuf]
  static constexpr int kODone = kPFull + kSBuf;      // [kSBuf]
  static constexpr int kDrain = kODone + kSBuf;
  static constexpr int kAppended = kDrain + 1;       // fused step: the new k / v row is in the cache
  static constexpr int kQStage = kAppended + 1;      // q_tma: the query rows' two boxes landed
  static constexpr int kNBars = kQStage + 1;
  static_assert(kNBars * 8 + 4 <= 512, "barrier area");
  static_assert((kXRows * (kD + 3)) * 4 <= kStages * kTileBytes, "cluster exchange area");
  static_assert((kBM * (kD + 4) + 3 * kBM) * 4 <= kStages * kTileBytes, "replica merge area (the K stages)");
  static_assert(kKOff >= kD * kBM * 2, "Q area");
};
static_assert(Lay<true>::kSmemBytes <= Lay<false>::kSmemBytes, "the bf16 layout is the larger one");

// e4m3_split4 out of line: the Q rows are split once per launch, and 32
// inlined copies of the code would only be cold instruction-cache misses.
__device__ __noinline__ uint2 e4m3_split4_once(float a, float b, float c, float d) {
  uint2 r;
  tc05::e4m3_split4(a, b, c, d, r.x, r.y);
  return r;
}

// The two stages of rope_k_bf16 for one packed bf16 pair, out of line: the
// fused step's append runs them a few times per block, and inlined copies
// would sit as cold code beside the softmax loop. The fp32 stage returns
// false when it leaves the rounding to the fp64 stage.
__device__ __noinline__ bool rope_k_packed_fast(uint32_t kp, double ang, uint32_t* out) {
  const float x = bf16lo_to_f32(kp), y = bf16hi_to_f32(kp);
  const float s = fabsf(x) + fabsf(y);
  if (!(s >= 0x1p-100f && s <= 1e37f)) return false;
  float sf, cf;
  sincosf(static_cast<float>(ang), &sf, &cf);
  __nv_bfloat162 r;
  if (!rope_k_bf16_fast(x, y, cf, sf, &r)) return false;
  *out = *reinterpret_cast<const uint32_t*>(&r);
  return true;
}
__device__ __noinline__ uint32_t rope_k_packed_fp64(uint32_t kp, double ang) {
  const __nv_bfloat162 r = rope_k_bf16_fp64(bf16lo_to_f32(kp), bf16hi_to_f32(kp), ang);
  return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t sw128(int r, int col) {  // byte offset of bf16 element (r, col) of a tile
  const int half = col >> 6, chunk = (col & 63) >> 3;
  return half * 16384 + r * 128 + ((chunk ^ (r & 7)) << 4) + (col & 7) * 2;
}

// CL: the two splits of a (sequence, kv head) are one cluster of two blocks
// that merge their partial results through distributed shared memory; block
// 0 writes the output (no combine launch, no partials in global memory).
// F8: fp8 e5m2 cache (the tensor maps describe the one-byte code tiles).
// PG: paged bf16 cache (PagedAttention, "Arsitektur Inferensi LLM", section
// 4): pages [num_pages, h_kv, page_size, 128] through the block table; a key
// tile is gathered page by page (rp = min(page_size, 64) rows per copy: the
// tiles start on multiples of 64, so a 64-key half never straddles a page).
template <int PARTS, bool FUSE, bool CL, bool F8, bool PG>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc05_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                     const __grid_constant__ CUtensorMap tmap_q, const Tc05Params p) {
  static_assert(!CL || PARTS > 1, "the cluster merge takes replicated rows (R <= 64)");
  static_assert(!(FUSE && F8), "the fused step is bf16 only");
  static_assert(!(PG && F8), "paged caches: bf16 only");
  using Y = Lay<F8>;
  constexpr int kStages = Y::kStages, kTileBytes = Y::kTileBytes, kQOff = Y::kQOff, kKOff = Y::kKOff,
                kVOff = Y::kVOff, kBarOff = Y::kBarOff, kXOff = Y::kXOff;
  constexpr int kQReady = Y::kQReady, kKFull = Y::kKFull, kKEmpty = Y::kKEmpty, kVFull = Y::kVFull,
                kVEmpty = Y::kVEmpty, kSFull = Y::kSFull, kPFull = Y::kPFull, kODone = Y::kODone,
                kDrain = Y::kDrain, kAppended = Y::kAppended, kQStage = Y::kQStage, kNBars = Y::kNBars;
  constexpr int kRPad = kBM / PARTS;  // rows per part
  constexpr int kKW = kBN / PARTS;    // keys of a tile per thread
  extern __shared__ unsigned char smem_raw[];
  // 1 KB aligned (128-byte swizzle atoms); offsetting the __shared__ array
  // itself keeps accesses through `smem` in the shared state space
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + kBarOff + kNBars * 8);
  __shared__ int s_abort, s_skip;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.group, n = p.n_new, R = G * n, S = p.num_splits;
  // block order: sequence fastest, then kv head, split, row block (row blocks
  // with the longest key ranges -- the last tokens -- first); CL: the split
  // (the block's rank in its cluster) fastest
  int cta = blockIdx.x;
  int cl_rank = 0;
  if constexpr (CL) {
    cl_rank = cta & 1;
    cta >>= 1;
  }
  const int b = cta % p.batch;
  cta /= p.batch;
  const int j = cta % p.h_kv;
  cta /= p.h_kv;
  const int split = CL ? cl_rank : cta % S;
  const int rb = CL ? 0 : p.row_blocks - 1 - cta / S;
  const int g0 = rb * kBM;
  const int rows = min(kBM, R - g0);

  long long limit = p.capacity < p.max_seq_len ? p.capacity : p.max_seq_len;
  // the length, the new position and the error word, requested together
  int L = p.seq_lens[b];
  const int apos = FUSE ? p.pos[b] : 0;  // fused step: the new token's position
  const int err0 = tid == 0 ? *reinterpret_cast<volatile int32_t*>(p.err) : 0;
  if (L < n || L > limit) {
    // reported; these rows are then unspecified, but the block still runs (a
    // fused step's append and q_rot land as they would without the error)
    if (tid == 0 && split == 0 && rb == 0 && j == 0) atomicOr(p.err, static_cast<int>(MQA_DEVERR_SEQ_LEN));
    L = L < n ? n : static_cast<int>(limit);
  }
  // CL: the exchange between the two blocks of the cluster. Every thread of
  // both blocks runs it exactly once, on every path through the kernel (the
  // cluster barriers have no timeout). Block 1 leaves (xo, xl) of its split
  // in its shared memory; block 0 reads them, merges them with its own by
  // their lse (as the combine does) and writes out and lse_out.
  float* xo = reinterpret_cast<float*>(smem + kXOff);  // [kXRows][kD]
  float* xl = xo + kXRows * kD;                         // [kXRows]
  float* xw = xl + kXRows;                              // [2][kXRows] (block 0)
  auto out_row = [&](int r) {
    const int i = (g0 + r) / G;
    return (static_cast<long long>(b) * n + i) * p.h_q + j * G + (g0 + r - i * G);
  };
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
        if (p.lse_out != nullptr) p.lse_out[out_row(tid)] = lse;
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
          const long long o = out_row(r) * kD + d;
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

  // an earlier block timed out: the result is invalid already
  if (tid == 0) s_skip = (err0 & static_cast<int>(MQA_DEVERR_TIMEOUT)) ? 1 : 0;
  __syncthreads();
  if (s_skip) {
    if constexpr (CL) {
      cl_empty();
      cl_exchange();
    }
    return;
  }
  const int Lp = L - n;  // new token i sits at position Lp + i
  const int pos_first = Lp + g0 / G, pos_last = Lp + (g0 + rows - 1) / G;
  const int ka_first = p.window > 0 ? max(0, pos_first + 1 - p.window) : 0;
  // the split's token range (as the other decode kernels cut it)
  const int t_lo = p.window > 0 ? max(0, Lp + 1 - p.window) : 0;
  const int t_begin = (t_lo / 64) * 64 + split * p.chunk;
  const int t_end = min(L, t_begin + p.chunk);
  const int kstart = max(t_begin, (ka_first / 64) * 64);
  const int kend = min(t_end, pos_last + 1);
  const int T = kend > kstart ? (kend - kstart + kBN - 1) / kBN : 0;  // key tiles of this block
  auto tile_key0 = [&](int it) { return kstart + it * kBN; };
  const bool split_out = S > 1 && !CL;
  // fused step: new token i (position apos + i) is appended by the split whose
  // token range holds it (else split 0), so that no block reads a row another
  // block writes (a fused step has one row block); a_first is this block's
  // first such token, a_pos its position
  const int tbase = (t_lo / 64) * 64;
  auto owner = [&](int i) {
    const int o = apos + i - tbase;
    return (o >= 0 && o / p.chunk < S) ? o / p.chunk : 0;
  };
  int a_first = -1;
  if constexpr (FUSE) {
    for (int i = n - 1; i >= 0; --i)
      if (owner(i) == split) a_first = i;
  }
  const bool writer = a_first >= 0;
  const int a_pos = apos + (writer ? a_first : 0);
  // the new tokens' cache rows exactly as the append kernel writes them: k
  // pair i turned and rounded once to bf16 (rope_k_bf16, equal to the fp64
  // rotation), v copied; a position outside the cache is reported and nothing
  // is written there. Then fenced for this block's TMA loads (async proxy).
  // The rows of kU tokens are requested together (one memory round trip per
  // kU tokens, not per token), and the pairs the fp32 stage of rope_k_bf16
  // leaves open are collected and finished in fp64 at the end, every lane at
  // once: a lane's open pair no longer stalls the whole warp on its own.
  const int32_t* trow = PG ? p.block_table + static_cast<long long>(b) * p.max_pages : nullptr;
  auto append_rows = [&]() {
    constexpr int kU = 2;  // (mqa8k, same-box A/B: 2 tokens 56.1 / 48.4 us isolated / back to back, 4: 61.4 / 49.3)
    __nv_bfloat16* kc = static_cast<__nv_bfloat16*>(const_cast<void*>(p.k_cache));
    __nv_bfloat16* vc = static_cast<__nv_bfloat16*>(const_cast<void*>(p.v_cache));
    const __nv_bfloat16* kn = static_cast<const __nv_bfloat16*>(p.k_new);
    const __nv_bfloat16* vn = static_cast<const __nv_bfloat16*>(p.v_new);
    bool bad_pos = false, bad_page = false;
    static_assert(2 * kMaxNewTokens <= 64, "the open-pair mask");
    uint64_t open = 0;  // bit 2 i + h: pair lane + 32 h of new token i left to the fp64 stage
    // the page of position ap (paged; entry checked by the caller)
    auto page_at = [&](int ap) { return PG ? __ldg(trow + ap / p.page_size) : 0; };
    auto dst_of = [&](int i, int page) -> long long {  // element offset of new token i's cache row
      const int ap = apos + i;
      if constexpr (PG)
        return ((static_cast<long long>(page) * p.h_kv + j) * p.page_size + (ap & (p.page_size - 1))) * kD;
      else
        return ((static_cast<long long>(b) * p.h_kv + j) * p.capacity + ap) * kD;
    };
    auto src_of = [&](int i) { return ((static_cast<long long>(b) * n + i) * p.h_kv + j) * kD; };
    for (int i0 = a_first; i0 < n; i0 += kU) {
      uint32_t kraw[kU][kD / 64], vraw[kU][kD / 64];
      int pg[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = i0 + u;
        if (i >= n || owner(i) != split || apos + i < 0 || apos + i >= p.capacity) continue;
        pg[u] = page_at(apos + i);
        const long long src = src_of(i);
#pragma unroll
        for (int h = 0; h < kD / 64; ++h) {  // pairs lane, lane + 32
          const int pi = lane + 32 * h;
          kraw[u][h] = *reinterpret_cast<const uint32_t*>(kn + src + 2 * pi);
          vraw[u][h] = *reinterpret_cast<const uint32_t*>(vn + src + 2 * pi);
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = i0 + u, ap = apos + i;
        if (i >= n || owner(i) != split) continue;
        if (ap < 0 || ap >= p.capacity) {
          bad_pos = true;
          continue;
        }
        if (PG && (pg[u] < 0 || pg[u] >= p.num_pages)) {
          bad_page = true;
          continue;
        }
        const long long dst = dst_of(i, pg[u]);
#pragma unroll
        for (int h = 0; h < kD / 64; ++h) {
          const int pi = lane + 32 * h;
          const double ang = reduce_two_pi(static_cast<double>(ap) * p.theta[pi]);
          uint32_t kr;
          if (rope_k_packed_fast(kraw[u][h], ang, &kr))
            *reinterpret_cast<uint32_t*>(kc + dst + 2 * pi) = kr;
          else
            open |= 1ull << (2 * i + h);
          *reinterpret_cast<uint32_t*>(vc + dst + 2 * pi) = vraw[u][h];
        }
      }
    }
    while (__any_sync(0xffffffffu, open != 0)) {
      if (open != 0) {
        const int bit = __ffsll(static_cast<long long>(open)) - 1;
        open &= open - 1;
        const int i = bit >> 1, pi = lane + 32 * (bit & 1);
        const uint32_t kp = *reinterpret_cast<const uint32_t*>(kn + src_of(i) + 2 * pi);
        const double ang = reduce_two_pi(static_cast<double>(apos + i) * p.theta[pi]);
        *reinterpret_cast<uint32_t*>(kc + dst_of(i, page_at(apos + i)) + 2 * pi) = rope_k_packed_fp64(kp, ang);
      }
    }
    if (bad_pos && lane == 0) atomicOr(p.err, static_cast<int>(MQA_DEVERR_POS_RANGE));
    if (bad_page && lane == 0) atomicOr(p.err, static_cast<int>(MQA_DEVERR_PAGE_RANGE));
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __syncwarp();
  };
  if (T == 0) {
    // no key of this split reaches these rows: an empty partial (weight 0 in
    // the combine); a fused step's rows owned by this split are still written
    if (FUSE && writer && warp == 7) append_rows();
    grid_dependency_wait();
    if constexpr (CL) {
      cl_empty();
      cl_exchange();
      return;
    }
    if (split_out) {
      for (int idx = tid; idx < rows * kD; idx += kThreads) {
        const int g = g0 + idx / kD, i = g / G;
        const long long grow = (static_cast<long long>(b) * n + i) * p.h_q + j * G + (g - i * G);
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
      mbar_init(bar(kKEmpty + s), 1);
      mbar_init(bar(kVFull + s), 1);
      mbar_init(bar(kVEmpty + s), 1);
    }
    for (int s = 0; s < kSBuf; ++s) {
      mbar_init(bar(kSFull + s), 1);
      mbar_init(bar(kPFull + s), 4);
      mbar_init(bar(kODone + s), 1);
    }
    mbar_init(bar(kDrain), 1);
    mbar_init(bar(kAppended), 1);  // the append warp
    mbar_init(bar(kQStage), 1);
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
  // q_rot and the new tokens' cache rows come from the preceding launch. After
  // the append kernel (early) every other cached row is final already: the
  // loaders stream those while it runs and wait only before a tile that holds
  // a new token; the softmax threads wait before reading q_rot.
  // the combine (or the next step) may be scheduled now; it waits for this
  // whole grid before it reads anything this grid writes
  grid_dependents_launch();
  if (!p.early) grid_dependency_wait();

  auto fail = [&](int role_lane0) {
    if (role_lane0) {
      s_abort = 1;
      atomicOr(p.err, static_cast<int>(MQA_DEVERR_TIMEOUT));
    }
  };
  auto stop = [&]() { return *reinterpret_cast<volatile int*>(&s_abort) != 0; };

  if (PG && (warp == 4 || warp == 5)) {
    // ------------------------------------ K (warp 4) / V (warp 5) loaders, paged
    // Lane c issues copy c of a tile (its rp rows, in two 64-dim halves at the
    // tile's two 16 KB halves). The page ids of the block's key range are held
    // 32 at a time, one per lane (wcur: pages wbase .., wnxt: the next 32). A
    // copy past the last page holding a key the block reads, or before the
    // first, loads nothing (page coordinate -1: the copy lands zeros) and its
    // entry is not read; an entry that a read needs and that is outside the
    // pool sets MQA_DEVERR_PAGE_RANGE, and its rows land as zeros.
    const bool is_k = warp == 4;
    const CUtensorMap* map = is_k ? &tmap_k : &tmap_v;
    const int full = is_k ? kKFull : kVFull, empty = is_k ? kKEmpty : kVEmpty;
    const uint32_t dst0 = sbase + (is_k ? kKOff : kVOff);
    const int ps = p.page_size, rp = ps < 64 ? ps : 64, copies = kBN / rp;
    const int lp_end = (kend + ps - 1) / ps, lp_first = ka_first / ps;
    auto entry = [&](int lp) { return (lp >= lp_first && lp < lp_end) ? __ldg(trow + lp) : -1; };
    int wbase = kstart / ps;
    int wcur = entry(wbase + lane), wnxt = entry(wbase + 32 + lane);
    bool bad = false;
    auto issue = [&](int it) {  // every lane
      const int s = it % kStages, key0 = tile_key0(it);
      while (key0 / ps - wbase >= 32) {
        wcur = wnxt;
        wbase += 32;
        wnxt = entry(wbase + 32 + lane);
      }
      const int k = key0 + lane * rp, lp = k / ps, off = lp - wbase;  // off < 32 + 8
      const int pc = __shfl_sync(0xffffffffu, wcur, off & 31), pn = __shfl_sync(0xffffffffu, wnxt, off & 31);
      int page = off < 32 ? pc : pn;
      const bool needed = lane < copies && lp >= lp_first && lp < lp_end;
      if (needed && (page < 0 || page >= p.num_pages)) bad = true;
      if (!needed || page < 0 || page >= p.num_pages) page = -1;
      if (lane == 0) mbar_arrive_expect_tx(bar(full + s), kTileBytes);
      __syncwarp();
      if (lane < copies) {
        const uint32_t d = dst0 + s * kTileBytes + lane * rp * 128;
        tma_load_5d(d, map, 0, k & (ps - 1), 0, j, page, bar(full + s));
        tma_load_5d(d + 16384, map, 0, k & (ps - 1), 1, j, page, bar(full + s));
      }
    };
    int it = 0;
    {
      const int npre = p.early && !p.q_tma ? kStages : kPreTiles;  // (q_tma: the query rows use stage kPreTiles on)
      const int lim = p.early ? Lp : (writer ? a_pos : 0x7fffffff);
      for (; it < T && it < npre && tile_key0(it) + kBN <= lim; ++it) issue(it);
    }
    named_bar_sync(2, kBM + 64);
    bool waited = !p.early, appended = !writer;
    for (; it < T; ++it) {
      const int s = it % kStages;
      bool ok = true;
      if (lane == 0) {
        if (it >= kStages) ok = mbar_wait(bar(empty + s), ((it - kStages) / kStages) & 1, p.wait_ns);
        if (ok && !appended && a_pos < tile_key0(it) + kBN) ok = mbar_wait(bar(kAppended), 0, p.wait_ns);
        if (!ok) fail(1);
        if (stop()) ok = false;
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      if (!appended && a_pos < tile_key0(it) + kBN) appended = true;
      if (!waited && Lp < tile_key0(it) + kBN) {  // this tile holds a new token's row
        grid_dependency_wait();
        waited = true;
      }
      issue(it);
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(p.err, static_cast<int>(MQA_DEVERR_PAGE_RANGE));
    // every tile this warp issued lands before the block can exit
    if (lane == 0)
      for (int k = it > kStages ? it - kStages : 0; k < it; ++k)
        (void)mbar_wait(bar(full + k % kStages), (k / kStages) & 1, kWaitLimitNs);
    __syncwarp();
  } else if (warp == 4 || warp == 5) {
    // ------------------------------------------------- K (warp 4) / V (warp 5) loaders
    const bool is_k = warp == 4;
    const CUtensorMap* map = is_k ? &tmap_k : &tmap_v;
    const int full = is_k ? kKFull : kVFull, empty = is_k ? kKEmpty : kVEmpty;
    const uint32_t dst0 = sbase + (is_k ? kKOff : kVOff);
    const int row = b * p.h_kv + j;
    auto issue = [&](int it) {
      const int s = it % kStages;
      mbar_arrive_expect_tx(bar(full + s), kTileBytes);
      if constexpr (F8)
        tma_load_3d(dst0 + s * kTileBytes, map, 0, tile_key0(it), row, bar(full + s));
      else
        tma_load_4d(dst0 + s * kTileBytes, map, 0, tile_key0(it), 0, row, bar(full + s));
    };
    int it = 0;
    {
      // the first tiles before the Q rows are in (while the append kernel
      // runs, the ring's first fill), none holding a row that the preceding
      // launch or this block's append writes
      const int npre = p.early && !p.q_tma ? kStages : kPreTiles;  // (q_tma: the query rows use stage kPreTiles on)
      const int lim = p.early ? Lp : (writer ? a_pos : 0x7fffffff);
      for (; it < T && it < npre && tile_key0(it) + kBN <= lim; ++it)
        if (lane == 0) issue(it);
    }
    // the rest only once the Q rows are in
    named_bar_sync(2, kBM + 64);
    if (lane == 0) {
      bool waited = !p.early, appended = !writer;
      for (; it < T; ++it) {
        const int s = it % kStages;
        if (it >= kStages && !mbar_wait(bar(empty + s), ((it - kStages) / kStages) & 1, p.wait_ns)) {
          fail(1);
          break;
        }
        if (stop()) break;
        if (!waited && Lp < tile_key0(it) + kBN) {  // this tile holds a new token's row
          grid_dependency_wait();
          waited = true;
        }
        if (!appended && a_pos < tile_key0(it) + kBN) {  // ... written by this block's append warp
          if (!mbar_wait(bar(kAppended), 0, p.wait_ns)) {
            fail(1);
            break;
          }
          appended = true;
        }
        issue(it);
      }
      // every tile this warp issued (it of them) lands before the block can
      // exit: after a timeout nothing else may wait for them
      for (int k = it > kStages ? it - kStages : 0; k < it; ++k)
        (void)mbar_wait(bar(full + k % kStages), (k / kStages) & 1, kWaitLimitNs);
    }
    __syncwarp();
  } else if (warp == 6) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      const uint32_t id_s = F8 ? tc05::idesc_e4m3_e5m2_f32(kBM, kBN, false, false)
                               : tc05::idesc_bf16_f32(kBM, kBN, false, false);
      const uint32_t id_o = F8 ? tc05::idesc_e4m3_e5m2_f32(kBM, kD, false, true)
                               : tc05::idesc_bf16_f32(kBM, kD, false, true);
      const uint32_t q_s = sbase + kQOff;
      bool ok = mbar_wait(bar(kQReady), 0, p.wait_ns);
      // S of tile it into buffer it % kSBuf. That buffer last held P of tile
      // it - kSBuf, whose PV was issued before: MMAs of this thread execute in order.
      auto issue_s = [&](int it) {
        const int s = it % kStages, sb = it % kSBuf;
        tc05::fence_after_sync();
        const uint32_t k_s = sbase + kKOff + s * kTileBytes;
        if constexpr (F8) {
          // S = Q_hi K^T + Q_lo K^T, 32 head dims per MMA (K-major 8-bit rows)
#pragma unroll
          for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int ks = 0; ks < kD / 32; ++ks)
              tc05::mma_f8(tmem + kColS + sb * 128, tc05::smem_desc_sw128(q_s + part * 16384 + ks * 32, 16, 1024),
                           tc05::smem_desc_sw128(k_s + ks * 32, 16, 1024), id_s, part > 0 || ks > 0);
        } else {
#pragma unroll
          for (int ks = 0; ks < kD / 16; ++ks) {
            const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
            tc05::mma_bf16(tmem + kColS + sb * 128, tc05::smem_desc_sw128(q_s + off, 16, 1024),
                           tc05::smem_desc_sw128(k_s + off, 16, 1024), id_s, ks > 0);
          }
        }
        tc05::commit(bar(kSFull + sb));
        tc05::commit(bar(kKEmpty + s));
      };
      auto issue_pv = [&](int it) {
        const int s = it % kStages, pb = it % kSBuf;
        tc05::fence_after_sync();
        const uint32_t v_s = sbase + kVOff + s * kTileBytes;
        if constexpr (F8) {
          // O += P_hi V + P_lo V, 32 keys per MMA: P from tensor memory (hi in
          // the buffer's columns 0-31, lo in 32-63), V MN-major (8-bit rows of
          // 128 dims, 8-key groups 1 KB apart)
#pragma unroll
          for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int ks = 0; ks < kBN / 32; ++ks)
              tc05::mma_f8_ta(tmem + kColO, tmem + kColS + pb * 128 + part * 32 + ks * 8,
                              tc05::smem_desc_sw128(v_s + ks * 4096, 16384, 1024), id_o,
                              it > 0 || part > 0 || ks > 0);
        } else {
#pragma unroll
          for (int ks = 0; ks < kBN / 16; ++ks)
            tc05::mma_bf16_ta(tmem + kColO, tmem + kColS + pb * 128 + ks * 8,
                              tc05::smem_desc_sw128(v_s + ks * 2048, 16384, 1024), id_o, it > 0 || ks > 0);
        }
        tc05::commit(bar(kODone + pb));
        tc05::commit(bar(kVEmpty + s));
      };
      // Issue S and PV as their inputs land: S of tile ns needs its K tile and
      // (buffer reuse) the PV of tile ns - kSBuf issued; PV of tile np needs its P
      // and V tile. Neither waits behind the other.
      int ns = 0, np = 0;
      unsigned long long t_idle = global_timer_ns();
      while (ok && np < T) {
        bool progress = false;
        if (ns < T && ns <= np + (kSBuf - 1) && mbar_test(bar(kKFull + ns % kStages), (ns / kStages) & 1)) {
          issue_s(ns++);
          progress = true;
        }
        if (np < ns && mbar_test(bar(kPFull + np % kSBuf), (np / kSBuf) & 1) &&
            mbar_test(bar(kVFull + np % kStages), (np / kStages) & 1)) {
          issue_pv(np++);
          progress = true;
        }
        if (progress) {
          t_idle = global_timer_ns();
        } else if (stop() || global_timer_ns() - t_idle > p.wait_ns) {
          ok = false;
        } else {
          __nanosleep(32);  // leave the issue slots to the softmax warp sharing this scheduler
        }
      }
      if (!ok) fail(1);
    }
    __syncwarp();
  } else if (warp == 7) {
    // ---------------------------------------------- append (fused step only)
    // The loaders wait for it only before the first tile that holds one of
    // this block's rows.
    if (FUSE && writer) {
      append_rows();
      if (lane == 0) mbar_arrive(bar(kAppended));
    }
  } else {
    // --------------------------------------------------- softmax (row = tid)
    const int r = tid;
    const int part = r / kRPad, gr = r - part * kRPad;  // key slice and row of this thread
    const bool live = gr < rows;
    const int gi = (g0 + gr) / G;                      // new token of this row
    const int hh = j * G + (g0 + gr - gi * G);         // its query head
    const long long grow_row = (static_cast<long long>(b) * n + gi) * p.h_q + hh;  // output row [B, n, H_q]
    if (!FUSE && p.q_tma) {
      // The block's 128 rows of q_rot as two TMA boxes of 64 rows (64 / G
      // tokens x G heads x 128 fp32 dims) into stages the first tile
      // requests leave free (bf16: K and V stage kPreTiles; fp8: K stages
      // kPreTiles .. kPreTiles + 3); a warp then builds its 32 rows of the Q
      // tile, lane l taking dims 4 l .. 4 l + 3 (a warp reads 512 contiguous
      // bytes per row), and only then are the loaders released. Read with
      // plain loads, a block's 4096 outstanding 16-byte misses drain a few
      // hundred at a time.
      if (p.early) grid_dependency_wait();
      const int qa = kKOff + kPreTiles * kTileBytes;
      const int qb = F8 ? qa + 32768 : kVOff + kPreTiles * kTileBytes;
      static_assert(F8 ? (kPreTiles + 4) * kTileBytes <= kStages * kTileBytes : kTileBytes >= 64 * kD * 4,
                    "query boxes in the free stages");
      if (tid == 0) {
        mbar_arrive_expect_tx(bar(kQStage), 2 * 64 * kD * 4);
        tma_load_3d(sbase + qa, &tmap_q, 0, j * G, b * n + g0 / G, bar(kQStage));
        tma_load_3d(sbase + qb, &tmap_q, 0, j * G, b * n + (g0 + 64) / G, bar(kQStage));
      }
      const bool landed = __all_sync(0xffffffffu, mbar_wait(bar(kQStage), 0, p.wait_ns));
      if (landed) {
#pragma unroll 4
        for (int i = 0; i < 32; ++i) {
          const int rq = 32 * warp + i;                       // row of the Q tile
          const int gq = rq - (rq / kRPad) * kRPad;           // its row of the block
          float4 v = *reinterpret_cast<const float4*>(smem + (gq < 64 ? qa : qb) + (gq & 63) * (kD * 4) + lane * 16);
          if (gq >= rows) v = make_float4(0.f, 0.f, 0.f, 0.f);
          if constexpr (F8) {
            const float qs = p.scale_log2 * kQScaleF8;
            const uint2 hl = e4m3_split4_once(v.x * qs, v.y * qs, v.z * qs, v.w * qs);
            const uint32_t off = rq * 128 + (((lane >> 2) ^ (rq & 7)) << 4) + (lane & 3) * 4;
            *reinterpret_cast<uint32_t*>(smem + kQOff + off) = hl.x;
            *reinterpret_cast<uint32_t*>(smem + kQOff + 16384 + off) = hl.y;
          } else {
            uint2 w;
            w.x = pack_bf16x2(v.x * p.scale_log2, v.y * p.scale_log2);
            w.y = pack_bf16x2(v.z * p.scale_log2, v.w * p.scale_log2);
            *reinterpret_cast<uint2*>(smem + kQOff + sw128(rq, 4 * lane)) = w;
          }
        }
      } else {
        if (lane == 0) fail(1);
        if (tid == 0) (void)mbar_wait(bar(kQStage), 0, kWaitLimitNs);  // the boxes land before the block exits
      }
      named_bar_arrive(2, kBM + 64);  // the boxes are read: the loaders may go on
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (landed && lane == 0) mbar_arrive(bar(kQReady));
    } else {
      // Q row, pre-scaled into the log2 domain, as bf16 in the swizzled tile.
      // The whole row is requested at once (one memory round trip), and the
      // K / V loaders are released only then: behind their burst of tile
      // requests these loads would wait microseconds.
      if (p.early) grid_dependency_wait();
      float4 qv[kD / 4];
      if constexpr (FUSE) {
        // fused step: q_new (bf16) rotated here, pair i of new token t by the
        // fp32 cosine / sine of the fp64-reduced angle (apos + t) theta_i, as
        // the append kernel forms q_rot. The tokens' tables [n][cos | sin]
        // (row stride kD + 1: the rows of a warp read different banks) sit in
        // the last K stage, which no tile request reaches before the Q rows
        // have landed (named barrier 2).
        static_assert(kPreTiles < kStages && kMaxNewTokens * (kD + 1) * 4 <= kTileBytes, "fused cos / sin tables");
        float* cst = reinterpret_cast<float*>(smem + kKOff + (kStages - 1) * kTileBytes);
        const uint4* qn = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.q_new) + grow_row * kD);
        uint4 raw[kD / 8];
#pragma unroll
        for (int c = 0; c < kD / 8; ++c) raw[c] = live ? qn[c] : make_uint4(0u, 0u, 0u, 0u);
        for (int e = tid; e < n * (kD / 2); e += kBM) {
          const int t = e / (kD / 2), pi = e - t * (kD / 2);
          const double ang = reduce_two_pi(static_cast<double>(apos + t) * p.theta[pi]);
          float sf, cf;
          sincosf(static_cast<float>(ang), &sf, &cf);
          cst[t * (kD + 1) + pi] = cf;
          cst[t * (kD + 1) + kD / 2 + pi] = sf;
        }
        named_bar_sync(3, kBM);  // the cos / sin tables
        const float* tcs = cst + min(gi, n - 1) * (kD + 1);  // this row's token
#pragma unroll
        for (int c = 0; c < kD / 8; ++c) {
          const uint32_t w4[4] = {raw[c].x, raw[c].y, raw[c].z, raw[c].w};
          float rv[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int pi = 4 * c + e;  // pair (2 pi, 2 pi + 1)
            const float x = bf16lo_to_f32(w4[e]), y = bf16hi_to_f32(w4[e]);
            const float cs = tcs[pi], sn = tcs[kD / 2 + pi];
            rv[2 * e] = x * cs - y * sn;
            rv[2 * e + 1] = x * sn + y * cs;
          }
          qv[2 * c] = make_float4(rv[0], rv[1], rv[2], rv[3]);
          qv[2 * c + 1] = make_float4(rv[4], rv[5], rv[6], rv[7]);
        }
        if (live && part == 0 && split == 0) {  // one copy of each row to q_rot
          float4* qo = reinterpret_cast<float4*>(p.q_rot_out + grow_row * kD);
#pragma unroll
          for (int c = 0; c < kD / 4; ++c) qo[c] = qv[c];
        }
      } else {
        const float4* q = reinterpret_cast<const float4*>(p.q_rot + grow_row * kD);
#pragma unroll
        for (int c = 0; c < kD / 4; ++c) qv[c] = live ? q[c] : make_float4(0.f, 0.f, 0.f, 0.f);
        named_bar_arrive(2, kBM + 64);  // (prefill and multi-token steps: the Q rows requested)
      }
      if constexpr (F8) {
        // e4m3 hi + lo of q * scale * log2(e) * 2^6: 16 dims per 16-byte chunk,
        // chunk c of row r at c ^ (r mod 8) (128-byte swizzle)
        const float qs = p.scale_log2 * kQScaleF8;
#pragma unroll
        for (int c = 0; c < kD / 16; ++c) {
          uint4 hi, lo;
          uint32_t* h = &hi.x;
          uint32_t* o = &lo.x;
#pragma unroll
          for (int w4 = 0; w4 < 4; ++w4) {
            const float4 a = qv[4 * c + w4];
            const uint2 hl = e4m3_split4_once(a.x * qs, a.y * qs, a.z * qs, a.w * qs);
            h[w4] = hl.x;
            o[w4] = hl.y;
          }
          const uint32_t off = r * 128 + ((c ^ (r & 7)) << 4);
          *reinterpret_cast<uint4*>(smem + kQOff + off) = hi;
          *reinterpret_cast<uint4*>(smem + kQOff + 16384 + off) = lo;
        }
      } else {
#pragma unroll
        for (int c = 0; c < kD; c += 8) {
          const float4 a = qv[c / 4], bq = qv[c / 4 + 1];
          uint4 v;
          v.x = pack_bf16x2(a.x * p.scale_log2, a.y * p.scale_log2);
          v.y = pack_bf16x2(a.z * p.scale_log2, a.w * p.scale_log2);
          v.z = pack_bf16x2(bq.x * p.scale_log2, bq.y * p.scale_log2);
          v.w = pack_bf16x2(bq.z * p.scale_log2, bq.w * p.scale_log2);
          *reinterpret_cast<uint4*>(smem + kQOff + sw128(r, c)) = v;
        }
      }
      if constexpr (FUSE) named_bar_arrive(2, kBM + 64);  // the Q rows have landed: the loaders may go on
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kQReady));
    }
    const int pos = live ? min(Lp + gi, t_end - 1) : -1;  // last key of this row in the split (none: padding)
    const int ka = p.window > 0 ? max(0, Lp + gi + 1 - p.window) : 0;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int it = 0; it < T; ++it) {
      const int sb = it % kSBuf;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(kSFull + sb), (it / kSBuf) & 1, p.wait_ns) && !stop());
      if (!ok) break;
      tc05::fence_after_sync();
      float s[kKW];
      // this thread's keys of the tile: columns part * kKW .. + kKW (loads in flight, one wait)
#pragma unroll
      for (int c = 0; c < kKW; c += 32)
        tc05::ld_32x32b_x32(tmem + lane_base + kColS + sb * 128 + part * kKW + c,
                            *reinterpret_cast<float(*)[32]>(&s[c]));
      tc05::wait_ld();
#pragma unroll
      for (int c = 0; c < kKW; c += 32) tc05::reg_fence(*reinterpret_cast<float(*)[32]>(&s[c]));
      if constexpr (F8) {
#pragma unroll
        for (int c = 0; c < kKW; ++c) s[c] *= 1.f / kQScaleF8;  // exact: a power of two
      }
      // keys of this tile outside [ka, pos] are masked
      const int key0 = tile_key0(it);
      if (key0 + kBN > t_end) {
        // rows past the split may hold anything: past the sequence any bit
        // pattern (NaN included), and the next split's first rows may be the
        // new token's, being written by another block of a fused step. P = 0
        // there, and 0 * NaN would still poison O: zero the V row of this
        // thread's key once that tile has landed
        ok = __all_sync(0xffffffffu, mbar_wait(bar(kVFull + it % kStages), (it / kStages) & 1, p.wait_ns));
        if (!ok) break;
        if (key0 + r >= t_end) {
          unsigned char* vrow = smem + kVOff + (it % kStages) * kTileBytes + r * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            *reinterpret_cast<uint4*>(vrow + c * 16) = make_uint4(0u, 0u, 0u, 0u);
            if constexpr (!F8) *reinterpret_cast<uint4*>(vrow + 16384 + c * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
      }
      const int kk0 = key0 + part * kKW;  // first key of this thread's slice
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
        ok = __all_sync(0xffffffffu,
                        mbar_wait(bar(kODone + (it - 1) % kSBuf), ((it - 1) / kSBuf) & 1, p.wait_ns) && !stop());
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
      // P of this thread's keys as bf16 pairs over its own S columns; the
      // other parts' columns of this row carry zeros
      const uint32_t prow = tmem + lane_base + kColS + sb * 128;
      if constexpr (F8) {
        // P as e4m3 hi + lo, four keys per column: hi over the buffer's columns
        // 0-31, lo over 32-63; this thread's keys at its part's columns, zeros
        // over the other parts'
        if constexpr (PARTS == 1) {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t ph[16], pl[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float pv[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                pv[k] = fast_exp2(s[64 * half + 4 * i + k] - e);
                sm8[(4 * i + k) & 7] += pv[k];
              }
              tc05::e4m3_split4(pv[0], pv[1], pv[2], pv[3], ph[i], pl[i]);
            }
            tc05::st_32x32b_x16_u(prow + 16 * half, ph);
            tc05::st_32x32b_x16_u(prow + 32 + 16 * half, pl);
          }
        } else {
          constexpr int kW8 = kKW / 4;  // columns of this thread's P_hi (and of its P_lo)
          uint32_t ph[kW8], pl[kW8], z[kW8];
#pragma unroll
          for (int i = 0; i < kW8; ++i) {
            float pv[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              pv[k] = fast_exp2(s[4 * i + k] - e);
              sm8[(4 * i + k) & 7] += pv[k];
            }
            tc05::e4m3_split4(pv[0], pv[1], pv[2], pv[3], ph[i], pl[i]);
            z[i] = 0u;
          }
#pragma unroll
          for (int q = 0; q < PARTS; ++q) {
            if constexpr (PARTS == 4) {
              tc05::st_32x32b_x8_u(prow + 8 * q, q == part ? ph : z);
              tc05::st_32x32b_x8_u(prow + 32 + 8 * q, q == part ? pl : z);
            } else {
              tc05::st_32x32b_x16_u(prow + 16 * q, q == part ? ph : z);
              tc05::st_32x32b_x16_u(prow + 32 + 16 * q, q == part ? pl : z);
            }
          }
        }
      } else if constexpr (PARTS == 1) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float p0 = fast_exp2(s[64 * half + 2 * i] - e), p1 = fast_exp2(s[64 * half + 2 * i + 1] - e);
            sm8[(2 * i) & 7] += p0;
            sm8[(2 * i + 1) & 7] += p1;
            pk[i] = pack_bf16x2(p0, p1);
          }
          tc05::st_32x32b_x32_u(prow + 32 * half, pk);
        }
      } else {
        constexpr int kCols = kKW / 2;  // 32-bit columns of this thread's P
        uint32_t pk[kCols];
#pragma unroll
        for (int i = 0; i < kCols; ++i) {
          const float p0 = fast_exp2(s[2 * i] - e), p1 = fast_exp2(s[2 * i + 1] - e);
          sm8[(2 * i) & 7] += p0;
          sm8[(2 * i + 1) & 7] += p1;
          pk[i] = pack_bf16x2(p0, p1);
        }
        if constexpr (PARTS == 2) {
          uint32_t z[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) z[i] = 0u;
          tc05::st_32x32b_x32_u(prow + 32 * part, *reinterpret_cast<uint32_t(*)[32]>(pk));
          tc05::st_32x32b_x32_u(prow + 32 * (1 - part), z);
        } else {
          uint32_t z[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) z[i] = 0u;
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            if (q4 == part)
              tc05::st_32x32b_x16_u(prow + 16 * q4, *reinterpret_cast<uint32_t(*)[16]>(pk));
            else
              tc05::st_32x32b_x16_u(prow + 16 * q4, z);
          }
        }
      }
      l += ((sm8[0] + sm8[1]) + (sm8[2] + sm8[3])) + ((sm8[4] + sm8[5]) + (sm8[6] + sm8[7]));
      tc05::wait_st();
      tc05::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kPFull + sb));
    }
    if (ok && T > 0)
      ok = __all_sync(0xffffffffu, mbar_wait(bar(kODone + (T - 1) % kSBuf), ((T - 1) / kSBuf) & 1, p.wait_ns));
    if (!ok && lane == 0) fail(1);
    if (ok) tc05::fence_after_sync();
    {
      if constexpr (PARTS == 1) {
        if (ok) {
        // ---- epilogue: O / l, lse = ln(sum exp(score)); a split writes its partial
        const float inv = l > 0.f ? 1.f / l : 0.f;
  #pragma unroll
        for (int c = 0; c < kD / 32; ++c) {
          float v[32];
          tc05::ld_32x32b_x32(tmem + lane_base + kColO + c * 32, v);
          tc05::wait_ld();
          tc05::reg_fence(v);
          if (live) {
            if (split_out) {
              float* dst = p.o_part + (grow_row * S + split) * kD + c * 32;
  #pragma unroll
              for (int i = 0; i < 32; i += 4)
                *reinterpret_cast<float4*>(dst + i) = make_float4(v[i] * inv, v[i + 1] * inv, v[i + 2] * inv,
                                                                  v[i + 3] * inv);
            } else if (p.out_dtype == kDtypeBf16) {
              __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + grow_row * kD + c * 32;
  #pragma unroll
              for (int i = 0; i < 32; i += 8) {
                uint4 w;
                w.x = pack_bf16x2(v[i] * inv, v[i + 1] * inv);
                w.y = pack_bf16x2(v[i + 2] * inv, v[i + 3] * inv);
                w.z = pack_bf16x2(v[i + 4] * inv, v[i + 5] * inv);
                w.w = pack_bf16x2(v[i + 6] * inv, v[i + 7] * inv);
                *reinterpret_cast<uint4*>(dst + i) = w;
              }
            } else {
              float* dst = static_cast<float*>(p.out) + grow_row * kD + c * 32;
  #pragma unroll
              for (int i = 0; i < 32; i += 4)
                *reinterpret_cast<float4*>(dst + i) = make_float4(v[i] * inv, v[i + 1] * inv, v[i + 2] * inv,
                                                                  v[i + 3] * inv);
            }
          }
        }
        const float lse = l > 0.f ? (m_ref + log2f(l)) * 0.69314718055994530942f : -INFINITY;
        if (live && split_out)
          p.lse_part[grow_row * S + split] = lse;
        else if (live && p.lse_out != nullptr)
          p.lse_out[grow_row] = lse;
        }
      } else {
        // ---- merge the PARTS partial softmaxes of each row through shared
        // memory (the K stages: every K tile has been consumed by now)
        constexpr int kStride = kD + 4;
        float* mo = reinterpret_cast<float*>(smem + kKOff);  // [128][kStride] unnormalised O
        float* mm = mo + kBM * kStride;                        // [128] reference maxima
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
              *reinterpret_cast<float4*>(mo + r * kStride + c * 32 + i) =
                  make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
          }
          mm[r] = m_ref;
          ml[r] = l;
        }
        // every softmax warp arrives, also after a timeout (which set s_abort first)
        named_bar_sync(1, kBM);
        // thread r < rows: the weight of each part in row r (its partial
        // softmax renormalised to the row's maximum and divided by the row's
        // total), the row's lse and output row
        float* mw = ml + kBM;                                  // [PARTS][kRPad]
        long long* mrow = reinterpret_cast<long long*>(mw + kBM);  // [kRPad]
        if (r < rows && !stop()) {
          float mx = -INFINITY;
#pragma unroll
          for (int q = 0; q < PARTS; ++q) mx = fmaxf(mx, mm[q * kRPad + r]);
          float w[PARTS], den = 0.f;
#pragma unroll
          for (int q = 0; q < PARTS; ++q) {
            w[q] = mx == -INFINITY ? 0.f : exp2f(mm[q * kRPad + r] - mx);
            den = fmaf(w[q], ml[q * kRPad + r], den);
          }
          const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
          for (int q = 0; q < PARTS; ++q) mw[q * kRPad + r] = w[q] * inv;
          const int ti = (g0 + r) / G;
          const long long orow = (static_cast<long long>(b) * n + ti) * p.h_q + j * G + (g0 + r - ti * G);
          mrow[r] = orow;
          const float lse = den > 0.f ? (mx + log2f(den)) * 0.69314718055994530942f : -INFINITY;
          if constexpr (CL)
            xl[r] = lse;
          else if (split_out)
            p.lse_part[orow * S + split] = lse;
          else if (p.lse_out != nullptr)
            p.lse_out[orow] = lse;
        }
        named_bar_sync(1, kBM);
        // thread = head dim: every row's output element, rows independent
        const int d = r;
        if (!stop()) {
#pragma unroll 4
          for (int row = 0; row < rows; ++row) {
            float ov = 0.f;
#pragma unroll
            for (int q = 0; q < PARTS; ++q)
              ov = fmaf(mw[q * kRPad + row], mo[(q * kRPad + row) * kStride + d], ov);
            const long long orow = mrow[row];
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
        (void)mbar_wait(bar(kDrain), 0, kWaitLimitNs);
      }
      __syncwarp();
    }
    tc05::fence_after_sync();
    tc05::tmem_dealloc(tmem, kTmemCols);
  }
  if constexpr (CL) cl_exchange();
}

}  // namespace

KernelShape tc05_shape() { return {kThreads, Lay<false>::kSmemBytes, kBM, 1}; }

int tc05_f8_box_rows() { return kBN; }

template <int PARTS, bool FUSE, bool CL, bool F8, bool PG>
cudaError_t launch_parts(const Tc05Params& p, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tq,
                         cudaStream_t stream) {
  auto kern = attn_tc05_kernel<PARTS, FUSE, CL, F8, PG>;
  constexpr int smem = Lay<F8>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.batch) * p.h_kv * p.num_splits * p.row_blocks);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
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
  return cudaLaunchKernelEx(&cfg, kern, tk, tv, tq, p);
}

template <int PARTS, bool F8, bool PG>
cudaError_t launch_fuse(const Tc05Params& p, bool cl, const CUtensorMap& tk, const CUtensorMap& tv,
                        const CUtensorMap& tq, cudaStream_t stream) {
  if constexpr (F8) {  // (several new tokens: never fused)
    return cl ? launch_parts<PARTS, false, true, true, false>(p, tk, tv, tq, stream)
              : launch_parts<PARTS, false, false, true, false>(p, tk, tv, tq, stream);
  } else {
    if (cl)
      return p.fuse ? launch_parts<PARTS, true, true, false, PG>(p, tk, tv, tq, stream)
                    : launch_parts<PARTS, false, true, false, PG>(p, tk, tv, tq, stream);
    return p.fuse ? launch_parts<PARTS, true, false, false, PG>(p, tk, tv, tq, stream)
                  : launch_parts<PARTS, false, false, false, PG>(p, tk, tv, tq, stream);
  }
}

template <bool F8, bool PG>
cudaError_t launch_rows(const Tc05Params& p, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tq,
                        cudaStream_t stream) {
  // replicate few rows over the 128 MMA rows so that all four softmax warps work
  const long long rows = static_cast<long long>(p.group) * p.n_new;
  const bool cl = tc05_merges_splits(p);
  // (a fused step has one row block: p.fuse implies row_blocks == 1)
  if (p.row_blocks == 1 && rows <= 32) return launch_fuse<4, F8, PG>(p, cl, tk, tv, tq, stream);
  if (p.row_blocks == 1 && rows <= 64) return launch_fuse<2, F8, PG>(p, cl, tk, tv, tq, stream);
  if constexpr (F8)
    return launch_parts<1, false, false, true, false>(p, tk, tv, tq, stream);
  else
    return p.fuse ? launch_parts<1, true, false, false, PG>(p, tk, tv, tq, stream)
                  : launch_parts<1, false, false, false, PG>(p, tk, tv, tq, stream);
}

bool tc05_merges_splits(const Tc05Params& p) {
  return p.num_splits == 2 && p.row_blocks == 1 && static_cast<long long>(p.group) * p.n_new <= 64;
}

cudaError_t launch_tc05_attention(const Tc05Params& p, const CUtensorMap& tk, const CUtensorMap& tv,
                                  const CUtensorMap* tq, cudaStream_t stream) {
  if (p.q_tma && tq == nullptr) return cudaErrorInvalidValue;
  const CUtensorMap& q = tq ? *tq : tk;  // (unused unless p.q_tma)
  if (p.f8) return launch_rows<true, false>(p, tk, tv, q, stream);
  return p.paged ? launch_rows<false, true>(p, tk, tv, q, stream) : launch_rows<false, false>(p, tk, tv, q, stream);
}

}  // namespace mqa
