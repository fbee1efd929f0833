// Prefill attention on the 5th-generation tensor cores ("KV Cache" explainer,
// Langkah 1 and 4: the prompt's keys and values are computed in one pass and
// stored, and the work is compute-bound), two query tiles per block.
//
// The rows of kv head j are its (new token i, query head h = j G + hl) pairs,
// row = i G + hl. A block takes 256 consecutive rows of one (sequence, kv
// head) as two 128-row query tiles, Q0 and Q1, which share every K / V tile
// it loads: half the L2-to-SM bytes per FLOP of one tile per block, whose
// K / V loads were measured to be the limit (a tile's V landing 2.4 us after
// its request under load, three stages deep). Row (i, hl), at position
// p = L - n_new + i, attends to the keys [max(0, p + 1 - W) if windowed else
// 0, p]. For each 128-key tile:
//   S_q = Q_q K^T   tcgen05.mma M=128 N=128 K=128 per query tile, S (f32)
//                   into tensor memory
//   online softmax  one row per thread, warps 0-3 for Q0 and 4-7 for Q1 (two
//                   warps per scheduler: one's softmax runs while the other's
//                   waits on its product); P (bf16) written over its S columns
//   O_q += P_q V    tcgen05.mma with A = P from tensor memory, V from shared
//                   memory; O_q stays in tensor memory
// with FlashAttention's running maximum ("Arsitektur Inferensi LLM", section
// 5) and the same lazy rescale as the decode kernel (O only rescaled when a
// row's maximum grows by more than 2^8). Tensor memory: S/P of Q0 and Q1
// (128 columns each) and O of each (128 each), 512 columns. S_q of the next
// tile is issued right after PV_q of this one (the products of one thread
// run in order, so PV_q has read P_q before S_q overwrites it), so the tensor
// core alternates between the two query tiles while each warpgroup works on
// the other's products. A softmax warpgroup publishes P in two halves (keys
// 0-63, then 64-127) and each half's four products are issued as soon as it
// is written (8 x 4096 step 1178 -> 1164 us).
//
// K / V tiles (32 KB) share one ring of kSlots slots in load order K(0),
// V(0), K(1), V(1), ...; slots are released in that order too (K(t) after
// S_1(t), V(t) after PV_1(t)). Warp 8 loads (TMA), warp 9 issues the MMAs
// (one thread) and owns the tensor memory; warps 10 and 11 only complete the
// third warpgroup.
//
// The block's 256 query rows (fp32 q_rot, 128 KB) arrive as one TMA box in
// ring slots 1-4 while K(0) lands in slot 0; the softmax warps scale them into
// the bf16 query tiles, and only then does the ring take V(0) and the rest.
// Read with plain loads instead (still done when the group is not a power of
// two), the rows took 8-9 us per block: a block's 8192 outstanding 16-byte
// misses drain a few hundred at a time.
#include <cuda_bf16.h>

#include "../../include/mqa_decode.h"
#include "launch.h"
#include "ptx.cuh"
#include "tc05.cuh"

namespace mqa {
namespace {

constexpr int kD = 128;
constexpr int kBM = 128;  // rows of a query tile
constexpr int kQT = 2;    // query tiles per block
constexpr int kBN = 128;  // keys per tile
constexpr int kThreads = 384;  // three warpgroups (setmaxnreg works per warpgroup)
// Registers: launched at 168 a thread (the most 384 threads can have: three
// warps per scheduler); the loader / MMA warpgroup drops to kRegsAux and the
// two softmax warpgroups take what it frees (a row's 128 scores stay in
// registers). The shares add up to the launch's total exactly:
// 384 x 168 = 2 x 128 x kRegsSoftmax + 128 x kRegsAux.
constexpr int kRegsLaunch = 168, kRegsSoftmax = 216, kRegsAux = 72;
static_assert(kThreads * kRegsLaunch == 2 * 128 * kRegsSoftmax + 128 * kRegsAux, "register split");
constexpr int kSlots = 5;
constexpr int kTileBytes = kBN * kD * 2;
constexpr int kQBytes = kBM * kD * 2;
constexpr int kQOff = 0;
constexpr int kRingOff = kQT * kQBytes;
constexpr int kBarOff = kRingOff + kSlots * kTileBytes;
constexpr int kSmemBytes = kBarOff + 256 + 1024;  // + 1 KB alignment slack
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColO = 256;  // S/P of tile q at 128 q, O of tile q at 256 + 128 q
constexpr float kRescaleLog2 = 8.0f;
// F8: Q enters scaled by 2^6 (its values then sit in e4m3's normal range); the
// scores come out 2^6 too large and are scaled back exactly
constexpr float kQScaleF8 = 64.f;
// mbarriers (8 bytes each) at kBarOff
constexpr int kQReady = 0;                // [kQT] the query tile is in shared memory (4 warps)
constexpr int kFull = kQReady + kQT;      // [kSlots]
constexpr int kEmpty = kFull + kSlots;    // [kSlots]
constexpr int kSFull = kEmpty + kSlots;   // [kQT]
constexpr int kPLo = kSFull + kQT;        // [kQT] P of keys 0-63 written (4 warps)
constexpr int kPHi = kPLo + kQT;          // [kQT] P of keys 64-127 written (4 warps)
constexpr int kODone = kPHi + kQT;        // every product done (committed once)
constexpr int kDrain = kODone + 1;
constexpr int kQStage = kDrain + 1;       // the query rows' box landed (ring slots 1-4)
constexpr int kNBars = kQStage + 1;
constexpr int kQStageBytes = kQT * kBM * kD * 4;
static_assert(kSlots >= 5 && 4 * kTileBytes == kQStageBytes, "query box in ring slots 1-4");
static_assert(kNBars * 8 + 4 <= 256, "barrier area");
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

__device__ __forceinline__ uint32_t sw128(int r, int col) {  // byte offset of bf16 element (r, col) of a tile
  const int half = col >> 6, chunk = (col & 63) >> 3;
  return half * 16384 + r * 128 + ((chunk ^ (r & 7)) << 4) + (col & 7) * 2;
}

// PG: paged bf16 pool [num_pages, h_kv, page_size, 128] through the block
// table; a key tile is gathered page by page (rp = min(page_size, 64) rows per
// copy: tiles start on multiples of 64, so a 64-key half never straddles a
// page).
// The softmax's fp32 arithmetic on the sm_100 family's packed and
// three-input forms: two subtractions or additions per instruction (each
// rounded as the scalar one), and a maximum of three values (exact). The
// results are those of the scalar code; the instruction count of a row's
// softmax drops by about a fifth (8 x 4096 prefill step 1221 -> 1178 us with
// the packed pairs).
__device__ __forceinline__ float2 sub2(float2 a, float b) {
  float2 r;
  asm("{\n\t.reg .b64 ra, rb, rr;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %4};\n\t"
      "sub.rn.f32x2 rr, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rr;\n\t}"
      : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b));
  return r;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 r;
  asm("{\n\t.reg .b64 ra, rb, rr;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rr, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rr;\n\t}"
      : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

// F8: contiguous fp8 e5m2 cache. K and V code tiles (16 KB, one per ring
// slot) are the MMAs' B operands as TMA lands them (kind::f8f6f4, K = 32 per
// instruction); Q (scaled by 2^6 into e4m3's normal range) and P each enter
// as two e4m3 parts, hi = e4m3(x) and lo = e4m3(x - hi), as in the fp8 form
// of attn_tc05_kernel, so the scores and outputs equal that kernel's up to the
// order of fp32 accumulation.
template <bool PG, bool F8>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc05_prefill_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                             const __grid_constant__ CUtensorMap tmap_q, const Tc05Params p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + kBarOff + kNBars * 8);
  __shared__ int s_abort, s_skip;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  static_assert(!(PG && F8), "e5m2: contiguous caches only");
  constexpr int kLoadBytes = F8 ? kBN * kD : kTileBytes;  // bytes of one K / V tile (a ring slot holds one)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.group, n = p.n_new, R = G * n;
  // block order: sequence fastest, then kv head, then row pair (the pairs with
  // the longest key ranges -- the last tokens -- first)
  int cta = blockIdx.x;
  const int b = cta % p.batch;
  cta /= p.batch;
  const int j = cta % p.h_kv;
  const int pair = p.row_blocks - 1 - cta / p.h_kv;
  const int g0 = pair * kQT * kBM;
  const int rows = min(kQT * kBM, R - g0);

  long long limit = p.capacity < p.max_seq_len ? p.capacity : p.max_seq_len;
  int L = p.seq_lens[b];
  const int err0 = tid == 0 ? *reinterpret_cast<volatile int32_t*>(p.err) : 0;
  if (L < n || L > limit) {
    if (tid == 0 && pair == 0 && j == 0) atomicOr(p.err, static_cast<int>(MQA_DEVERR_SEQ_LEN));
    L = L < n ? n : static_cast<int>(limit);
  }
  if (tid == 0) s_skip = (err0 & static_cast<int>(MQA_DEVERR_TIMEOUT)) ? 1 : 0;
  __syncthreads();
  if (s_skip) return;  // an earlier block timed out: the result is invalid already

  const int Lp = L - n;  // new token i sits at position Lp + i
  const int pos_first = Lp + g0 / G, pos_last = Lp + (g0 + rows - 1) / G;
  const int ka_first = p.window > 0 ? max(0, pos_first + 1 - p.window) : 0;
  const int kstart = (ka_first / 64) * 64;
  const int kend = min(L, pos_last + 1);
  const int T = (kend - kstart + kBN - 1) / kBN;  // >= 1: pos_last >= pos_first >= ka_first
  auto tile_key0 = [&](int it) { return kstart + it * kBN; };

  if (tid == 0) {
    s_abort = 0;
    for (int q = 0; q < kQT; ++q) {
      mbar_init(bar(kQReady + q), 4);
      mbar_init(bar(kSFull + q), 1);
      mbar_init(bar(kPLo + q), 4);
      mbar_init(bar(kPHi + q), 4);
    }
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(bar(kFull + s), 1);
      mbar_init(bar(kEmpty + s), 1);
    }
    mbar_init(bar(kODone), 1);
    mbar_init(bar(kDrain), 1);
    mbar_init(bar(kQStage), 1);
    fence_mbar_init();
  }
  if (warp == 9) {
    tc05::tmem_alloc(smem_u32(tslot), kTmemCols);
    tc05::tmem_relinquish();
  }
  tc05::fence_before_sync();
  __syncthreads();
  tc05::fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tslot);
  const uint32_t sbase = smem_u32(smem);
  // q_rot and the prompt's cache rows come from the preceding append launch
  // (early): every other cached row is final already, so the loader streams
  // those while it runs and waits only before a tile that holds a new row;
  // the softmax warps wait before reading q_rot
  grid_dependents_launch();
  if (!p.early) grid_dependency_wait();

  auto fail = [&](int role_lane0) {
    if (role_lane0) {
      s_abort = 1;
      atomicOr(p.err, static_cast<int>(MQA_DEVERR_TIMEOUT));
    }
  };
  auto stop = [&]() { return *reinterpret_cast<volatile int*>(&s_abort) != 0; };

  // each role sets its warpgroup's register share first thing (warps 8-11
  // give, warps 0-7 take)
  auto regs_aux = [&]() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsAux)); };
  if (warp == 8) {
    regs_aux();
    // ------------------------------------------------------------- loader
    // load u = 2 t + 0 / 1: K / V of tile t, into slot u % kSlots
    const int row = b * p.h_kv + j;
    const int32_t* trow = PG ? p.block_table + static_cast<long long>(b) * p.max_pages : nullptr;
    // paged: the page ids of the block's key range, 32 at a time, one per
    // lane (wcur: pages wbase .., wnxt: the next 32); entries outside the
    // attended range are not read, and a copy there lands zeros (page -1)
    const int ps = PG ? p.page_size : 64, rp = ps < 64 ? ps : 64, copies = kBN / rp;
    const int lp_end = (kend + ps - 1) / ps, lp_first = ka_first / ps;
    auto entry = [&](int lp) { return (PG && lp >= lp_first && lp < lp_end) ? __ldg(trow + lp) : -1; };
    int wbase = kstart / ps;
    int wcur = entry(wbase + lane), wnxt = entry(wbase + 32 + lane);
    bool bad = false;
    auto issue = [&](int u) {  // every lane
      const int slot = u % kSlots, t = u >> 1;
      const CUtensorMap* map = (u & 1) ? &tmap_v : &tmap_k;
      const uint32_t dst = sbase + kRingOff + slot * kTileBytes;
      if constexpr (PG) {
        const int key0 = tile_key0(t);
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
        if (lane == 0) mbar_arrive_expect_tx(bar(kFull + slot), kTileBytes);
        __syncwarp();
        if (lane < copies) {
          const uint32_t d = dst + lane * rp * 128;
          tma_load_5d(d, map, 0, k & (ps - 1), 0, j, page, bar(kFull + slot));
          tma_load_5d(d + 16384, map, 0, k & (ps - 1), 1, j, page, bar(kFull + slot));
        }
      } else if (lane == 0) {
        mbar_arrive_expect_tx(bar(kFull + slot), kLoadBytes);
        if constexpr (F8)
          tma_load_3d(dst, map, 0, tile_key0(t), row, bar(kFull + slot));
        else
          tma_load_4d(dst, map, 0, tile_key0(t), 0, row, bar(kFull + slot));
      }
    };
    bool waited = !p.early;
    const bool q_tma = p.q_tma != 0;
    if (q_tma) {
      // the query rows (written by the preceding launch): 256 / G tokens x G
      // heads x 128 dims, block row r at row r of the box
      if (!waited) {
        grid_dependency_wait();
        waited = true;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(kQStage), kQStageBytes);
        tma_load_3d(sbase + kRingOff + kTileBytes, &tmap_q, 0, j * G, b * n + g0 / G, bar(kQStage));
      }
    }
    int u = 0;
    for (; u < 2 * T; ++u) {
      const int slot = u % kSlots;
      bool ok = true;
      if (lane == 0) {
        if (u >= kSlots)
          ok = mbar_wait(bar(kEmpty + slot), ((u / kSlots) - 1) & 1, p.wait_ns);
        else if (q_tma && u == 1)  // slots 1-4 are free once both query tiles are built
          ok = mbar_wait(bar(kQReady + 0), 0, p.wait_ns) && mbar_wait(bar(kQReady + 1), 0, p.wait_ns);
        if (!ok) fail(1);
        if (stop()) ok = false;
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      if (!waited && Lp < tile_key0(u >> 1) + kBN) {  // this tile holds a new row
        grid_dependency_wait();
        waited = true;
      }
      issue(u);
    }
    if (PG && __any_sync(0xffffffffu, bad) && lane == 0) atomicOr(p.err, static_cast<int>(MQA_DEVERR_PAGE_RANGE));
    // every copy this warp issued lands before the block can exit
    if (lane == 0) {
      if (q_tma) (void)mbar_wait(bar(kQStage), 0, kWaitLimitNs);
      for (int k = u > kSlots ? u - kSlots : 0; k < u; ++k)
        (void)mbar_wait(bar(kFull + k % kSlots), (k / kSlots) & 1, kWaitLimitNs);
    }
    __syncwarp();
  } else if (warp == 9) {
    regs_aux();
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr uint32_t id_s = F8 ? tc05::idesc_e4m3_e5m2_f32(kBM, kBN, false, false)
                                   : tc05::idesc_bf16_f32(kBM, kBN, false, false);
      constexpr uint32_t id_o = F8 ? tc05::idesc_e4m3_e5m2_f32(kBM, kD, false, true)
                                   : tc05::idesc_bf16_f32(kBM, kD, false, true);
      // waits poll (test_wait): a suspended try_wait woke a third of a
      // microsecond after the phase completed, once per product group
      // (8 x 4096: 1608 -> 1532 us per step)
      auto wait = [&](int id, int parity) {
        const unsigned long long t0 = global_timer_ns();
        while (!mbar_test(bar(id), parity))
          if (stop() || global_timer_ns() - t0 > p.wait_ns) return false;
        return true;
      };
      auto issue_s = [&](int q, int t) {  // S_q = Q_q K(t)^T
        const uint32_t q_s = sbase + kQOff + q * kQBytes, k_s = sbase + kRingOff + ((2 * t) % kSlots) * kTileBytes;
        tc05::fence_after_sync();
        if constexpr (F8) {
          // S = Q_hi K^T + Q_lo K^T, 32 head dims per product (K-major 8-bit rows)
#pragma unroll
          for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int ks = 0; ks < kD / 32; ++ks)
              tc05::mma_f8(tmem + kColS + q * 128, tc05::smem_desc_sw128(q_s + part * 16384 + ks * 32, 16, 1024),
                           tc05::smem_desc_sw128(k_s + ks * 32, 16, 1024), id_s, part > 0 || ks > 0);
        } else {
#pragma unroll
          for (int ks = 0; ks < kD / 16; ++ks) {
            const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
            tc05::mma_bf16(tmem + kColS + q * 128, tc05::smem_desc_sw128(q_s + off, 16, 1024),
                           tc05::smem_desc_sw128(k_s + off, 16, 1024), id_s, ks > 0);
          }
        }
        tc05::commit(bar(kSFull + q));
      };
      auto issue_pv = [&](int q, int t, int h) {  // O_q += P_q V(t), keys 64 h .. 64 h + 63
        const uint32_t v_s = sbase + kRingOff + ((2 * t + 1) % kSlots) * kTileBytes;
        tc05::fence_after_sync();
        if constexpr (F8) {
          // O += P_hi V + P_lo V, 32 keys per product: P from tensor memory
          // (hi in the buffer's columns 0-31, lo in 32-63, four keys a
          // column), V MN-major (8-bit rows of 128 dims)
#pragma unroll
          for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int ks = 2 * h; ks < 2 * h + 2; ++ks)
              tc05::mma_f8_ta(tmem + kColO + q * 128, tmem + kColS + q * 128 + part * 32 + ks * 8,
                              tc05::smem_desc_sw128(v_s + ks * 4096, 16384, 1024), id_o, t > 0 || h > 0 || part > 0 || ks > 0);
        } else {
#pragma unroll
          for (int ks = 4 * h; ks < 4 * h + 4; ++ks)
            tc05::mma_bf16_ta(tmem + kColO + q * 128, tmem + kColS + q * 128 + ks * 8,
                              tc05::smem_desc_sw128(v_s + ks * 2048, 16384, 1024), id_o, t > 0 || ks > 0);
        }
      };
      auto full = [&](int u) { return wait(kFull + u % kSlots, (u / kSlots) & 1); };
      bool ok = wait(kQReady + 0, 0) && wait(kQReady + 1, 0) && full(0);
      if (ok) {
        issue_s(0, 0);
        issue_s(1, 0);
        tc05::commit(bar(kEmpty + 0));  // K(0)
      }
      for (int t = 0; ok && t < T; ++t) {
        // PV_0(t), then S_0(t + 1) (P_0 read before S_0 is overwritten: in
        // order); each half of a PV as soon as its half of P is written
        ok = wait(kPLo + 0, t & 1) && full(2 * t + 1);
        if (!ok) break;
        issue_pv(0, t, 0);
        ok = wait(kPHi + 0, t & 1);
        if (!ok) break;
        issue_pv(0, t, 1);
        if (t + 1 < T) {
          ok = full(2 * t + 2);
          if (!ok) break;
          issue_s(0, t + 1);
        }
        ok = wait(kPLo + 1, t & 1);
        if (!ok) break;
        issue_pv(1, t, 0);
        ok = wait(kPHi + 1, t & 1);
        if (!ok) break;
        issue_pv(1, t, 1);
        tc05::commit(bar(kEmpty + (2 * t + 1) % kSlots));  // V(t)
        if (t + 1 < T) {
          issue_s(1, t + 1);
          tc05::commit(bar(kEmpty + (2 * t + 2) % kSlots));  // K(t + 1)
        }
      }
      if (ok) tc05::commit(bar(kODone));
      if (!ok) fail(1);
    }
    __syncwarp();
  } else if (warp >= 10) {
    regs_aux();
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    // --------------------------------------------- softmax of query tile q
    const int q = warp >> 2, r = tid - q * kBM;  // row r of query tile q
    const int gr = q * kBM + r;                  // row of the block
    const bool live = gr < rows;
    const int gi = (g0 + gr) / G;                // new token of this row
    const int hh = j * G + (g0 + gr - gi * G);   // its query head
    const long long grow_row = (static_cast<long long>(b) * n + gi) * p.h_q + hh;
    unsigned char* qtile = smem + kQOff + q * kQBytes;
    bool qok = true;
    if (p.q_tma) {
      // this warp's 32 rows of query tile q from the landed box, pre-scaled
      // into the log2 domain, as bf16 in the swizzled tile (rows past the
      // block's rows zero): lane l takes dims 4 l .. 4 l + 3 of one row at a
      // time, so a warp reads 512 contiguous bytes per row
      qok = __all_sync(0xffffffffu, mbar_wait(bar(kQStage), 0, p.wait_ns));
      if (qok) {
        const unsigned char* stage = smem + kRingOff + kTileBytes;
        const int rbase = (warp & 3) * 32;
#pragma unroll 4
        for (int i = 0; i < 32; ++i) {
          const int rr = rbase + i;
          float4 v = *reinterpret_cast<const float4*>(stage + (q * kBM + rr) * (kD * 4) + lane * 16);
          if (q * kBM + rr >= rows) v = make_float4(0.f, 0.f, 0.f, 0.f);
          if constexpr (F8) {
            // e4m3 hi + lo of q * scale * log2(e) * 2^6, chunk c of row rr at c ^ (rr mod 8)
            const float qs = p.scale_log2 * kQScaleF8;
            uint32_t hi, lo;
            tc05::e4m3_split4(v.x * qs, v.y * qs, v.z * qs, v.w * qs, hi, lo);
            const uint32_t off = rr * 128 + (((lane >> 2) ^ (rr & 7)) << 4) + (lane & 3) * 4;
            *reinterpret_cast<uint32_t*>(qtile + off) = hi;
            *reinterpret_cast<uint32_t*>(qtile + 16384 + off) = lo;
          } else {
            uint2 w;
            w.x = pack_bf16x2(v.x * p.scale_log2, v.y * p.scale_log2);
            w.y = pack_bf16x2(v.z * p.scale_log2, v.w * p.scale_log2);
            *reinterpret_cast<uint2*>(qtile + sw128(rr, 4 * lane)) = w;
          }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kQReady + q));
      } else if (lane == 0) {
        fail(1);
      }
    } else {
      // Q row, pre-scaled into the log2 domain, as bf16 in the swizzled tile
      if (p.early) grid_dependency_wait();
      const float4* qs = reinterpret_cast<const float4*>(p.q_rot + grow_row * kD);
      float4 qv[kD / 4];
#pragma unroll
      for (int c = 0; c < kD / 4; ++c) qv[c] = live ? qs[c] : make_float4(0.f, 0.f, 0.f, 0.f);
      if constexpr (F8) {
        const float qs = p.scale_log2 * kQScaleF8;
#pragma unroll
        for (int c = 0; c < kD / 16; ++c) {  // 16 dims per 16-byte chunk
          uint4 hi, lo;
          uint32_t* h4 = &hi.x;
          uint32_t* l4 = &lo.x;
#pragma unroll
          for (int w4 = 0; w4 < 4; ++w4) {
            const float4 a = qv[4 * c + w4];
            tc05::e4m3_split4(a.x * qs, a.y * qs, a.z * qs, a.w * qs, h4[w4], l4[w4]);
          }
          const uint32_t off = r * 128 + ((c ^ (r & 7)) << 4);
          *reinterpret_cast<uint4*>(qtile + off) = hi;
          *reinterpret_cast<uint4*>(qtile + 16384 + off) = lo;
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
          *reinterpret_cast<uint4*>(qtile + sw128(r, c)) = v;
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kQReady + q));
    }
    const int pos = live ? Lp + gi : -1;  // last key of this row (none: padding)
    const int ka = p.window > 0 ? max(0, Lp + gi + 1 - p.window) : 0;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t scol = tmem + lane_base + kColS + q * 128, ocol = tmem + lane_base + kColO + q * 128;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = qok;
    for (int t = 0; ok && t < T; ++t) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar(kSFull + q), t & 1, p.wait_ns) && !stop());
      if (!ok) break;
      tc05::fence_after_sync();
      float s[kBN];
#pragma unroll
      for (int c = 0; c < kBN; c += 32) tc05::ld_32x32b_x32(scol + c, *reinterpret_cast<float(*)[32]>(&s[c]));
      tc05::wait_ld();
#pragma unroll
      for (int c = 0; c < kBN; c += 32) tc05::reg_fence(*reinterpret_cast<float(*)[32]>(&s[c]));
      if constexpr (F8) {
#pragma unroll
        for (int c = 0; c < kBN; ++c) s[c] *= 1.f / kQScaleF8;  // exact: a power of two
      }
      const int key0 = tile_key0(t);
      if (q == 0 && key0 + kBN > L) {
        // rows at or past L may hold anything (NaN included); P = 0 there, and
        // 0 * NaN would still poison O: zero the V rows once the tile has
        // landed (before P_0 is published, so before either PV reads them)
        ok = __all_sync(0xffffffffu, mbar_wait(bar(kFull + (2 * t + 1) % kSlots), ((2 * t + 1) / kSlots) & 1,
                                               p.wait_ns));
        if (!ok) break;
        if (key0 + r >= L) {
          unsigned char* vrow = smem + kRingOff + ((2 * t + 1) % kSlots) * kTileBytes + r * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            *reinterpret_cast<uint4*>(vrow + c * 16) = make_uint4(0u, 0u, 0u, 0u);
            if constexpr (!F8) *reinterpret_cast<uint4*>(vrow + 16384 + c * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
      }
      // keys of this tile outside [ka, pos] are masked
      if (key0 < ka || key0 + kBN - 1 > pos) {
#pragma unroll
        for (int c = 0; c < kBN; ++c)
          if (key0 + c < ka || key0 + c > pos) s[c] = -INFINITY;
      }
      float mx8[8];  // eight independent chains, two new scores per step
      static_assert(kBN % 16 == 0, "max chains");
#pragma unroll
      for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(s[i], s[8 + i]);
#pragma unroll
      for (int c = 16; c < kBN; c += 16) {
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = max3(mx8[i], s[c + i], s[c + 8 + i]);
      }
      const float mt = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      // a new reference maximum only when the row's maximum grew by more than 2^8
      const bool grow = mt > m_ref + kRescaleLog2 || (m_ref == -INFINITY && mt != -INFINITY);
      const float m_new = grow ? mt : m_ref;
      if (t > 0 && __any_sync(0xffffffffu, grow && m_ref != -INFINITY)) {
        // O is rescaled. PV_q(t - 1) is done: it was issued before S_q(t),
        // whose completion this thread has seen
        const float alpha = (grow && m_ref != -INFINITY) ? fast_exp2(m_ref - m_new) : 1.f;
#pragma unroll
        for (int c = 0; c < kD / 32; ++c) {
          float v[32];
          tc05::ld_32x32b_x32(ocol + c * 32, v);
          tc05::wait_ld();
          tc05::reg_fence(v);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= alpha;
          tc05::st_32x32b_x32(ocol + c * 32, v);
        }
        l *= alpha;
      }
      m_ref = m_new;
      const float e = m_ref == -INFINITY ? 0.f : m_ref;
      float2 sm4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        if constexpr (F8) {
          // P as e4m3 hi + lo, four keys per column: hi over columns 0-31,
          // lo over 32-63 (this half: 16 + 16 of them)
          uint32_t ph[16], pl[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int k0 = 64 * half + 4 * i;
            const float2 d0 = sub2(make_float2(s[k0], s[k0 + 1]), e), d1 = sub2(make_float2(s[k0 + 2], s[k0 + 3]), e);
            const float p0 = fast_exp2(d0.x), p1 = fast_exp2(d0.y), p2 = fast_exp2(d1.x), p3 = fast_exp2(d1.y);
            sm4[(2 * i) & 3] = add2(sm4[(2 * i) & 3], make_float2(p0, p1));
            sm4[(2 * i + 1) & 3] = add2(sm4[(2 * i + 1) & 3], make_float2(p2, p3));
            tc05::e4m3_split4(p0, p1, p2, p3, ph[i], pl[i]);
          }
          tc05::st_32x32b_x16_u(scol + 16 * half, ph);
          tc05::st_32x32b_x16_u(scol + 32 + 16 * half, pl);
        } else {
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float2 dd = sub2(make_float2(s[64 * half + 2 * i], s[64 * half + 2 * i + 1]), e);
            const float p0 = fast_exp2(dd.x), p1 = fast_exp2(dd.y);
            sm4[i & 3] = add2(sm4[i & 3], make_float2(p0, p1));
            pk[i] = pack_bf16x2(p0, p1);
          }
          tc05::st_32x32b_x32_u(scol + 32 * half, pk);
        }
        // this half of P is in tensor memory: its products may start
        tc05::wait_st();
        tc05::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar((half == 0 ? kPLo : kPHi) + q));
      }
      l += ((sm4[0].x + sm4[0].y) + (sm4[1].x + sm4[1].y)) + ((sm4[2].x + sm4[2].y) + (sm4[3].x + sm4[3].y));
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(kODone), 0, p.wait_ns));
    if (!ok && lane == 0) fail(1);
    if (ok) {
      tc05::fence_after_sync();
      // ---- epilogue: O / l, lse = ln(sum exp(score))
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int c = 0; c < kD / 32; ++c) {
        float v[32];
        tc05::ld_32x32b_x32(ocol + c * 32, v);
        tc05::wait_ld();
        tc05::reg_fence(v);
        if (live) {
          if (p.out_dtype == kDtypeBf16) {
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
              *reinterpret_cast<float4*>(dst + i) =
                  make_float4(v[i] * inv, v[i + 1] * inv, v[i + 2] * inv, v[i + 3] * inv);
          }
        }
      }
      if (live && p.lse_out != nullptr)
        p.lse_out[grow_row] = l > 0.f ? (m_ref + log2f(l)) * 0.69314718055994530942f : -INFINITY;
    }
  }

  // ---- teardown: every role is done with tensor memory
  tc05::fence_before_sync();
  __syncthreads();
  if (warp == 9) {
    if (*reinterpret_cast<volatile int*>(&s_abort)) {
      // products may still be in flight after a timeout: wait (bounded) for
      // them before the columns are released
      if (lane == 0) {
        tc05::commit(bar(kDrain));
        (void)mbar_wait(bar(kDrain), 0, kWaitLimitNs);
      }
      __syncwarp();
    }
    tc05::fence_after_sync();
    tc05::tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool PG, bool F8>
cudaError_t launch_prefill_t(const Tc05Params& p, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tq,
                             cudaStream_t stream) {
  auto kern = attn_tc05_prefill_kernel<PG, F8>;
  // the register split holds only for the launch count it was made for: a
  // build that launches with fewer registers would leave setmaxnreg.inc
  // waiting for registers that never come, so such a build is not launched
  static int launch_regs = -1;
  if (launch_regs < 0) {
    cudaFuncAttributes fa;
    cudaError_t ea = cudaFuncGetAttributes(&fa, kern);
    if (ea != cudaSuccess) return ea;
    launch_regs = fa.numRegs;
  }
  if (launch_regs != kRegsLaunch) return cudaErrorInvalidConfiguration;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.batch) * p.h_kv * p.row_blocks);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tk, tv, tq, p);
}

}  // namespace

int tc05_prefill_rows_per_block() { return kQT * kBM; }

cudaError_t launch_tc05_prefill(const Tc05Params& p, const CUtensorMap& tk, const CUtensorMap& tv,
                                const CUtensorMap& tq, cudaStream_t stream) {
  if (p.f8) return p.paged ? cudaErrorInvalidValue : launch_prefill_t<false, true>(p, tk, tv, tq, stream);
  return p.paged ? launch_prefill_t<true, false>(p, tk, tv, tq, stream) : launch_prefill_t<false, false>(p, tk, tv, tq, stream);
}

}  // namespace mqa
