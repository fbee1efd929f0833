// Causal attention of the last n_new tokens of every sequence -- prefill,
// "KV Cache" explainer, Langkah 1 and 4: the prompt's keys and values are
// computed in one pass and stored, and the work is compute-bound -- on the
// 5th-generation tensor cores.
//
// Block = (sequence b, query head h, 128 consecutive new tokens). Query row r
// (token t0 + r, position p = L - n_new + t0 + r) attends to the keys
// [max(0, p + 1 - W) if windowed else 0, p] of kv head floor(h / G). For each
// 128-key tile of that range:
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
// Warps: 0-3 softmax and epilogue (row = thread), 4 K loader, 5 V loader
// (TMA, 3 stages each; a K stage is released when its S is computed, a V
// stage when its PV is), 6 MMA issue (one thread) and tensor-memory
// allocation.
#include <cuda_bf16.h>

#include "../../include/mqa_decode.h"
#include "launch.h"
#include "ptx.cuh"
#include "tc05.cuh"

namespace mqa {
namespace {

constexpr int kD = 128;       // head_dim
constexpr int kBM = 128;      // query rows (tokens of one head) per block
constexpr int kBN = 128;      // keys per tile
constexpr int kStages = 3;    // K tiles and V tiles in flight
constexpr int kThreads = 224;
constexpr int kTileBytes = kBN * kD * 2;                 // 32 KB: [2 halves][128 rows][128 B]
constexpr int kQOff = 0;
constexpr int kKOff = kTileBytes;                        // K stages
constexpr int kVOff = kKOff + kStages * kTileBytes;      // V stages
constexpr int kBarOff = kVOff + kStages * kTileBytes;
constexpr int kSmemBytes = kBarOff + 256 + 1024;
constexpr uint32_t kTmemCols = 512;                      // S0, S1, O (+ unused)
constexpr uint32_t kColS = 0, kColO = 256;
constexpr float kRescaleLog2 = 8.0f;

// mbarriers (8 bytes each) at kBarOff
enum Bar {
  kQReady = 0,
  kKFull = 1,    // [kStages]
  kKEmpty = 4,   // [kStages]
  kVFull = 7,    // [kStages]
  kVEmpty = 10,  // [kStages]
  kSFull = 13,   // [2]
  kPFull = 15,   // [2]
  kODone = 17,   // [2]
  kDrain = 19,
  kNBars = 20
};

__device__ __forceinline__ uint32_t sw128(int r, int col) {  // byte offset of bf16 element (r, col) of a tile
  const int half = col >> 6, chunk = (col & 63) >> 3;
  return half * 16384 + r * 128 + ((chunk ^ (r & 7)) << 4) + (col & 7) * 2;
}

__device__ __forceinline__ bool aborted(const PrefillParams& p) {
  return (*reinterpret_cast<volatile int32_t*>(p.err) & static_cast<int>(MQA_DEVERR_TIMEOUT)) != 0;
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                   const PrefillParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + kBarOff + kNBars * 8);
  __shared__ int s_abort, s_skip;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.group, n = p.n_new;
  const int n_mb = (n + kBM - 1) / kBM;
  int cta = blockIdx.x;
  const int hg = cta % G;
  cta /= G;
  const int j = cta % p.h_kv;
  cta /= p.h_kv;
  const int b = cta % p.batch;
  const int mb = n_mb - 1 - cta / p.batch;  // the longest key ranges first
  const int h = j * G + hg;
  const int t0 = mb * kBM;
  const int rows = min(kBM, n - t0);

  long long limit = p.capacity < p.max_seq_len ? p.capacity : p.max_seq_len;
  const int L = p.seq_lens[b];
  if (L < n || L > limit) {
    if (tid == 0 && mb == 0 && h == 0) atomicOr(p.err, static_cast<int>(MQA_DEVERR_SEQ_LEN));
    return;
  }
  if (tid == 0) s_skip = aborted(p) ? 1 : 0;  // an earlier block timed out: the result is invalid already
  __syncthreads();
  if (s_skip) return;
  const int Lp = L - n;    // prefix length: token t0 + r sits at position Lp + t0 + r
  const int pos_first = Lp + t0, pos_last = Lp + t0 + rows - 1;
  const int ka_first = p.window > 0 ? max(0, pos_first + 1 - p.window) : 0;
  const int kt0 = ka_first / kBN;
  const int T = (pos_last + 1 + kBN - 1) / kBN - kt0;  // key tiles of this block

  if (tid == 0) {
    s_abort = 0;
    mbar_init(bar(kQReady), 4);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kKFull + s), 1);
      mbar_init(bar(kKEmpty + s), 1);
      mbar_init(bar(kVFull + s), 1);
      mbar_init(bar(kVEmpty + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kSFull + s), 1);
      mbar_init(bar(kPFull + s), 4);
      mbar_init(bar(kODone + s), 1);
    }
    mbar_init(bar(kDrain), 1);
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

  auto fail = [&](int role_lane0) {
    if (role_lane0) {
      s_abort = 1;
      atomicOr(p.err, static_cast<int>(MQA_DEVERR_TIMEOUT));
    }
  };
  auto stop = [&]() { return *reinterpret_cast<volatile int*>(&s_abort) != 0; };

  if (warp == 4 || warp == 5) {
    // ------------------------------------------------- K (warp 4) / V (warp 5) loaders
    if (lane == 0) {
      const bool is_k = warp == 4;
      const CUtensorMap* map = is_k ? &tmap_k : &tmap_v;
      const int full = is_k ? kKFull : kVFull, empty = is_k ? kKEmpty : kVEmpty;
      const uint32_t dst0 = sbase + (is_k ? kKOff : kVOff);
      const int row = b * p.h_kv + j;
      for (int it = 0; it < T; ++it) {
        const int s = it % kStages;
        if (it >= kStages && !mbar_wait(bar(empty + s), ((it - kStages) / kStages) & 1)) {
          fail(1);
          break;
        }
        if (stop()) break;
        mbar_arrive_expect_tx(bar(full + s), kTileBytes);
        tma_load_4d(dst0 + s * kTileBytes, map, 0, (kt0 + it) * kBN, 0, row, bar(full + s));
      }
    }
    __syncwarp();
  } else if (warp == 6) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      const uint32_t id_s = tc05::idesc_bf16_f32(kBM, kBN, false, false);
      const uint32_t id_o = tc05::idesc_bf16_f32(kBM, kD, false, true);
      const uint32_t q_s = sbase + kQOff;
      bool ok = mbar_wait(bar(kQReady), 0);
      // S of tile it into buffer it % 2. That buffer last held P of tile it - 2,
      // whose PV was issued before: MMAs of this thread execute in order.
      auto issue_s = [&](int it) -> bool {
        const int s = it % kStages, sb = it & 1;
        if (!mbar_wait(bar(kKFull + s), (it / kStages) & 1)) return false;
        tc05::fence_after_sync();
        const uint32_t k_s = sbase + kKOff + s * kTileBytes;
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
          const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
          tc05::mma_bf16(tmem + kColS + sb * 128, tc05::smem_desc_sw128(q_s + off, 16, 1024),
                         tc05::smem_desc_sw128(k_s + off, 16, 1024), id_s, ks > 0);
        }
        tc05::commit(bar(kSFull + sb));
        tc05::commit(bar(kKEmpty + s));
        return true;
      };
      auto issue_pv = [&](int it) -> bool {
        const int s = it % kStages, pb = it & 1;
        if (!mbar_wait(bar(kPFull + pb), (it >> 1) & 1)) return false;
        if (!mbar_wait(bar(kVFull + s), (it / kStages) & 1)) return false;
        tc05::fence_after_sync();
        const uint32_t v_s = sbase + kVOff + s * kTileBytes;
#pragma unroll
        for (int ks = 0; ks < kBN / 16; ++ks)
          tc05::mma_bf16_ta(tmem + kColO, tmem + kColS + pb * 128 + ks * 8,
                            tc05::smem_desc_sw128(v_s + ks * 2048, 16384, 1024), id_o, it > 0 || ks > 0);
        tc05::commit(bar(kODone + pb));
        tc05::commit(bar(kVEmpty + s));
        return true;
      };
      if (ok && T > 0) ok = issue_s(0);
      for (int it = 0; ok && it < T; ++it) {
        if (stop()) {
          ok = false;
          break;
        }
        if (it + 1 < T && !issue_s(it + 1)) ok = false;
        if (ok && !issue_pv(it)) ok = false;
      }
      if (!ok) fail(1);
    }
    __syncwarp();
  } else {
    // --------------------------------------------------- softmax (row = tid)
    const int r = tid;
    const bool live = r < rows;
    {
      // Q row, pre-scaled into the log2 domain, as bf16 in the swizzled tile
      const float* q = p.q_rot + ((static_cast<long long>(b) * n + t0 + r) * p.h_q + h) * kD;
#pragma unroll 4
      for (int c = 0; c < kD; c += 8) {
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f), bq = a;
        if (live) {
          a = *reinterpret_cast<const float4*>(q + c);
          bq = *reinterpret_cast<const float4*>(q + c + 4);
        }
        uint4 v;
        v.x = pack_bf16x2(a.x * p.scale_log2, a.y * p.scale_log2);
        v.y = pack_bf16x2(a.z * p.scale_log2, a.w * p.scale_log2);
        v.z = pack_bf16x2(bq.x * p.scale_log2, bq.y * p.scale_log2);
        v.w = pack_bf16x2(bq.z * p.scale_log2, bq.w * p.scale_log2);
        *reinterpret_cast<uint4*>(smem + kQOff + sw128(r, c)) = v;
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kQReady));
    }
    const int pos = live ? Lp + t0 + r : -1;  // last key of this row (none for padding rows)
    const int ka = p.window > 0 ? max(0, pos + 1 - p.window) : 0;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int it = 0; it < T; ++it) {
      const int sb = it & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(kSFull + sb), (it >> 1) & 1) && !stop());
      if (!ok) break;
      tc05::fence_after_sync();
      float s[kBN];
      // four loads in flight, one wait
      tc05::ld_32x32b_x32(tmem + lane_base + kColS + sb * 128 + 0, *reinterpret_cast<float(*)[32]>(&s[0]));
      tc05::ld_32x32b_x32(tmem + lane_base + kColS + sb * 128 + 32, *reinterpret_cast<float(*)[32]>(&s[32]));
      tc05::ld_32x32b_x32(tmem + lane_base + kColS + sb * 128 + 64, *reinterpret_cast<float(*)[32]>(&s[64]));
      tc05::ld_32x32b_x32(tmem + lane_base + kColS + sb * 128 + 96, *reinterpret_cast<float(*)[32]>(&s[96]));
      tc05::wait_ld();
#pragma unroll
      for (int c = 0; c < kBN; c += 32) tc05::reg_fence(*reinterpret_cast<float(*)[32]>(&s[c]));
      // keys of this tile outside [ka, pos] are masked
      const int key0 = (kt0 + it) * kBN;
      if (key0 + kBN > L) {
        // cache rows past the sequence may hold anything (NaN bit patterns
        // included); P = 0 there, and 0 * NaN would still poison O: zero the
        // V row of this thread's key once that tile has landed
        ok = __all_sync(0xffffffffu, mbar_wait(bar(kVFull + it % kStages), (it / kStages) & 1));
        if (!ok) break;
        if (key0 + r >= L) {
          unsigned char* vrow = smem + kVOff + (it % kStages) * kTileBytes + r * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            *reinterpret_cast<uint4*>(vrow + c * 16) = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(vrow + 16384 + c * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
      }
      if (key0 < ka || key0 + kBN - 1 > pos) {
#pragma unroll
        for (int c = 0; c < kBN; ++c)
          if (key0 + c < ka || key0 + c > pos) s[c] = -INFINITY;
      }
      float mx8[8];  // eight independent chains
#pragma unroll
      for (int i = 0; i < 8; ++i) mx8[i] = s[i];
#pragma unroll
      for (int c = 8; c < kBN; c += 8) {
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
        ok = __all_sync(0xffffffffu, mbar_wait(bar(kODone + ((it - 1) & 1)), ((it - 1) >> 1) & 1) && !stop());
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
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t pk[32];  // P of keys 64 half .. 64 half + 63 as bf16 pairs
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float p0 = fast_exp2(s[64 * half + 2 * i] - e), p1 = fast_exp2(s[64 * half + 2 * i + 1] - e);
          sm8[(2 * i) & 7] += p0;
          sm8[(2 * i + 1) & 7] += p1;
          pk[i] = pack_bf16x2(p0, p1);
        }
        tc05::st_32x32b_x32_u(tmem + lane_base + kColS + sb * 128 + 32 * half, pk);
      }
      l += ((sm8[0] + sm8[1]) + (sm8[2] + sm8[3])) + ((sm8[4] + sm8[5]) + (sm8[6] + sm8[7]));
      tc05::wait_st();
      tc05::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kPFull + sb));
    }
    if (ok && T > 0) ok = __all_sync(0xffffffffu, mbar_wait(bar(kODone + ((T - 1) & 1)), ((T - 1) >> 1) & 1));
    if (!ok) {
      if (lane == 0) fail(1);
    } else {
      tc05::fence_after_sync();
      // ---- epilogue: O / l, lse = ln(sum exp(score))
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const long long grow_row = (static_cast<long long>(b) * n + t0 + r) * p.h_q + h;
#pragma unroll
      for (int c = 0; c < kD / 32; ++c) {
        float v[32];
        tc05::ld_32x32b_x32(tmem + lane_base + kColO + c * 32, v);
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
              *reinterpret_cast<float4*>(dst + i) = make_float4(v[i] * inv, v[i + 1] * inv, v[i + 2] * inv,
                                                                v[i + 3] * inv);
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

}  // namespace

KernelShape prefill_shape() { return {kThreads, kSmemBytes, kBM, 1}; }

cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const int n_mb = (p.n_new + kBM - 1) / kBM;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.batch) * p.h_q * n_mb);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, prefill_kernel, tk, tv, p);
}

}  // namespace mqa
