// gqa_decode_attention on tensor cores for a paged bf16 cache of 16-token
// pages, head_dim 128: one block per (sequence, group of HG kv heads, split).
//
// In the page pool [num_pages, h_kv, 16, 128] the slices of HG consecutive kv
// heads of a page are one contiguous run of HG x 4 KB. One TMA box fetches
// that run, so every HBM access is HG x 4 KB long instead of 4 KB (measured
// on GB300: 4 KB runs cap the stream near 5.3 TB/s, 16 KB runs stream at
// about 7 TB/s). Pages are gathered through the block table ("KV Cache
// 최적화 심층 분석", PagedKVCache; "Arsitektur Inferensi LLM", section 4).
//
// Block = HG consumer warps + 1 producer warp. Each stage holds one page of
// the HG heads; consumer warp w owns kv head jg * HG + w and its G <= 16
// query heads (the MMA rows), runs its own online softmax over all tokens of
// the block's range, and writes its rows itself: no cross-warp merge.
#include <cuda_bf16.h>

#include "../../include/mqa_decode.h"
#include "launch.h"
#include "mma_warp.cuh"
#include "ptx.cuh"

#ifndef MQA_HEADS_STAGES
#define MQA_HEADS_STAGES 3
#endif

namespace mqa {
namespace {

constexpr int kPage = 16;  // tokens per page (and per stage)

template <int HG, int STAGES>
struct HeadsCfg {
  static constexpr int D = 128;
  static constexpr int kConsumerWarps = HG;
  static constexpr int kThreads = 32 * (HG + 1);
  static constexpr int kHeadBytes = kPage * D * 2;  // one head's page: 4 KB
  static constexpr int kBoxBytes = HG * kHeadBytes;
  static constexpr int kStageBytes = 2 * kBoxBytes;  // K and V
  static constexpr int kSmemBytes = STAGES * kStageBytes + 2 * STAGES * 8 + 1024;
};

template <int HG, int STAGES>
__global__ void __launch_bounds__(HeadsCfg<HG, STAGES>::kThreads)
    decode_mma_heads_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                            const DecodeParams p) {
  using C = HeadsCfg<HG, STAGES>;
  constexpr int D = C::D;
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
      mbar_init(smem_u32(&empty[s]), C::kConsumerWarps);
    }
    fence_mbar_init();
  }
  if (warp == C::kConsumerWarps && lane == 0) {
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
  }
  __syncthreads();
  // See decode_mma.cu: after the append kernel everything but q_rot and the
  // new token's row may be read before the dependency wait.
  // the combine (or the next step) may be scheduled now; it waits for this
  // whole grid before it reads anything this grid writes
  grid_dependents_launch();
  if (!p.early) grid_dependency_wait();
  long long limit = static_cast<long long>(p.max_pages) * kPage;
  if (limit > p.max_seq_len) limit = p.max_seq_len;
  int L = p.seq_lens[b];
  if (L < 1 || L > limit) {
    if (threadIdx.x == 0 && split == 0 && jg == 0) atomicOr(p.err, static_cast<int>(MQA_DEVERR_SEQ_LEN));
    L = L < 0 ? 0 : static_cast<int>(L > limit ? limit : L);
  }
  // sliding window: tokens [t_lo, L); splits start at t_lo's page
  const int t_lo = p.window > 0 ? max(0, L - p.window) : 0;
  const int t_base = (t_lo / kPage) * kPage;
  const int t_begin = t_base + split * p.chunk;
  const int t_end = min(L, t_begin + p.chunk);
  const int n_tiles = t_end > t_begin ? (t_end - t_begin + kPage - 1) / kPage : 0;

  // the fused append (no append launch precedes this one): one block per
  // sequence and group of kv heads writes the new token's rows
  const int apos = p.fuse_append ? p.pos[b] : 0;
  const bool awaits = p.fuse_append && split == append_split(apos - t_base, p.chunk, S);
  if (warp == C::kConsumerWarps) {
    // ------------------------------------------------------------ producer
    const int32_t* trow = p.block_table + static_cast<long long>(b) * p.max_pages;
    const int n_pages_seq = (L + kPage - 1) / kPage;
    int wbase = t_begin / kPage;  // logical page window [wbase, wbase + 32), next window preloaded
    int wcur = (wbase + lane < n_pages_seq) ? __ldg(trow + wbase + lane) : -1;
    int wnxt = (wbase + 32 + lane < n_pages_seq) ? __ldg(trow + wbase + 32 + lane) : -1;
    int issued = 0;
    bool waited = !p.early;
    // the fused append, by this warp (a sixth warp for it measured slower
    // here): its reads issued now, its rows written once the first pages are
    // in flight, and fenced just before the page that holds them
    AppendRows<D, HG> ar;
    if (awaits) ar.load(p, b, jg * HG, apos, lane);
    bool written = !awaits, published = !awaits;
    for (int it = 0; it < n_tiles; ++it) {
      const int stage = it % STAGES;
      if (!written && it == STAGES) {
        ar.write(p, apos, lane);
        written = true;
      }
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
      const int t0 = t_begin + it * kPage;
      if (!waited && L - 1 < t0 + kPage) {  // this page holds the appended token
        grid_dependency_wait();
        waited = true;
      }
      if (!published && apos < t0 + kPage) {  // this page holds the rows this block appends
        if (!written) ar.write(p, apos, lane);
        written = true;
        ar.publish();
        published = true;
      }
      const int lp = t0 / kPage;  // < n_pages_seq since t0 < t_end <= L
      while (lp >= wbase + 32) {  // warp-uniform window advance
        wbase += 32;
        wcur = wnxt;
        wnxt = (wbase + 32 + lane < n_pages_seq) ? __ldg(trow + wbase + 32 + lane) : -1;
      }
      const int page = __shfl_sync(0xffffffffu, wcur, lp - wbase);
      if (lane == 0) {
        // a bad entry reads the TMA fill value (out-of-range coordinate); it is reported
        if (page < 0 || page >= p.num_pages) atomicOr(p.err, static_cast<int>(MQA_DEVERR_PAGE_RANGE));
        const uint32_t kdst = smem_u32(smem + stage * C::kStageBytes);
        const uint32_t fb = smem_u32(&full[stage]);
        mbar_arrive_expect_tx(fb, C::kStageBytes);
        tma_load_5d(kdst, &tmap_k, 0, 0, 0, jg * HG, page, fb);
        tma_load_5d(kdst + C::kBoxBytes, &tmap_v, 0, 0, 0, jg * HG, page, fb);
      }
      __syncwarp();
      issued = it + 1;
    }
    if (!written) ar.write(p, apos, lane);  // rows this block never reads
    // every copy this warp issued lands before the block can exit: after a
    // timeout the consumers may have stopped waiting for them
    for (int it = (issued > STAGES ? issued - STAGES : 0); it < issued; ++it)
      (void)mbar_wait(smem_u32(&full[it % STAGES]), (it / STAGES) & 1, kWaitLimitNs);
    return;
  }

  // -------------------------------------------------------------- consumers
  const int j = jg * HG + warp;  // this warp's kv head
  const int r0 = lane >> 2, c2 = (lane & 3) * 2;
  WarpAttn<D> wa;
  if (p.rope_q) {
    // rotate q_new here: nothing the consumers read comes from the append kernel
    // (the q loads are issued before the cos / sin table is formed)
    __shared__ float s_cs[D];
    const long long qoff = (static_cast<long long>(b) * p.h_q + j * G) * D;
    uint32_t qraw[D / 16][4];
    WarpAttn<D>::load_q(static_cast<const __nv_bfloat16*>(p.q_new) + qoff, G, lane, qraw);
    rope_table<D>(s_cs, p, p.pos[b], threadIdx.x, 2, C::kConsumerWarps * 32);
    wa.init_rope(qraw, G, s_cs, p.scale_log2, lane, (p.fuse_append && split == 0) ? p.q_rot_out + qoff : nullptr);
  } else {
    if (p.early) grid_dependency_wait();  // q_rot comes from the append kernel
    wa.init(p.q_rot + (static_cast<long long>(b) * p.h_q + j * G) * D, G, p.scale_log2, lane);
  }

  bool ok = true;
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
    const int t0 = t_begin + it * kPage;
    const int lo = max(0, t_lo - t0), hi = min(kPage, t_end - t0);  // lo < hi: the page holds a window token
    unsigned char* kt = smem + stage * C::kStageBytes + warp * C::kHeadBytes;
    unsigned char* vt = kt + C::kBoxBytes;
    wa.step(smem_u32(kt), smem_u32(vt), vt, 0, lo, hi, 4, lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[stage]));
  }
  wa.finish_sums();
  if (!ok || *reinterpret_cast<volatile int*>(&s_abort)) return;

  // ------------------------------------------------ this warp's rows out
  const float i0 = wa.l0 > 0.f ? 1.f / wa.l0 : 0.f;
  const float i1 = wa.l1 > 0.f ? 1.f / wa.l1 : 0.f;
  const long long row0 = static_cast<long long>(b) * p.h_q + j * G;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int r = r0 + 8 * half;
    if (r >= G) continue;
    const float inv = half ? i1 : i0;
    const float l = half ? wa.l1 : wa.l0;
    const float m = half ? wa.m1 : wa.m0;
    const long long grow = row0 + r;
    const float lse = l > 0.f ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
    if (S > 1) {
      float* dst = p.o_part + (grow * S + split) * D;
#pragma unroll
      for (int n = 0; n < D / 8; ++n)
        *reinterpret_cast<float2*>(dst + n * 8 + c2) = make_float2(wa.o[n][2 * half] * inv, wa.o[n][2 * half + 1] * inv);
      if ((lane & 3) == 0) p.lse_part[grow * S + split] = lse;
    } else {
      if (p.out_dtype == kDtypeBf16) {
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + grow * D;
#pragma unroll
        for (int n = 0; n < D / 8; ++n)
          *reinterpret_cast<uint32_t*>(dst + n * 8 + c2) =
              pack_bf16x2(wa.o[n][2 * half] * inv, wa.o[n][2 * half + 1] * inv);
      } else {
        float* dst = static_cast<float*>(p.out) + grow * D;
#pragma unroll
        for (int n = 0; n < D / 8; ++n)
          *reinterpret_cast<float2*>(dst + n * 8 + c2) =
              make_float2(wa.o[n][2 * half] * inv, wa.o[n][2 * half + 1] * inv);
      }
      if ((lane & 3) == 0 && p.lse_out != nullptr) p.lse_out[grow] = lse;
    }
  }
}

template <int HG>
cudaError_t launch_heads_t(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                           cudaStream_t stream) {
  constexpr int ST = MQA_HEADS_STAGES;
  using C = HeadsCfg<HG, ST>;
  auto kern = decode_mma_heads_kernel<HG, ST>;
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
  return cudaLaunchKernelEx(&cfg, kern, tk, tv, p);
}

}  // namespace

int decode_mma_heads_group(const DecodeParams& p) {
  if (!p.paged || p.page_size != kPage || p.head_dim != 128 || p.group > 16 || p.n_new > 1) return 0;
  if (p.h_kv % 4 == 0) return 4;
  if (p.h_kv % 2 == 0) return 2;
  return 0;
}

KernelShape decode_mma_heads_shape(int hg) {
  if (hg == 4) return {HeadsCfg<4, MQA_HEADS_STAGES>::kThreads, HeadsCfg<4, MQA_HEADS_STAGES>::kSmemBytes, 0, 0};
  return {HeadsCfg<2, MQA_HEADS_STAGES>::kThreads, HeadsCfg<2, MQA_HEADS_STAGES>::kSmemBytes, 0, 0};
}

cudaError_t launch_decode_mma_heads(const DecodeParams& p, int hg, const CUtensorMap& tk, const CUtensorMap& tv,
                                    cudaStream_t stream) {
  if (hg == 4) return launch_heads_t<4>(p, tk, tv, stream);
  return launch_heads_t<2>(p, tk, tv, stream);
}

}  // namespace mqa
