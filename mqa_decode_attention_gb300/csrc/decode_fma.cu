// gqa_decode_attention on CUDA cores (fp32 FMA), for bf16 and fp32 caches.
//
// Computes, for the query heads of one kv head j = g(h) and one token range
// of sequence b, O_h = softmax(scale * q_h K_j^T) V_j ("Grouped-query
// attention" page, equations for A_h and O_h), with FlashAttention's running
// max and sum so the scores never leave the chip ("Arsitektur Inferensi LLM",
// section 5).
//
// Block = 4 consumer warps + 1 producer warp. The producer streams K and V
// tiles of 64 tokens into a ring of shared-memory stages with 1-D bulk copies
// (TMA), one mbarrier pair per stage. A consumer lane owns a 16-byte slice of
// a token row: lanes per token = row bytes / 16 (max 16), so each quarter-warp
// reads 128 contiguous bytes (no bank conflicts). Every lane keeps q and the
// output accumulator for its slice and for HBLK query heads; scores are
// reduced across the lanes of a token with xor shuffles. Each lane group runs
// its own online softmax over its tokens; the groups merge once at the end.
#include <cuda_bf16.h>

#include "../../include/mqa_decode.h"
#include "launch.h"
#include "ptx.cuh"

namespace mqa {
namespace {

template <typename T, int D, int HBLK, int STAGES>
struct FmaCfg {
  static constexpr int kEsize = sizeof(T);
  static constexpr int kRowBytes = D * kEsize;
  static constexpr int kChunksPerRow = kRowBytes / 16;
  static constexpr int kLPT = kChunksPerRow >= 16 ? 16 : kChunksPerRow;  // lanes per token
  static constexpr int kVPL = kChunksPerRow / kLPT;                       // 16-byte vectors per lane
  static constexpr int kEPC = 16 / kEsize;                                // elements per vector
  static constexpr int kEPL = kVPL * kEPC;                                // elements per lane
  static constexpr int kConsumerThreads = 128;
  static constexpr int kConsumerWarps = kConsumerThreads / 32;
  static constexpr int kGroups = kConsumerThreads / kLPT;  // token groups
  static constexpr int kTPG = kTile / kGroups;             // tokens per group per tile
  static constexpr int kThreads = kConsumerThreads + 32;
  static constexpr int kTileBytes = kTile * kRowBytes;
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kMergeStride = D + 4;  // floats per merged row
  static constexpr int kMergeBytes = kGroups * HBLK * kMergeStride * 4 + 2 * kGroups * HBLK * 4;
  static constexpr int kBodyBytes = (STAGES * kStageBytes > kMergeBytes) ? STAGES * kStageBytes : kMergeBytes;
  static constexpr int kSmemBytes = kBodyBytes + 2 * STAGES * 8 + 128;
  static_assert(kRowBytes % 16 == 0, "row must be a whole number of 16-byte vectors");
  static_assert(kTile % kGroups == 0, "tile must split evenly over token groups");
};

template <typename T>
__device__ __forceinline__ void unpack16(const uint4& v, float* out);

template <>
__device__ __forceinline__ void unpack16<__nv_bfloat16>(const uint4& v, float* out) {
  out[0] = bf16lo_to_f32(v.x);
  out[1] = bf16hi_to_f32(v.x);
  out[2] = bf16lo_to_f32(v.y);
  out[3] = bf16hi_to_f32(v.y);
  out[4] = bf16lo_to_f32(v.z);
  out[5] = bf16hi_to_f32(v.z);
  out[6] = bf16lo_to_f32(v.w);
  out[7] = bf16hi_to_f32(v.w);
}

template <>
__device__ __forceinline__ void unpack16<float>(const uint4& v, float* out) {
  out[0] = __uint_as_float(v.x);
  out[1] = __uint_as_float(v.y);
  out[2] = __uint_as_float(v.z);
  out[3] = __uint_as_float(v.w);
}

// Logical page window of the producer warp: lane l holds the block-table entry
// of logical page (base + l); the next window is loaded one window ahead.
struct PageWindow {
  const int32_t* row;
  int n_valid;  // logical pages the sequence owns
  int base;
  int cur, nxt;
  __device__ __forceinline__ int load(int lp, int lane) const {
    const int i = lp + lane;
    return i < n_valid ? __ldg(row + i) : -1;
  }
  __device__ __forceinline__ void init(const int32_t* r, int n, int first, int lane) {
    row = r;
    n_valid = n;
    base = first;
    cur = load(base, lane);
    nxt = load(base + 32, lane);
  }
  // warp-uniform call: physical page of logical page lp (>= base)
  __device__ __forceinline__ int page(int lp, int lane) {
    while (lp >= base + 32) {
      base += 32;
      cur = nxt;
      nxt = load(base + 32, lane);
    }
    return __shfl_sync(0xffffffffu, cur, lp - base);
  }
};

template <typename T, int D, int HBLK, int STAGES>
__global__ void __launch_bounds__(FmaCfg<T, D, HBLK, STAGES>::kThreads)
    decode_fma_kernel(const DecodeParams p) {
  using C = FmaCfg<T, D, HBLK, STAGES>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
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
  const int head0 = hsb * HBLK;                 // first head of this block within the group
  const int n_heads = min(HBLK, G - head0);     // heads this block serves

  // --- sequence length, validated against the cache it must fit in
  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), C::kConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  // q_rot and the appended slot come from the preceding append launch.
  // the combine (or the next step) may be scheduled now; it waits for this
  // whole grid before it reads anything this grid writes
  grid_dependents_launch();
  grid_dependency_wait();
  // Lengths are read only after the preceding grid is complete and visible.
  long long limit = p.paged ? static_cast<long long>(p.max_pages) * p.page_size : p.capacity;
  if (limit > p.max_seq_len) limit = p.max_seq_len;
  int L = p.seq_lens[b];
  if (L < 1 || L > limit) {
    if (threadIdx.x == 0 && split == 0 && hsb == 0) atomicOr(p.err, static_cast<int>(MQA_DEVERR_SEQ_LEN));
    L = L < 0 ? 0 : static_cast<int>(L > limit ? limit : L);
  }
  // sliding window: tokens [t_lo, L); splits start at t_lo rounded down to a tile
  const int t_lo = p.window > 0 ? max(0, L - p.window) : 0;
  const int t_begin = (t_lo / kTile) * kTile + split * p.chunk;
  const int t_end = min(L, t_begin + p.chunk);
  const int n_tiles = t_end > t_begin ? (t_end - t_begin + kTile - 1) / kTile : 0;


  const T* kbase = static_cast<const T*>(p.k_cache);
  const T* vbase = static_cast<const T*>(p.v_cache);

  if (warp == C::kConsumerWarps) {
    // ------------------------------------------------------------ producer
    PageWindow win;
    const int ps = p.page_size;
    if (p.paged) win.init(p.block_table + static_cast<long long>(b) * p.max_pages, (L + ps - 1) / ps, t_begin / ps, lane);
    // (pages before the window are skipped below; the window may start past
    //  t_begin, and win.page only moves forward)
    int issued = 0;
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
      const int nrow = min(kTile, t_end - t0);
      const uint32_t kdst = smem_u32(smem + stage * C::kStageBytes);
      const uint32_t vdst = kdst + C::kTileBytes;
      const uint32_t fb = smem_u32(&full[stage]);
      if (!p.paged) {
        if (lane == 0) {
          const long long off = ((static_cast<long long>(b) * p.h_kv + j) * p.capacity + t0) * D;
          const uint32_t bytes = nrow * C::kRowBytes;
          mbar_arrive_expect_tx(fb, 2 * bytes);
          bulk_g2s(kdst, kbase + off, bytes, fb);
          bulk_g2s(vdst, vbase + off, bytes, fb);
        }
      } else {
        const int rpc = ps < kTile ? ps : kTile;  // rows per copy
        const int pieces = (nrow + rpc - 1) / rpc;
        int pg[kTile / 16];
        uint32_t total = 0;
#pragma unroll
        for (int k = 0; k < kTile / 16; ++k) {
          pg[k] = -1;
          if (k < pieces && t0 + (k + 1) * rpc > t_lo) {  // pieces wholly before the window are not read
            const int t = t0 + k * rpc;
            pg[k] = win.page(t / ps, lane);
            if (pg[k] < 0 || pg[k] >= p.num_pages) {
              if (lane == 0) atomicOr(p.err, static_cast<int>(MQA_DEVERR_PAGE_RANGE));
              pg[k] = -1;
            } else {
              total += 2u * min(rpc, nrow - k * rpc) * C::kRowBytes;
            }
          }
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(fb, total);
#pragma unroll
          for (int k = 0; k < kTile / 16; ++k) {
            if (k >= pieces || pg[k] < 0) continue;
            const int t = t0 + k * rpc;
            const uint32_t bytes = min(rpc, nrow - k * rpc) * C::kRowBytes;
            const long long off = ((static_cast<long long>(pg[k]) * p.h_kv + j) * ps + (t % ps)) * D;
            bulk_g2s(kdst + k * rpc * C::kRowBytes, kbase + off, bytes, fb);
            bulk_g2s(vdst + k * rpc * C::kRowBytes, vbase + off, bytes, fb);
          }
        }
      }
      __syncwarp();
      issued = it + 1;
    }
    // every copy this warp issued lands before the block can exit: after a
    // timeout the consumers may have stopped waiting for them
    for (int it = (issued > STAGES ? issued - STAGES : 0); it < issued; ++it)
      (void)mbar_wait(smem_u32(&full[it % STAGES]), (it / STAGES) & 1, kWaitLimitNs);
    return;
  }

  // -------------------------------------------------------------- consumers
  const int tid = threadIdx.x;
  const int gi = tid / C::kLPT;  // token group
  const int li = tid % C::kLPT;  // lane within the token
  float qv[HBLK][C::kEPL];
  float acc[HBLK][C::kEPL];
  float m[HBLK], l[HBLK];
  {
    const float* q = p.q_rot + (static_cast<long long>(b) * p.h_q + j * G + head0) * D;
#pragma unroll
    for (int h = 0; h < HBLK; ++h) {
#pragma unroll
      for (int v = 0; v < C::kVPL; ++v) {
#pragma unroll
        for (int e = 0; e < C::kEPC; ++e) {
          const int d = (li + v * C::kLPT) * C::kEPC + e;
          qv[h][v * C::kEPC + e] = h < n_heads ? q[h * D + d] * p.scale_log2 : 0.f;
          acc[h][v * C::kEPC + e] = 0.f;
        }
      }
      m[h] = -INFINITY;
      l[h] = 0.f;
    }
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
    const unsigned char* ktile = smem + stage * C::kStageBytes;
    const unsigned char* vtile = ktile + C::kTileBytes;
    const int nrow = min(kTile, t_end - (t_begin + it * kTile));
    const int lo_row = t_lo - (t_begin + it * kTile);  // rows before it are outside the window

    float s[C::kTPG][HBLK];
#pragma unroll
    for (int k = 0; k < C::kTPG; ++k) {
      const int row = gi + k * C::kGroups;
      float kv[C::kEPL];
#pragma unroll
      for (int v = 0; v < C::kVPL; ++v) {
        const uint4 raw =
            *reinterpret_cast<const uint4*>(ktile + row * C::kRowBytes + (li + v * C::kLPT) * 16);
        unpack16<T>(raw, kv + v * C::kEPC);
      }
#pragma unroll
      for (int h = 0; h < HBLK; ++h) {
        float dsum = 0.f;
#pragma unroll
        for (int e = 0; e < C::kEPL; ++e) dsum = fmaf(qv[h][e], kv[e], dsum);
        s[k][h] = dsum;
      }
    }
#pragma unroll
    for (int k = 0; k < C::kTPG; ++k) {
#pragma unroll
      for (int h = 0; h < HBLK; ++h) {
#pragma unroll
        for (int off = 1; off < C::kLPT; off <<= 1) s[k][h] += __shfl_xor_sync(0xffffffffu, s[k][h], off);
        const int row = gi + k * C::kGroups;
        if (row >= nrow || row < lo_row) s[k][h] = -INFINITY;
      }
    }
    float base[HBLK];
#pragma unroll
    for (int h = 0; h < HBLK; ++h) {
      float mt = s[0][h];
#pragma unroll
      for (int k = 1; k < C::kTPG; ++k) mt = fmaxf(mt, s[k][h]);
      const float mn = fmaxf(m[h], mt);
      const float alpha = mn == -INFINITY ? 1.f : exp2f(m[h] - mn);
      base[h] = mn == -INFINITY ? 0.f : mn;
      m[h] = mn;
      l[h] *= alpha;
#pragma unroll
      for (int e = 0; e < C::kEPL; ++e) acc[h][e] *= alpha;
    }
#pragma unroll
    for (int k = 0; k < C::kTPG; ++k) {
      const int row = gi + k * C::kGroups;
      if (row < nrow && row >= lo_row) {
        float vv[C::kEPL];
#pragma unroll
        for (int v = 0; v < C::kVPL; ++v) {
          const uint4 raw =
              *reinterpret_cast<const uint4*>(vtile + row * C::kRowBytes + (li + v * C::kLPT) * 16);
          unpack16<T>(raw, vv + v * C::kEPC);
        }
#pragma unroll
        for (int h = 0; h < HBLK; ++h) {
          const float pr = exp2f(s[k][h] - base[h]);
          l[h] += pr;
#pragma unroll
          for (int e = 0; e < C::kEPL; ++e) acc[h][e] = fmaf(pr, vv[e], acc[h][e]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[stage]));
  }

  // ----------------------------------------------- merge the token groups
  // one decision for every consumer warp (the producer may time out and set
  // s_abort at any moment); the barrier also ends their reads of the stages
  if (bar_any(2, C::kConsumerThreads, *reinterpret_cast<volatile int*>(&s_abort) || !ok)) return;
  float* mo = reinterpret_cast<float*>(smem);                       // [groups][HBLK][stride]
  float* mm = mo + C::kGroups * HBLK * C::kMergeStride;             // [groups][HBLK]
  float* ml = mm + C::kGroups * HBLK;                               // [groups][HBLK]
#pragma unroll
  for (int h = 0; h < HBLK; ++h) {
#pragma unroll
    for (int v = 0; v < C::kVPL; ++v) {
#pragma unroll
      for (int e = 0; e < C::kEPC; ++e)
        mo[(gi * HBLK + h) * C::kMergeStride + (li + v * C::kLPT) * C::kEPC + e] = acc[h][v * C::kEPC + e];
    }
    if (li == 0) {
      mm[gi * HBLK + h] = m[h];
      ml[gi * HBLK + h] = l[h];
    }
  }
  named_bar_sync(1, C::kConsumerThreads);

  const bool split_out = S > 1;
  for (int idx = tid; idx < n_heads * D; idx += C::kConsumerThreads) {
    const int h = idx / D, d = idx - h * D;
    float mx = -INFINITY;
    for (int g = 0; g < C::kGroups; ++g) mx = fmaxf(mx, mm[g * HBLK + h]);
    float num = 0.f, den = 0.f;
    if (mx != -INFINITY) {
      for (int g = 0; g < C::kGroups; ++g) {
        const float w = exp2f(mm[g * HBLK + h] - mx);
        num = fmaf(w, mo[(g * HBLK + h) * C::kMergeStride + d], num);
        den = fmaf(w, ml[g * HBLK + h], den);
      }
    }
    const float o = den > 0.f ? num / den : 0.f;
    const float lse = den > 0.f ? (mx + log2f(den)) * 0.69314718055994530942f : -INFINITY;
    const long long row = static_cast<long long>(b) * p.h_q + j * G + head0 + h;
    if (split_out) {
      p.o_part[(row * S + split) * D + d] = o;
      if (d == 0) p.lse_part[row * S + split] = lse;
    } else {
      if (p.out_dtype == kDtypeBf16)
        static_cast<__nv_bfloat16*>(p.out)[row * D + d] = __float2bfloat16_rn(o);
      else
        static_cast<float*>(p.out)[row * D + d] = o;
      if (d == 0 && p.lse_out != nullptr) p.lse_out[row] = lse;
    }
  }
}

template <typename T, int D, int HBLK>
constexpr int fma_stages() {
  return FmaCfg<T, D, HBLK, 1>::kStageBytes >= 65536 ? 2 : 3;
}

template <typename T, int D, int HBLK>
cudaError_t launch_fma_t(const DecodeParams& p, cudaStream_t stream) {
  constexpr int ST = fma_stages<T, D, HBLK>();
  using C = FmaCfg<T, D, HBLK, ST>;
  auto kern = decode_fma_kernel<T, D, HBLK, ST>;
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
  return cudaLaunchKernelEx(&cfg, kern, p);
}

int fma_hblk(int group) { return group >= 4 ? 4 : (group >= 2 ? 2 : 1); }

template <int HBLK>
cudaError_t launch_fma_h(const DecodeParams& p, cudaStream_t stream) {
  if (p.cache_dtype == kDtypeBf16) {
    if (p.head_dim == 128) return launch_fma_t<__nv_bfloat16, 128, HBLK>(p, stream);
    return launch_fma_t<__nv_bfloat16, 64, HBLK>(p, stream);
  }
  if (p.head_dim == 128) return launch_fma_t<float, 128, HBLK>(p, stream);
  return launch_fma_t<float, 64, HBLK>(p, stream);
}

template <typename T, int D, int HBLK>
KernelShape shape_t() {
  constexpr int ST = fma_stages<T, D, HBLK>();
  using C = FmaCfg<T, D, HBLK, ST>;
  return {C::kThreads, C::kSmemBytes, HBLK, 0};
}

template <int HBLK>
KernelShape shape_h(int cache_dtype, int head_dim) {
  if (cache_dtype == kDtypeBf16) return head_dim == 128 ? shape_t<__nv_bfloat16, 128, HBLK>() : shape_t<__nv_bfloat16, 64, HBLK>();
  return head_dim == 128 ? shape_t<float, 128, HBLK>() : shape_t<float, 64, HBLK>();
}

}  // namespace

KernelShape decode_fma_shape(int cache_dtype, int head_dim, int group) {
  switch (fma_hblk(group)) {
    case 4: return shape_h<4>(cache_dtype, head_dim);
    case 2: return shape_h<2>(cache_dtype, head_dim);
    default: return shape_h<1>(cache_dtype, head_dim);
  }
}

cudaError_t launch_decode_fma(const DecodeParams& p, cudaStream_t stream) {
  switch (fma_hblk(p.group)) {
    case 4: return launch_fma_h<4>(p, stream);
    case 2: return launch_fma_h<2>(p, stream);
    default: return launch_fma_h<1>(p, stream);
  }
}

}  // namespace mqa
