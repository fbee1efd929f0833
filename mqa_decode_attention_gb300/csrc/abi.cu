// The C ABI of libmqa_decode.so (declared in include/mqa_decode.h):
// host-side argument checks, split choice, TMA descriptor encoding, launches.
// Nothing here allocates device memory or synchronises.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/mqa_decode.h"
#include "launch.h"

namespace {
thread_local char g_cuda_error[256] = "";
}  // namespace

void mqa::record_cuda_error(cudaError_t e) {
  snprintf(g_cuda_error, sizeof(g_cuda_error), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
}

namespace {

using namespace mqa;

mqa_status fail_cuda(cudaError_t e) {
  record_cuda_error(e);
  return MQA_ERR_CUDA;
}

unsigned long long wait_limit(const mqa_kv_layout* L) {
  return L->wait_limit_ns > 0 ? static_cast<unsigned long long>(L->wait_limit_ns) : kWaitLimitNs;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool is_pow2(long long x) { return x > 0 && (x & (x - 1)) == 0; }


mqa_status check_layout(const mqa_kv_layout* L) {
  if (L == nullptr) return MQA_ERR_INVALID_ARG;
  if (L->cache_dtype != MQA_BF16 && L->cache_dtype != MQA_F32 && L->cache_dtype != MQA_U8 &&
      L->cache_dtype != MQA_FP8_E5M2)
    return MQA_ERR_UNSUPPORTED;
  if (L->cache_dtype == MQA_U8) {
    if (L->k_scale_zero == nullptr || L->v_scale_zero == nullptr) return MQA_ERR_INVALID_ARG;
    if (!aligned(L->k_scale_zero, 16) || !aligned(L->v_scale_zero, 16)) return MQA_ERR_INVALID_ARG;
    // the (scale, zero) rows of a kv head are copied by TMA: 16-byte strides
    if (!L->paged && L->capacity % 2 != 0) return MQA_ERR_UNSUPPORTED;
  }
  if (L->batch < 1 || L->h_q < 1 || L->h_kv < 1 || L->h_q % L->h_kv != 0) return MQA_ERR_INVALID_ARG;
  if (L->head_dim != 64 && L->head_dim != 128) return MQA_ERR_UNSUPPORTED;
  if (L->k_cache == nullptr || L->v_cache == nullptr) return MQA_ERR_INVALID_ARG;
  if (!aligned(L->k_cache, 16) || !aligned(L->v_cache, 16)) return MQA_ERR_INVALID_ARG;
  if (L->paged != 0 && L->paged != 1) return MQA_ERR_INVALID_ARG;
  if (L->window < 0) return MQA_ERR_INVALID_ARG;
  if (!L->paged) {
    if (L->capacity < 1 || L->capacity > (1ll << 31) - 1) return MQA_ERR_INVALID_ARG;
  } else {
    if (L->page_size < 16 || L->page_size > 256 || !is_pow2(L->page_size)) return MQA_ERR_UNSUPPORTED;
    if (L->num_pages < 1 || L->max_pages_per_seq < 1 || L->block_table == nullptr) return MQA_ERR_INVALID_ARG;
    if (!aligned(L->block_table, 4)) return MQA_ERR_INVALID_ARG;
    if (static_cast<long long>(L->max_pages_per_seq) * L->page_size > (1ll << 31) - 1) return MQA_ERR_INVALID_ARG;
  }
  return MQA_OK;
}

long long token_limit(const mqa_kv_layout* L) {
  return L->paged ? static_cast<long long>(L->max_pages_per_seq) * L->page_size : L->capacity;
}

int resolve_variant(const mqa_kv_layout* L, int variant) {
  if (variant == MQA_VARIANT_AUTO) return L->cache_dtype == MQA_F32 ? MQA_VARIANT_CUDA_CORE : MQA_VARIANT_TENSOR_CORE;
  return variant;
}

// Which cache dtypes a kernel family reads: tensor cores bf16, uint8 and fp8
// e5m2, CUDA cores bf16 and fp32.
bool variant_supports(int variant, int cache_dtype) {
  if (variant == MQA_VARIANT_TENSOR_CORE)
    return cache_dtype == MQA_BF16 || cache_dtype == MQA_U8 || cache_dtype == MQA_FP8_E5M2;
  return cache_dtype == MQA_BF16 || cache_dtype == MQA_F32;
}

int dtype_code(int cache_dtype) {
  switch (cache_dtype) {
    case MQA_BF16: return kDtypeBf16;
    case MQA_F32: return kDtypeF32;
    case MQA_U8: return kDtypeU8;
    default: return kDtypeF8;
  }
}

// one-byte caches: uint8 codes with (scale, zero) rows, or fp8 e5m2
bool byte_cache(int cache_dtype) { return cache_dtype == MQA_U8 || cache_dtype == MQA_FP8_E5M2; }

struct DeviceInfo {
  int sms = 0;
  int smem_per_sm = 0;
  int threads_per_sm = 0;
};

DeviceInfo device_info(int dev) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  std::lock_guard<std::mutex> lock(mu);
  DeviceInfo& d = cache[dev & 63];
  if (d.sms == 0) {
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    cudaDeviceGetAttribute(&d.threads_per_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev);
    if (d.sms <= 0) d.sms = 1;
  }
  return d;
}

// Query rows per kv head from which the tensor-memory (tcgen05) kernel takes
// the decode attention: 16-row mma.sync tiles run out of latency hiding there
// (MQA's G = 32, several new tokens per sequence).
constexpr int kTc05MinRows = 32;

// Contiguous bf16 caches; paged bf16 pools with several new tokens per
// sequence (a one-token paged step keeps the warp-MMA kernels); contiguous fp8
// e5m2 caches with several new tokens per sequence (the kernel's fp8 form: the
// code tiles enter the MMAs as they are; a one-token e5m2 MQA step takes
// attn_tc05_widen.cu, measured faster there).
bool use_tc05(const mqa_kv_layout* L, int variant, int n_new) {
  if (variant != MQA_VARIANT_TENSOR_CORE || L->head_dim != 128) return false;
  if ((L->h_q / L->h_kv) * n_new < kTc05MinRows) return false;
  if (L->cache_dtype == MQA_BF16) return !L->paged || n_new > 1;
  return L->cache_dtype == MQA_FP8_E5M2 && !L->paged && n_new > 1;
}


// n_new: query tokens per sequence; a kv head then has G x n_new query rows.
KernelShape decode_shape(const mqa_kv_layout* L, int variant, int n_new = 1) {
  const int G = L->h_q / L->h_kv;
  if (use_tc05(L, variant, n_new)) return tc05_shape();
  if (variant == MQA_VARIANT_TENSOR_CORE && byte_cache(L->cache_dtype))
    return !tc05_keys_applies(G, n_new, L->head_dim, L->paged)
               ? decode_u8_shape(L->head_dim, G * n_new, L->cache_dtype == MQA_FP8_E5M2)
               : (L->cache_dtype == MQA_U8 ? tc05_keys_shape() : tc05_widen_shape());
  if (variant == MQA_VARIANT_TENSOR_CORE) return decode_mma_shape(L->head_dim, G * n_new);
  return decode_fma_shape(L->cache_dtype == MQA_BF16 ? kDtypeBf16 : kDtypeF32, L->head_dim, G);
}

int head_blocks(const mqa_kv_layout* L, const KernelShape& ks, int n_new = 1) {
  const int rows = (L->h_q / L->h_kv) * n_new;
  return (rows + ks.heads_per_cta - 1) / ks.heads_per_cta;
}


// Multi-token decode runs on the tensor-core kernels: bf16 (warp-MMA or
// tcgen05), uint8 and e5m2 (the one-byte warp-MMA kernel, or the tcgen05
// kernel's fp8 form for 32 or more rows per kv head over a contiguous e5m2
// cache).
bool multi_supported(const mqa_kv_layout* L, int variant, int n_new) {
  return n_new == 1 || (variant == MQA_VARIANT_TENSOR_CORE && (L->cache_dtype == MQA_BF16 || byte_cache(L->cache_dtype)));
}

// Tokens one (sequence, kv head) may need read: the bound, or with a sliding
// window W the window plus the alignment of its start down to a tile.
int read_span(const mqa_kv_layout* L, int max_len, int n_new = 1) {
  if (L->window > 0 && L->window + kTile + n_new - 1 < max_len) return L->window + kTile + n_new - 1;
  return max_len;
}

// Token-axis split count. Blocks of one (sequence, kv head) are independent,
// so the only reasons to split are (a) too few units to fill the GPU in one
// wave, and (b) device-side lengths that may vary up to max_seq_len, where
// bounded chunks keep long sequences from finishing last. Measured on GB300:
// a single wave of equal blocks streams best (more, smaller blocks add
// partial-output traffic and a second wave), and 4096-token chunks balance a
// paged batch of lengths spread over [128, 16384].
int choose_splits(const mqa_kv_layout* L, int max_len_in, int variant, int n_new = 1) {
  const int max_len = read_span(L, max_len_in);
  int dev = 0;
  cudaGetDevice(&dev);
  const DeviceInfo di = device_info(dev);
  const KernelShape ks = decode_shape(L, variant, n_new);
  const int by_smem = ks.smem_bytes > 0 ? di.smem_per_sm / (ks.smem_bytes + 1024) : 8;
  const int by_threads = di.threads_per_sm / ks.threads;
  int per_sm = std::max(1, std::min(by_smem, by_threads));
  if (ks.max_ctas_per_sm > 0) per_sm = std::min(per_sm, ks.max_ctas_per_sm);
  const long long slots = static_cast<long long>(di.sms) * per_sm;
  const long long units = static_cast<long long>(L->batch) * L->h_kv * head_blocks(L, ks, n_new);
  const int tiles = (max_len + kTile - 1) / kTile;
  int s = 1;
  if (L->paged) {
    const int chunk_tiles = 65;  // 4096 tokens, plus one tile for a window's unaligned start
    s = (tiles + chunk_tiles - 1) / chunk_tiles;
  } else if (units < slots) {
    s = static_cast<int>(slots / units);  // at most one wave
  }
  return std::max(1, std::min(s, tiles));
}

// Effective split count and chunk for a requested count.
void split_plan(int requested, int max_len, int* splits, int* chunk) {
  const int per = (max_len + requested - 1) / requested;
  const int c = ((per + kTile - 1) / kTile) * kTile;
  *chunk = c;
  *splits = (max_len + c - 1) / c;
}

size_t partial_bytes(const mqa_kv_layout* L, int splits, int n_new = 1) {
  if (splits <= 1) return 0;
  const size_t rows = static_cast<size_t>(L->batch) * n_new * L->h_q;
  const size_t o_bytes = ((rows * splits * L->head_dim * 4) + 255) / 256 * 256;
  return o_bytes + rows * splits * 4;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// q_rot [batch n_new tokens][h_q][128] fp32 for the prefill kernel: a box is
// `rows` consecutive rows (group) of one kv head, i.e. rows / group tokens x
// the group's heads x 128 dims, unswizzled (512-byte rows).
bool make_q_map(CUtensorMap* map, const float* q_rot, int batch, int n_new, int h_q, int group, int rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(h_q), static_cast<cuuint64_t>(batch) * n_new};
  const cuuint64_t strides[2] = {128 * 4, static_cast<cuuint64_t>(h_q) * 128 * 4};
  const cuuint32_t box[3] = {128, static_cast<cuuint32_t>(group), static_cast<cuuint32_t>(rows / group)};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(q_rot), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// attn_tc05_kernel reading q_rot (not a fused step) with full 128-row blocks
// (prefill, many new tokens): when the group divides 64, a block's rows come
// as two boxes of 64 rows (p->q_tma set); else, and for fewer rows, the
// kernel reads them with plain loads. False only if the encoder fails.
bool tc05_q_map(Tc05Params* p, CUtensorMap* tq) {
  p->q_tma = 0;
  if (p->fuse || p->q_rot == nullptr || p->group > 64 || (p->group & (p->group - 1)) != 0 ||
      static_cast<long long>(p->group) * p->n_new < 128)
    return true;
  if (!make_q_map(tq, p->q_rot, p->batch, p->n_new, p->h_q, p->group, 64)) return false;
  p->q_tma = 1;
  return true;
}

// TMA descriptors for the tensor-core path: 128-byte swizzled boxes of
// 64 columns, kTile rows (contiguous) or one page (paged, pages shorter than
// a tile). With `merged`, head_dim 128 is described as 64 columns x 2 halves
// where the half dimension has the smaller stride (128 bytes) than the row
// (256 bytes): one box then carries both halves of its rows and lands in
// shared memory as two 64-column spans, so a tile needs half as many copies.
// `heads` > 1 (paged, merged only): a box also spans that many consecutive kv
// heads of one page, which are contiguous in the pool.
bool make_tensor_map(CUtensorMap* map, void* base, const mqa_kv_layout* L, bool merged, int heads = 1,
                     int box_rows = 0) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t D = L->head_dim;
  const cuuint64_t row_bytes = D * 2;
  cuuint64_t dims[5];
  cuuint64_t strides[4];
  cuuint32_t box[5];
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const cuuint32_t rows = box_rows > 0 ? static_cast<cuuint32_t>(box_rows)
                                       : static_cast<cuuint32_t>(L->paged ? (L->page_size < kTile ? L->page_size : kTile)
                                                                          : kTile);
  const cuuint64_t outer_rows = L->paged ? static_cast<cuuint64_t>(L->page_size) : static_cast<cuuint64_t>(L->capacity);
  cuuint32_t rank;
  if (merged) {
    dims[0] = 64;
    dims[1] = outer_rows;
    dims[2] = D / 64;
    strides[0] = row_bytes;
    strides[1] = 128;
    box[0] = 64;
    box[1] = rows;
    box[2] = static_cast<cuuint32_t>(D / 64);
    if (!L->paged) {
      rank = 4;
      dims[3] = static_cast<cuuint64_t>(L->batch) * L->h_kv;
      strides[2] = static_cast<cuuint64_t>(L->capacity) * row_bytes;
      box[3] = 1;
    } else {
      rank = 5;
      dims[3] = static_cast<cuuint64_t>(L->h_kv);
      dims[4] = static_cast<cuuint64_t>(L->num_pages);
      strides[2] = static_cast<cuuint64_t>(L->page_size) * row_bytes;
      strides[3] = static_cast<cuuint64_t>(L->h_kv) * L->page_size * row_bytes;
      box[3] = static_cast<cuuint32_t>(heads);
      box[4] = 1;
    }
  } else {
    dims[0] = D;
    dims[1] = outer_rows;
    strides[0] = row_bytes;
    box[0] = 64;
    box[1] = rows;
    if (!L->paged) {
      rank = 3;
      dims[2] = static_cast<cuuint64_t>(L->batch) * L->h_kv;
      strides[1] = static_cast<cuuint64_t>(L->capacity) * row_bytes;
      box[2] = 1;
    } else {
      rank = 4;
      dims[2] = static_cast<cuuint64_t>(L->h_kv);
      dims[3] = static_cast<cuuint64_t>(L->num_pages);
      strides[1] = static_cast<cuuint64_t>(L->page_size) * row_bytes;
      strides[2] = static_cast<cuuint64_t>(L->h_kv) * L->page_size * row_bytes;
      box[2] = 1;
      box[3] = 1;
    }
  }
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, base, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// TMA descriptors of a uint8 cache: maps[0], maps[1] the K / V codes (boxes
// of head_dim x `rows` rows x `heads` kv heads; 128-byte swizzle for 128-byte
// rows, 64-byte swizzle for 64-byte rows), maps[2], maps[3] their (scale,
// zero) rows as float32 runs of 2 x `rows` values per head. `heads` > 1 only
// for paged pools, where the heads of one page are consecutive.
bool make_u8_maps(CUtensorMap* maps, const mqa_kv_layout* L, int rows_in, int heads) {
  const bool f8 = L->cache_dtype == MQA_FP8_E5M2;  // codes only: the (scale, zero) maps repeat the code maps
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t D = L->head_dim;
  const cuuint32_t rows = static_cast<cuuint32_t>(rows_in);
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapSwizzle swz = D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  void* codes[2] = {L->k_cache, L->v_cache};
  void* sz[2] = {L->k_scale_zero, L->v_scale_zero};
  for (int i = 0; i < 2; ++i) {
    cuuint64_t dims[4], strides[3];
    cuuint32_t box[4];
    cuuint32_t rank;
    dims[0] = D;
    box[0] = static_cast<cuuint32_t>(D);
    box[1] = rows;
    strides[0] = D;
    if (!L->paged) {
      rank = 3;
      dims[1] = static_cast<cuuint64_t>(L->capacity);
      dims[2] = static_cast<cuuint64_t>(L->batch) * L->h_kv;
      strides[1] = static_cast<cuuint64_t>(L->capacity) * D;
      box[2] = 1;
    } else {
      rank = 4;
      dims[1] = static_cast<cuuint64_t>(L->page_size);
      dims[2] = static_cast<cuuint64_t>(L->h_kv);
      dims[3] = static_cast<cuuint64_t>(L->num_pages);
      strides[1] = static_cast<cuuint64_t>(L->page_size) * D;
      strides[2] = static_cast<cuuint64_t>(L->h_kv) * L->page_size * D;
      box[2] = static_cast<cuuint32_t>(heads);
      box[3] = 1;
    }
    if (fn(&maps[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, rank, codes[i], dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  if (f8) {
    maps[2] = maps[0];
    maps[3] = maps[1];
    return true;
  }
  for (int i = 0; i < 2; ++i) {
    cuuint64_t dims[3], strides[2];
    cuuint32_t box[3];
    cuuint32_t rank;
    box[0] = 2 * rows;
    if (!L->paged) {
      rank = 2;
      dims[0] = 2 * static_cast<cuuint64_t>(L->capacity);
      dims[1] = static_cast<cuuint64_t>(L->batch) * L->h_kv;
      strides[0] = 2 * static_cast<cuuint64_t>(L->capacity) * 4;
      box[1] = 1;
    } else {
      rank = 3;
      dims[0] = 2 * static_cast<cuuint64_t>(L->page_size);
      dims[1] = static_cast<cuuint64_t>(L->h_kv);
      dims[2] = static_cast<cuuint64_t>(L->num_pages);
      strides[0] = 2 * static_cast<cuuint64_t>(L->page_size) * 4;
      strides[1] = static_cast<cuuint64_t>(L->h_kv) * strides[0];
      box[1] = static_cast<cuuint32_t>(heads);
      box[2] = 1;
    }
    if (fn(&maps[2 + i], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, rank, sz[i], dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  return true;
}

// Tensor maps of the tcgen05 kernel's K / V tiles: bf16 tiles, or the fp8
// kernel's code tiles (t->f8 set).
// TMA descriptor of a paged bf16 pool for the tcgen05 kernel: dims (64 dims,
// page rows, the two 64-dim halves, kv heads, pages), box 64 x rp x 1 x 1 x 1
// with rp = min(page_size, 64), 128-byte swizzle: one copy per (page run,
// half), landing at the tile's half and row offset.
bool make_tc05_paged_map(CUtensorMap* map, void* base, const mqa_kv_layout* L) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t row_bytes = 256, ps = static_cast<cuuint64_t>(L->page_size);
  const cuuint64_t dims[5] = {64, ps, 2, static_cast<cuuint64_t>(L->h_kv), static_cast<cuuint64_t>(L->num_pages)};
  const cuuint64_t strides[4] = {row_bytes, 128, ps * row_bytes, static_cast<cuuint64_t>(L->h_kv) * ps * row_bytes};
  const cuuint32_t box[5] = {64, static_cast<cuuint32_t>(L->page_size < 64 ? L->page_size : 64), 1, 1, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, base, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool tc05_maps(const mqa_kv_layout* L, Tc05Params* t, CUtensorMap* tk, CUtensorMap* tv) {
  if (L->paged) {
    t->paged = 1;
    t->page_size = L->page_size;
    t->max_pages = L->max_pages_per_seq;
    t->num_pages = L->num_pages;
    t->block_table = L->block_table;
    t->capacity = token_limit(L);
    return make_tc05_paged_map(tk, L->k_cache, L) && make_tc05_paged_map(tv, L->v_cache, L);
  }
  if (L->cache_dtype == MQA_FP8_E5M2) {
    CUtensorMap maps[4];
    if (!make_u8_maps(maps, L, tc05_f8_box_rows(), 1)) return false;
    *tk = maps[0];
    *tv = maps[1];
    t->f8 = 1;
    return true;
  }
  return make_tensor_map(tk, L->k_cache, L, true, 1, 128) && make_tensor_map(tv, L->v_cache, L, true, 1, 128);
}

void fill_theta(double* theta, int head_dim, double base) {
  for (int i = 0; i < head_dim / 2; ++i)
    theta[i] = std::pow(base, -2.0 * static_cast<double>(i) / static_cast<double>(head_dim));
}

mqa_status check_append_args(const mqa_kv_layout* layout, const void* q_new, const void* k_new, const void* v_new,
                             const int32_t* pos, double rope_base, const float* q_rot, const int32_t* err_word) {
  const mqa_status st = check_layout(layout);
  if (st != MQA_OK) return st;
  if (!q_new || !k_new || !v_new || !pos || !q_rot || !err_word) return MQA_ERR_INVALID_ARG;
  if (!aligned(q_new, 16) || !aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(q_rot, 16) ||
      !aligned(pos, 4) || !aligned(err_word, 4))
    return MQA_ERR_INVALID_ARG;
  if (!(rope_base > 0.0) || !std::isfinite(rope_base)) return MQA_ERR_INVALID_ARG;
  return MQA_OK;
}

mqa_status append_impl(const mqa_kv_layout* layout, const void* q_new, const void* k_new, const void* v_new,
                       const int32_t* pos, double rope_base, float* q_rot, int32_t* err_word, mqa_stream_t stream,
                       int n_new = 1) {
  const mqa_status st = check_append_args(layout, q_new, k_new, v_new, pos, rope_base, q_rot, err_word);
  if (st != MQA_OK) return st;
  if (n_new < 1 || static_cast<long long>(layout->batch) * n_new > (1ll << 31) - 1) return MQA_ERR_INVALID_ARG;
  AppendParams p;
  std::memset(&p, 0, sizeof(p));
  p.n_new = n_new;
  p.batch = layout->batch;
  p.h_q = layout->h_q;
  p.h_kv = layout->h_kv;
  p.head_dim = layout->head_dim;
  p.cache_dtype = dtype_code(layout->cache_dtype);
  p.paged = layout->paged;
  p.k_sz = static_cast<float2*>(layout->k_scale_zero);
  p.v_sz = static_cast<float2*>(layout->v_scale_zero);
  p.q_new = q_new;
  p.k_new = k_new;
  p.v_new = v_new;
  p.pos = pos;
  p.k_cache = layout->k_cache;
  p.v_cache = layout->v_cache;
  p.capacity = layout->capacity;
  p.page_size = layout->page_size;
  p.num_pages = layout->num_pages;
  p.max_pages = layout->max_pages_per_seq;
  p.block_table = layout->block_table;
  p.q_rot = q_rot;
  p.err = err_word;
  fill_theta(p.theta, layout->head_dim, rope_base);
  const cudaError_t e = launch_append_rope(p, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e);
  const cudaError_t e2 = cudaGetLastError();
  return e2 == cudaSuccess ? MQA_OK : fail_cuda(e2);
}

// The raw new-token query and its positions, when the attention launch
// directly follows the append launch (fused step): the tensor-core kernels
// then rotate q themselves instead of waiting for q_rot.
struct RopeArgs {
  const void* q_new;
  const int32_t* pos;
  double rope_base;
  int fuse_append;  // 1: no append launch precedes; the decode kernel appends k_new / v_new itself
  const void* k_new;
  const void* v_new;
  float* q_rot;
};

// The tensor-core kernels can take the append over when one block sees all
// query heads of its kv head (warp-MMA kernels: G <= 32; tcgen05: one
// 128-row block). One-byte caches: the warp-MMA kernels (decode_u8_kernel
// with one head block, the paged head-group kernel) and the one-token MQA
// kernels (attn_tc05_keys.cu for uint8, attn_tc05_widen.cu for e5m2).
bool fusable(const mqa_kv_layout* L, int variant) {
  if (variant != MQA_VARIANT_TENSOR_CORE) return false;
  if (byte_cache(L->cache_dtype)) {
    const int G = L->h_q / L->h_kv;
    if (tc05_keys_applies(G, 1, L->head_dim, L->paged)) return true;
    return head_blocks(L, decode_shape(L, variant)) == 1;
  }
  if (L->cache_dtype != MQA_BF16) return false;
  if (use_tc05(L, variant, 1)) return L->h_q / L->h_kv <= 128;  // one row block
  return head_blocks(L, decode_shape(L, variant)) == 1;
}

// Several new tokens per sequence (bf16 cache): the attention kernel takes the
// appends over when one block sees all (token, head) rows of its kv head --
// tcgen05: at most 128 rows; warp-MMA: one head block, and the tokens' cos /
// sin tables fit (at most kMaxFusedNewTokens).
bool fusable_multi(const mqa_kv_layout* L, int variant, int n_new) {
  if (variant != MQA_VARIANT_TENSOR_CORE || L->cache_dtype != MQA_BF16 || n_new < 2) return false;
  // tcgen05: one row block of 128 (token, head) rows, and at most
  // kMaxFusedNewTokensTc05 tokens: the block's append warp turns every new
  // key pair with an fp64-reduced angle, which past that outlasts the stream
  // of keys it hides behind (gqa4k, step vs append + attention: n = 8 90.8 vs
  // 100.0 us, n = 16 100.4 vs 106.4, n = 32 148 vs 113.6)
  if (use_tc05(L, variant, n_new)) return (L->h_q / L->h_kv) * n_new <= 128 && n_new <= kMaxFusedNewTokensTc05;
  if (n_new > kMaxFusedNewTokens) return false;
  return head_blocks(L, decode_shape(L, variant, n_new), n_new) == 1;
}

mqa_status attention_impl(const mqa_kv_layout* layout, const float* q_rot, const int32_t* seq_lens, int32_t max_seq_len,
                          float scale, int32_t num_splits, void* out, int32_t out_dtype, float* lse_out,
                          void* workspace, size_t workspace_bytes, int32_t variant, int32_t* err_word,
                          mqa_stream_t stream, int early, const RopeArgs* rope, int n_new = 1, int prefill = 0) {
  const mqa_status st = check_layout(layout);
  if (st != MQA_OK) return st;
  // (prefill over a one-byte cache takes this path with the whole prompt)
  if (n_new < 1 || (!prefill && n_new > kMaxNewTokens)) return MQA_ERR_INVALID_ARG;
  if (static_cast<long long>(layout->batch) * n_new * layout->h_q > (1ll << 31) - 1) return MQA_ERR_INVALID_ARG;
  if (!q_rot || !seq_lens || !out || !err_word) return MQA_ERR_INVALID_ARG;
  if (!aligned(q_rot, 16) || !aligned(seq_lens, 4) || !aligned(out, 16) || !aligned(err_word, 4) ||
      (lse_out && !aligned(lse_out, 4)))
    return MQA_ERR_INVALID_ARG;
  if (max_seq_len < n_new || max_seq_len > token_limit(layout)) return MQA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || num_splits < 0) return MQA_ERR_INVALID_ARG;
  if (out_dtype != MQA_BF16 && out_dtype != MQA_F32) return MQA_ERR_UNSUPPORTED;
  if (variant < MQA_VARIANT_AUTO || variant > MQA_VARIANT_TENSOR_CORE) return MQA_ERR_INVALID_ARG;
  const int v = resolve_variant(layout, variant);
  if (!variant_supports(v, layout->cache_dtype) || !multi_supported(layout, v, n_new)) return MQA_ERR_UNSUPPORTED;

  const int req = num_splits == 0 ? choose_splits(layout, max_seq_len, v, n_new) : num_splits;
  int splits, chunk;
  split_plan(req, read_span(layout, max_seq_len, n_new), &splits, &chunk);
  const size_t need = partial_bytes(layout, splits, n_new);
  if (need > 0) {
    if (workspace == nullptr || workspace_bytes < need) return MQA_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return MQA_ERR_INVALID_ARG;
  }

  const KernelShape ks = decode_shape(layout, v, n_new);
  bool merged = false;  // the attention launch merged its splits itself: no combine
  DecodeParams p;
  std::memset(&p, 0, sizeof(p));
  p.n_new = n_new;
  p.batch = layout->batch;
  p.h_q = layout->h_q;
  p.h_kv = layout->h_kv;
  p.group = layout->h_q / layout->h_kv;
  p.head_dim = layout->head_dim;
  p.cache_dtype = dtype_code(layout->cache_dtype);
  p.paged = layout->paged;
  p.k_cache = layout->k_cache;
  p.k_sz = static_cast<const float2*>(layout->k_scale_zero);
  p.v_sz = static_cast<const float2*>(layout->v_scale_zero);
  p.v_cache = layout->v_cache;
  p.capacity = layout->capacity;
  p.page_size = layout->page_size;
  p.num_pages = layout->num_pages;
  p.max_pages = layout->max_pages_per_seq;
  p.block_table = layout->block_table;
  p.q_rot = q_rot;
  p.seq_lens = seq_lens;
  p.max_seq_len = max_seq_len;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.num_splits = splits;
  p.chunk = chunk;
  p.head_blocks = head_blocks(layout, ks, n_new);
  p.window = layout->window;
  p.early = early;
  p.wait_ns = wait_limit(layout);
  // (one-byte caches and several new tokens: only in the fused step;
  // otherwise q_rot comes from the append launch)
  if (rope != nullptr && v == MQA_VARIANT_TENSOR_CORE &&
      ((n_new == 1 && (layout->cache_dtype == MQA_BF16 || (byte_cache(layout->cache_dtype) && rope->fuse_append))) ||
       (n_new > 1 && rope->fuse_append))) {
    p.rope_q = 1;
    p.q_new = rope->q_new;
    p.pos = rope->pos;
    fill_theta(p.theta, layout->head_dim, rope->rope_base);
    if (rope->fuse_append) {
      p.fuse_append = 1;
      p.early = 0;  // nothing of this step precedes the launch
      p.k_new = rope->k_new;
      p.v_new = rope->v_new;
      p.q_rot_out = rope->q_rot;
    }
  }
  p.out = out;
  p.out_dtype = out_dtype == MQA_BF16 ? kDtypeBf16 : kDtypeF32;
  p.lse_out = lse_out;
  p.err = err_word;
  if (splits > 1) {
    const size_t rows = static_cast<size_t>(layout->batch) * n_new * layout->h_q;
    const size_t o_bytes = ((rows * splits * layout->head_dim * 4) + 255) / 256 * 256;
    p.o_part = static_cast<float*>(workspace);
    p.lse_part = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) + o_bytes);
  }
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (use_tc05(layout, v, n_new)) {
    Tc05Params t;
    std::memset(&t, 0, sizeof(t));
    t.batch = layout->batch;
    t.h_q = layout->h_q;
    t.h_kv = layout->h_kv;
    t.group = p.group;
    t.n_new = n_new;
    t.row_blocks = (p.group * n_new + 127) / 128;
    t.num_splits = splits;
    t.chunk = chunk;
    t.k_cache = layout->k_cache;
    t.v_cache = layout->v_cache;
    t.capacity = layout->capacity;
    t.max_seq_len = max_seq_len;
    t.seq_lens = seq_lens;
    t.q_rot = q_rot;
    t.scale_log2 = p.scale_log2;
    t.window = layout->window;
    t.out = out;
    t.out_dtype = p.out_dtype;
    t.lse_out = lse_out;
    t.o_part = p.o_part;
    t.lse_part = p.lse_part;
    t.err = err_word;
    t.early = early;
    t.wait_ns = p.wait_ns;
    if (rope != nullptr && rope->fuse_append) {  // (fusable: one row block)
      t.fuse = 1;
      t.early = 0;  // nothing of this step precedes the launch
      t.q_new = rope->q_new;
      t.k_new = rope->k_new;
      t.v_new = rope->v_new;
      t.pos = rope->pos;
      t.q_rot_out = rope->q_rot;
      fill_theta(t.theta, layout->head_dim, rope->rope_base);
    }
    CUtensorMap tk, tv, tq;
    if (!tc05_maps(layout, &t, &tk, &tv) || !tc05_q_map(&t, &tq)) {
      snprintf(g_cuda_error, sizeof(g_cuda_error), "cuTensorMapEncodeTiled failed or is unavailable");
      return MQA_ERR_CUDA;
    }
    e = launch_tc05_attention(t, tk, tv, &tq, s);
    if (e != cudaSuccess) return fail_cuda(e);
    merged = tc05_merges_splits(t);
    goto combine;
  }
  if (v == MQA_VARIANT_TENSOR_CORE && byte_cache(layout->cache_dtype) &&
      tc05_keys_applies(p.group, n_new, layout->head_dim, layout->paged)) {
    // one-byte MQA step on tcgen05. e5m2: the heads on the MMA rows, converter
    // warps widening the code tiles (attn_tc05_widen.cu); uint8: the keys on
    // the MMA rows (attn_tc05_keys.cu), measured faster for uint8
    CUtensorMap maps[4];
    if (!make_u8_maps(maps, layout, 128, 1)) {
      snprintf(g_cuda_error, sizeof(g_cuda_error), "cuTensorMapEncodeTiled failed or is unavailable");
      return MQA_ERR_CUDA;
    }
    Tc05Params t;
    std::memset(&t, 0, sizeof(t));
    t.batch = layout->batch;
    t.h_q = layout->h_q;
    t.h_kv = layout->h_kv;
    t.group = p.group;
    t.n_new = 1;
    t.row_blocks = 1;
    t.num_splits = splits;
    t.chunk = chunk;
    t.k_cache = layout->k_cache;
    t.v_cache = layout->v_cache;
    t.capacity = layout->capacity;
    t.max_seq_len = max_seq_len;
    t.seq_lens = seq_lens;
    t.q_rot = q_rot;
    t.scale_log2 = p.scale_log2;
    t.window = layout->window;
    t.out = out;
    t.out_dtype = p.out_dtype;
    t.lse_out = lse_out;
    t.o_part = p.o_part;
    t.lse_part = p.lse_part;
    t.err = err_word;
    t.early = early;
    t.wait_ns = p.wait_ns;
    if (rope != nullptr && rope->fuse_append) {
      // one launch: the kernel rotates q_new and encodes the new row itself
      t.fuse = 1;
      t.early = 0;
      t.q_new = rope->q_new;
      t.k_new = rope->k_new;
      t.v_new = rope->v_new;
      t.pos = rope->pos;
      t.q_rot_out = rope->q_rot;
      t.k_sz = static_cast<float2*>(layout->k_scale_zero);
      t.v_sz = static_cast<float2*>(layout->v_scale_zero);
      fill_theta(t.theta, layout->head_dim, rope->rope_base);
    }
    if (layout->cache_dtype == MQA_U8) {
      e = launch_tc05_keys_attention(t, kDtypeU8, maps, s);
    } else {
      e = launch_tc05_widen_attention(t, maps[0], maps[1], s);
      if (e != cudaSuccess) return fail_cuda(e);
      merged = tc05_widen_merges_splits(t);
      goto combine;
    }
  } else if (v == MQA_VARIANT_TENSOR_CORE && byte_cache(layout->cache_dtype)) {
    CUtensorMap maps[4];
    // Paged 16- / 32-token pages: blocks over groups of kv heads, one box per
    // page and head group (long contiguous runs of the pool).
    const int hg = decode_u8_heads_group(p);
    const int rows = hg > 0 ? layout->page_size : (layout->paged && layout->page_size < kTile ? layout->page_size : kTile);
    if (!make_u8_maps(maps, layout, rows, hg > 0 ? hg : 1)) {
      snprintf(g_cuda_error, sizeof(g_cuda_error), "cuTensorMapEncodeTiled failed or is unavailable");
      return MQA_ERR_CUDA;
    }
    e = hg > 0 ? launch_decode_u8_heads(p, hg, maps, s) : launch_decode_u8(p, maps, s);
  } else if (v == MQA_VARIANT_TENSOR_CORE) {
    CUtensorMap tk, tv;
    // Paged 16-token pages: blocks over groups of kv heads, one box per page
    // and head group (long contiguous runs of the pool).
    const int hg = decode_mma_heads_group(p);
    if (hg > 0 && make_tensor_map(&tk, layout->k_cache, layout, true, hg) &&
        make_tensor_map(&tv, layout->v_cache, layout, true, hg)) {
      p.merged_halves = 1;
      p.head_blocks = 1;
      e = launch_decode_mma_heads(p, hg, tk, tv, s);
      if (e != cudaSuccess) return fail_cuda(e);
      goto combine;
    }
    p.merged_halves = layout->head_dim == 128 && make_tensor_map(&tk, layout->k_cache, layout, true) &&
                      make_tensor_map(&tv, layout->v_cache, layout, true);
    if (!p.merged_halves &&
        (!make_tensor_map(&tk, layout->k_cache, layout, false) || !make_tensor_map(&tv, layout->v_cache, layout, false))) {
      snprintf(g_cuda_error, sizeof(g_cuda_error), "cuTensorMapEncodeTiled failed or is unavailable");
      return MQA_ERR_CUDA;
    }
    e = launch_decode_mma(p, tk, tv, s);
  } else {
    e = launch_decode_fma(p, s);
  }
  if (e != cudaSuccess) return fail_cuda(e);
combine:
  if (splits > 1 && !merged) {
    CombineParams c;
    c.o_part = p.o_part;
    c.lse_part = p.lse_part;
    c.rows = layout->batch * n_new * layout->h_q;
    c.num_splits = splits;
    c.head_dim = layout->head_dim;
    c.out = out;
    c.out_dtype = p.out_dtype;
    c.lse_out = lse_out;
    e = launch_combine(c, s);
    if (e != cudaSuccess) return fail_cuda(e);
  }
  const cudaError_t e2 = cudaGetLastError();
  return e2 == cudaSuccess ? MQA_OK : fail_cuda(e2);
}

// Causal attention of the last n_new tokens of every sequence on tcgen05
// (prefill): contiguous bf16 cache, head_dim 128.
// Prefill over a uint8 cache, or a paged e5m2 pool: the one-byte warp-MMA
// kernel's multi-token form over the whole prompt (rows = (token, head) pairs,
// 32 per block; every block streams the keys up to its last row).
bool prefill_on_byte_kernel(const mqa_kv_layout* L) {
  return L->cache_dtype == MQA_U8 || (L->cache_dtype == MQA_FP8_E5M2 && L->paged);
}

// The cache types and shapes gqa_prefill_attention takes.
bool prefill_supported(const mqa_kv_layout* L) {
  if (prefill_on_byte_kernel(L)) return L->head_dim == 64 || L->head_dim == 128;
  return (L->cache_dtype == MQA_BF16 || L->cache_dtype == MQA_FP8_E5M2) && L->head_dim == 128;
}

mqa_status prefill_impl(const mqa_kv_layout* layout, int n_new, const float* q_rot, const int32_t* seq_lens,
                        int32_t max_seq_len, float scale, void* out, int32_t out_dtype, float* lse_out,
                        int32_t* err_word, mqa_stream_t stream, int early) {
  const mqa_status st = check_layout(layout);
  if (st != MQA_OK) return st;
  if (!prefill_supported(layout)) return MQA_ERR_UNSUPPORTED;
  if (prefill_on_byte_kernel(layout))
    return attention_impl(layout, q_rot, seq_lens, max_seq_len, scale, /*num_splits=*/1, out, out_dtype, lse_out,
                          nullptr, 0, MQA_VARIANT_TENSOR_CORE, err_word, stream, early, nullptr, n_new,
                          /*prefill=*/1);
  if (n_new < 1 || static_cast<long long>(layout->batch) * n_new > (1ll << 31) - 1) return MQA_ERR_INVALID_ARG;
  if (!q_rot || !seq_lens || !out || !err_word) return MQA_ERR_INVALID_ARG;
  if (!aligned(q_rot, 16) || !aligned(seq_lens, 4) || !aligned(out, 16) || !aligned(err_word, 4) ||
      (lse_out && !aligned(lse_out, 4)))
    return MQA_ERR_INVALID_ARG;
  if (max_seq_len < n_new || max_seq_len > token_limit(layout)) return MQA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return MQA_ERR_INVALID_ARG;
  if (out_dtype != MQA_BF16 && out_dtype != MQA_F32) return MQA_ERR_UNSUPPORTED;
  const long long blocks = static_cast<long long>(layout->batch) * layout->h_kv *
                           ((static_cast<long long>(layout->h_q / layout->h_kv) * n_new + 127) / 128);
  if (blocks > (1ll << 31) - 1) return MQA_ERR_INVALID_ARG;
  Tc05Params p;
  std::memset(&p, 0, sizeof(p));
  p.batch = layout->batch;
  p.h_q = layout->h_q;
  p.h_kv = layout->h_kv;
  p.group = layout->h_q / layout->h_kv;
  p.n_new = n_new;
  p.row_blocks = static_cast<int>((static_cast<long long>(p.group) * n_new + 127) / 128);
  p.num_splits = 1;
  p.chunk = ((max_seq_len + 63) / 64) * 64;
  p.k_cache = layout->k_cache;
  p.v_cache = layout->v_cache;
  p.capacity = layout->capacity;
  p.max_seq_len = max_seq_len;
  p.seq_lens = seq_lens;
  p.q_rot = q_rot;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.window = layout->window;
  p.out = out;
  p.out_dtype = out_dtype == MQA_BF16 ? kDtypeBf16 : kDtypeF32;
  p.lse_out = lse_out;
  p.err = err_word;
  p.early = early;
  p.wait_ns = wait_limit(layout);
  CUtensorMap tk, tv;
  if (!tc05_maps(layout, &p, &tk, &tv)) {
    snprintf(g_cuda_error, sizeof(g_cuda_error), "cuTensorMapEncodeTiled failed or is unavailable");
    return MQA_ERR_CUDA;
  }
  cudaError_t e;
  {
    // two 128-row query tiles per block sharing every K / V tile (bf16, or
    // e5m2 code tiles in the kernel's fp8 form)
    const int rpb = tc05_prefill_rows_per_block();
    p.row_blocks = static_cast<int>((static_cast<long long>(p.group) * n_new + rpb - 1) / rpb);
    // a block's rows are whole tokens when the group divides them: then they
    // come as one TMA box ([tokens][heads][128] fp32)
    CUtensorMap tq = tk;
    if (p.group <= 256 && (p.group & (p.group - 1)) == 0) {
      if (!make_q_map(&tq, q_rot, layout->batch, n_new, layout->h_q, p.group, rpb)) {
        snprintf(g_cuda_error, sizeof(g_cuda_error), "cuTensorMapEncodeTiled failed or is unavailable");
        return MQA_ERR_CUDA;
      }
      p.q_tma = 1;
    }
    e = launch_tc05_prefill(p, tk, tv, tq, reinterpret_cast<cudaStream_t>(stream));
  }
  if (e != cudaSuccess) return fail_cuda(e);
  const cudaError_t e2 = cudaGetLastError();
  return e2 == cudaSuccess ? MQA_OK : fail_cuda(e2);
}

}  // namespace

extern "C" {

mqa_status gqa_prefill_attention(const mqa_kv_layout* layout, int32_t n_new, const float* q_rot,
                                 const int32_t* seq_lens, int32_t max_seq_len, float scale, void* out,
                                 int32_t out_dtype, float* lse_out, int32_t* err_word, mqa_stream_t stream) {
  return prefill_impl(layout, n_new, q_rot, seq_lens, max_seq_len, scale, out, out_dtype, lse_out, err_word, stream,
                      /*early=*/0);
}

mqa_status mqa_prefill_step(const mqa_kv_layout* layout, int32_t n_new, const void* q_new, const void* k_new,
                            const void* v_new, const int32_t* pos, const int32_t* seq_lens, int32_t max_seq_len,
                            double rope_base, float scale, float* q_rot, void* out, int32_t out_dtype,
                            float* lse_out, int32_t* err_word, mqa_stream_t stream) {
  // the attention's own checks first, so nothing is launched for a call that fails
  const mqa_status st = check_layout(layout);
  if (st != MQA_OK) return st;
  if (!prefill_supported(layout)) return MQA_ERR_UNSUPPORTED;
  if (!seq_lens || !out || max_seq_len < n_new || max_seq_len > token_limit(layout)) return MQA_ERR_INVALID_ARG;
  if (out_dtype != MQA_BF16 && out_dtype != MQA_F32) return MQA_ERR_UNSUPPORTED;
  const mqa_status a = append_impl(layout, q_new, k_new, v_new, pos, rope_base, q_rot, err_word, stream, n_new);
  if (a != MQA_OK) return a;
  return prefill_impl(layout, n_new, q_rot, seq_lens, max_seq_len, scale, out, out_dtype, lse_out, err_word, stream,
                      /*early=*/1);
}

const char* mqa_status_string(mqa_status s) {
  switch (s) {
    case MQA_OK: return "ok";
    case MQA_ERR_INVALID_ARG: return "invalid argument";
    case MQA_ERR_UNSUPPORTED: return "unsupported configuration";
    case MQA_ERR_CUDA: return "CUDA error";
    case MQA_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

const char* mqa_last_cuda_error(void) { return g_cuda_error; }

mqa_status kv_append_rope(const mqa_kv_layout* layout, const void* q_new, const void* k_new, const void* v_new,
                          const int32_t* pos, double rope_base, float* q_rot, int32_t* err_word,
                          mqa_stream_t stream) {
  return append_impl(layout, q_new, k_new, v_new, pos, rope_base, q_rot, err_word, stream);
}

int32_t mqa_choose_splits_multi(const mqa_kv_layout* layout, int32_t n_new, int32_t max_seq_len, int32_t variant) {
  if (check_layout(layout) != MQA_OK || max_seq_len < 1 || max_seq_len > token_limit(layout)) return -1;
  if (variant < MQA_VARIANT_AUTO || variant > MQA_VARIANT_TENSOR_CORE) return -1;
  if (n_new < 1 || n_new > kMaxNewTokens || max_seq_len < n_new) return -1;
  return choose_splits(layout, max_seq_len, resolve_variant(layout, variant), n_new);
}

int32_t mqa_choose_splits(const mqa_kv_layout* layout, int32_t max_seq_len, int32_t variant) {
  return mqa_choose_splits_multi(layout, 1, max_seq_len, variant);
}

size_t mqa_workspace_size_multi(const mqa_kv_layout* layout, int32_t n_new, int32_t max_seq_len, int32_t num_splits,
                                int32_t variant) {
  if (check_layout(layout) != MQA_OK || max_seq_len < 1 || max_seq_len > token_limit(layout) || num_splits < 0)
    return 0;
  if (variant < MQA_VARIANT_AUTO || variant > MQA_VARIANT_TENSOR_CORE) return 0;
  if (n_new < 1 || n_new > kMaxNewTokens || max_seq_len < n_new) return 0;
  const int v = resolve_variant(layout, variant);
  const int req = num_splits == 0 ? choose_splits(layout, max_seq_len, v, n_new) : num_splits;
  int splits, chunk;
  split_plan(req, read_span(layout, max_seq_len, n_new), &splits, &chunk);
  return partial_bytes(layout, splits, n_new);
}

size_t mqa_workspace_size(const mqa_kv_layout* layout, int32_t max_seq_len, int32_t num_splits, int32_t variant) {
  return mqa_workspace_size_multi(layout, 1, max_seq_len, num_splits, variant);
}

int32_t mqa_step_launches(const mqa_kv_layout* layout, int32_t n_new, int32_t max_seq_len, int32_t num_splits,
                          int32_t variant, int32_t* fused_append) {
  if (check_layout(layout) != MQA_OK || max_seq_len < 1 || max_seq_len > token_limit(layout) || num_splits < 0)
    return -1;
  if (variant < MQA_VARIANT_AUTO || variant > MQA_VARIANT_TENSOR_CORE) return -1;
  if (n_new < 1 || n_new > kMaxNewTokens || max_seq_len < n_new) return -1;
  const int v = resolve_variant(layout, variant);
  if (!variant_supports(v, layout->cache_dtype) || !multi_supported(layout, v, n_new)) return -1;
  const int req = num_splits == 0 ? choose_splits(layout, max_seq_len, v, n_new) : num_splits;
  int splits, chunk;
  split_plan(req, read_span(layout, max_seq_len, n_new), &splits, &chunk);
  // the decisions step_impl and attention_impl take
  const bool fused = (n_new == 1 && fusable(layout, v)) || fusable_multi(layout, v, n_new);
  bool merged = false;
  if (splits > 1) {
    Tc05Params t;
    std::memset(&t, 0, sizeof(t));
    t.group = layout->h_q / layout->h_kv;
    t.n_new = n_new;
    t.num_splits = splits;
    t.row_blocks = (t.group * n_new + 127) / 128;
    if (use_tc05(layout, v, n_new))
      merged = tc05_merges_splits(t);
    else if (v == MQA_VARIANT_TENSOR_CORE && layout->cache_dtype == MQA_FP8_E5M2 &&
             tc05_keys_applies(t.group, n_new, layout->head_dim, layout->paged))
      merged = tc05_widen_merges_splits(t);
  }
  if (fused_append) *fused_append = fused ? 1 : 0;
  return (fused ? 1 : 2) + (splits > 1 && !merged ? 1 : 0);
}

mqa_status splitkv_combine(const float* o_part, const float* lse_part, int32_t batch, int32_t h_q,
                           int32_t num_splits, int32_t head_dim, void* out, int32_t out_dtype, float* lse_out,
                           mqa_stream_t stream) {
  if (!o_part || !lse_part || !out) return MQA_ERR_INVALID_ARG;
  if (batch < 1 || h_q < 1 || num_splits < 1 || head_dim < 1) return MQA_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return MQA_ERR_UNSUPPORTED;
  if (out_dtype != MQA_BF16 && out_dtype != MQA_F32) return MQA_ERR_UNSUPPORTED;
  if (!aligned(o_part, 4) || !aligned(lse_part, 4) || !aligned(out, 4) || (lse_out && !aligned(lse_out, 4)))
    return MQA_ERR_INVALID_ARG;
  CombineParams c;
  c.o_part = o_part;
  c.lse_part = lse_part;
  c.rows = batch * h_q;
  c.num_splits = num_splits;
  c.head_dim = head_dim;
  c.out = out;
  c.out_dtype = out_dtype == MQA_BF16 ? kDtypeBf16 : kDtypeF32;
  c.lse_out = lse_out;
  const cudaError_t e = launch_combine(c, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e);
  const cudaError_t e2 = cudaGetLastError();
  return e2 == cudaSuccess ? MQA_OK : fail_cuda(e2);
}

mqa_status gqa_decode_attention(const mqa_kv_layout* layout, const float* q_rot, const int32_t* seq_lens,
                                int32_t max_seq_len, float scale, int32_t num_splits, void* out,
                                int32_t out_dtype, float* lse_out, void* workspace, size_t workspace_bytes,
                                int32_t variant, int32_t* err_word, mqa_stream_t stream) {
  return attention_impl(layout, q_rot, seq_lens, max_seq_len, scale, num_splits, out, out_dtype, lse_out, workspace,
                        workspace_bytes, variant, err_word, stream, /*early=*/0, /*rope=*/nullptr);
}

mqa_status kv_append_rope_multi(const mqa_kv_layout* layout, int32_t n_new, const void* q_new, const void* k_new,
                                const void* v_new, const int32_t* pos, double rope_base, float* q_rot,
                                int32_t* err_word, mqa_stream_t stream) {
  return append_impl(layout, q_new, k_new, v_new, pos, rope_base, q_rot, err_word, stream, n_new);
}

mqa_status gqa_decode_attention_multi(const mqa_kv_layout* layout, int32_t n_new, const float* q_rot,
                                      const int32_t* seq_lens, int32_t max_seq_len, float scale, int32_t num_splits,
                                      void* out, int32_t out_dtype, float* lse_out, void* workspace,
                                      size_t workspace_bytes, int32_t variant, int32_t* err_word,
                                      mqa_stream_t stream) {
  return attention_impl(layout, q_rot, seq_lens, max_seq_len, scale, num_splits, out, out_dtype, lse_out, workspace,
                        workspace_bytes, variant, err_word, stream, /*early=*/0, /*rope=*/nullptr, n_new);
}

}  // extern "C"

namespace {

mqa_status step_impl(const mqa_kv_layout* layout, int n_new, const void* q_new, const void* k_new, const void* v_new,
                     const int32_t* pos, const int32_t* seq_lens, int32_t max_seq_len, double rope_base, float scale,
                     int32_t num_splits, float* q_rot, void* out, int32_t out_dtype, float* lse_out, void* workspace,
                     size_t workspace_bytes, int32_t variant, int32_t* err_word, mqa_stream_t stream) {
  // Check the attention's arguments too before anything is launched.
  const mqa_status st = check_layout(layout);
  if (st != MQA_OK) return st;
  if (n_new < 1 || n_new > kMaxNewTokens) return MQA_ERR_INVALID_ARG;
  if (!seq_lens || !out || max_seq_len < n_new || max_seq_len > token_limit(layout)) return MQA_ERR_INVALID_ARG;
  if (variant < MQA_VARIANT_AUTO || variant > MQA_VARIANT_TENSOR_CORE || num_splits < 0)
    return MQA_ERR_INVALID_ARG;
  if (out_dtype != MQA_BF16 && out_dtype != MQA_F32) return MQA_ERR_UNSUPPORTED;
  const int v = resolve_variant(layout, variant);
  if (!variant_supports(v, layout->cache_dtype) || !multi_supported(layout, v, n_new)) return MQA_ERR_UNSUPPORTED;
  {
    const int req = num_splits == 0 ? choose_splits(layout, max_seq_len, v, n_new) : num_splits;
    int splits, chunk;
    split_plan(req, read_span(layout, max_seq_len, n_new), &splits, &chunk);
    const size_t need = partial_bytes(layout, splits, n_new);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return MQA_ERR_WORKSPACE;
  }
  const mqa_status ca = check_append_args(layout, q_new, k_new, v_new, pos, rope_base, q_rot, err_word);
  if (ca != MQA_OK) return ca;
  if ((n_new == 1 && fusable(layout, v)) || fusable_multi(layout, v, n_new)) {
    // one launch: the attention kernel appends the new token(s) itself
    const RopeArgs rope{q_new, pos, rope_base, 1, k_new, v_new, q_rot};
    return attention_impl(layout, q_rot, seq_lens, max_seq_len, scale, num_splits, out, out_dtype, lse_out,
                          workspace, workspace_bytes, variant, err_word, stream, /*early=*/0, &rope, n_new);
  }
  const mqa_status a = append_impl(layout, q_new, k_new, v_new, pos, rope_base, q_rot, err_word, stream, n_new);
  if (a != MQA_OK) return a;
  const RopeArgs rope{q_new, pos, rope_base, 0, nullptr, nullptr, nullptr};
  return attention_impl(layout, q_rot, seq_lens, max_seq_len, scale, num_splits, out, out_dtype, lse_out, workspace,
                        workspace_bytes, variant, err_word, stream, /*early=*/1, &rope, n_new);
}

}  // namespace

extern "C" {

mqa_status mqa_decode_step(const mqa_kv_layout* layout, const void* q_new, const void* k_new, const void* v_new,
                           const int32_t* pos, const int32_t* seq_lens, int32_t max_seq_len, double rope_base,
                           float scale, int32_t num_splits, float* q_rot, void* out, int32_t out_dtype,
                           float* lse_out, void* workspace, size_t workspace_bytes, int32_t variant,
                           int32_t* err_word, mqa_stream_t stream) {
  return step_impl(layout, 1, q_new, k_new, v_new, pos, seq_lens, max_seq_len, rope_base, scale, num_splits, q_rot,
                   out, out_dtype, lse_out, workspace, workspace_bytes, variant, err_word, stream);
}

mqa_status mqa_decode_step_multi(const mqa_kv_layout* layout, int32_t n_new, const void* q_new, const void* k_new,
                                 const void* v_new, const int32_t* pos, const int32_t* seq_lens, int32_t max_seq_len,
                                 double rope_base, float scale, int32_t num_splits, float* q_rot, void* out,
                                 int32_t out_dtype, float* lse_out, void* workspace, size_t workspace_bytes,
                                 int32_t variant, int32_t* err_word, mqa_stream_t stream) {
  return step_impl(layout, n_new, q_new, k_new, v_new, pos, seq_lens, max_seq_len, rope_base, scale, num_splits,
                   q_rot, out, out_dtype, lse_out, workspace, workspace_bytes, variant, err_word, stream);
}

}  // extern "C"
