// Internal launch interface between the C ABI (abi.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mqa {

// A spin on an mbarrier gives up after a limit (the kernel then sets
// MQA_DEVERR_TIMEOUT and winds down). The limit of the waits for progress is
// a launch parameter (the layout's wait_limit_ns, by default this constant);
// the waits that let a kernel's own copies and MMAs in flight land before it
// exits always use this constant. A healthy wait lasts microseconds.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

// Records `e` as the calling thread's last CUDA error (the text
// mqa_last_cuda_error returns).
void record_cuda_error(cudaError_t e);

constexpr int kTile = 64;          // tokens per pipeline stage of the decode kernels
constexpr int kMaxNewTokens = 32;      // new tokens per sequence the multi-token attention takes
constexpr int kMaxFusedNewTokens = 8;  // new tokens per sequence a fused warp-MMA multi-token step takes
constexpr int kMaxFusedNewTokensTc05 = 16;  // ... a fused tcgen05 multi-token step takes
constexpr int kMaxHalfDim = 64;    // RoPE frequencies held in the append kernel's parameters
constexpr int kDtypeBf16 = 0;
constexpr int kDtypeF32 = 1;
constexpr int kDtypeU8 = 2;  // cache only: uint8 codes + float2 (scale, zero point) per row
constexpr int kDtypeF8 = 3;  // cache only: fp8 e5m2 values

struct AppendParams {
  int batch, h_q, h_kv, head_dim, cache_dtype, paged;
  int n_new;  // new tokens per sequence: token i at position pos[b] + i; q/k/v_new, q_rot [B, n_new, H, d]
  const void* q_new;
  const void* k_new;
  const void* v_new;
  const int32_t* pos;
  void* k_cache;
  void* v_cache;
  long long capacity;
  int page_size, num_pages, max_pages;
  const int32_t* block_table;
  float* q_rot;
  int32_t* err;
  float2* k_sz;  // uint8 cache: (scale, zero point) per row
  float2* v_sz;
  double theta[kMaxHalfDim];  // RoPE inverse frequencies base^(-2i/d)
};

struct DecodeParams {
  int batch, h_q, h_kv, group, head_dim, cache_dtype, paged;
  int n_new;  // query tokens per sequence (the last n_new of its L); rows of a kv head = group * n_new
  const void* k_cache;
  const void* v_cache;
  long long capacity;
  int page_size, num_pages, max_pages;
  const int32_t* block_table;
  const float2* k_sz;  // uint8 cache: (scale, zero point) per row
  const float2* v_sz;
  const float* q_rot;
  const int32_t* seq_lens;
  int max_seq_len;
  float scale_log2;  // score scale times log2(e): scores live in the log2 domain
  int num_splits;    // token-axis splits per (sequence, kv head); 1 = write `out` directly
  int chunk;         // tokens per split, a multiple of kTile
  int head_blocks;   // blocks of query heads a (sequence, kv head) is cut into
  int window;        // 0: all tokens; W > 0: only tokens [max(0, L - W), L)
  int early;         // 1: the preceding launch is the append kernel; stream K/V before waiting for it
  unsigned long long wait_ns;  // limit of the waits for progress (the drains use kWaitLimitNs)
  int merged_halves; // tensor-core path: one TMA box carries both 64-column halves of a row block
  int rope_q;        // 1: rotate q_new (bf16) in the kernel instead of reading q_rot (fused step)
  int fuse_append;   // 1: the kernel also performs the append of the new token (single-launch step)
  const void* q_new;
  const void* k_new;
  const void* v_new;
  float* q_rot_out;  // fused step: where the kernel stores RoPE(q_new)
  const int32_t* pos;
  double theta[kMaxHalfDim];  // RoPE inverse frequencies, used when rope_q
  void* out;
  int out_dtype;
  float* lse_out;
  float* o_part;     // [batch, h_q, num_splits, head_dim] when num_splits > 1
  float* lse_part;   // [batch, h_q, num_splits]
  int32_t* err;
};

// Attention on tcgen05 over blocks of 128 (new token, query head) rows of
// one kv head: prefill, MQA decode, multi-token decode. head_dim 128; bf16
// cache (contiguous or paged) or contiguous fp8 e5m2 cache.
struct Tc05Params {
  int batch, h_q, h_kv, group, n_new;
  int row_blocks;  // ceil(group * n_new / 128)
  int f8;          // attn_tc05: 1 = fp8 e5m2 cache (code tiles), 0 = bf16
  int paged;       // attn_tc05: 1 = paged bf16 cache [num_pages, h_kv, page_size, 128] through block_table
  int page_size, max_pages, num_pages;
  const int32_t* block_table;  // [batch, max_pages] (paged)
  int num_splits;  // token-axis splits; 1 = write `out` directly
  int chunk;       // tokens per split, a multiple of 64
  const void* k_cache;
  const void* v_cache;
  long long capacity;  // tokens a sequence can hold (paged: max_pages * page_size)
  int max_seq_len;
  const int32_t* seq_lens;
  const float* q_rot;  // [B, n_new, H_q, 128] fp32
  float scale_log2;
  int window;
  void* out;  // [B, n_new, H_q, 128]
  int out_dtype;
  float* lse_out;   // [B, n_new, H_q] or null
  float* o_part;    // [B, n_new, H_q, num_splits, 128] when num_splits > 1
  float* lse_part;  // [B, n_new, H_q, num_splits]
  int32_t* err;
  int early;  // 1: the preceding launch is the append kernel; stream K/V before waiting for it
  unsigned long long wait_ns;  // limit of the waits for progress (the drains use kWaitLimitNs)
  // 1 = the block's query rows arrive as TMA boxes through the q_rot tensor
  // map (prefill kernel: one box of 256 rows, group a power of two <= 256;
  // attn_tc05 without a fused append: two boxes of 64 rows, group a power of
  // two <= 64)
  int q_tma;
  // 1: single-launch step (one row block): the kernel rotates q_new itself
  // and the block whose split holds a new token's position appends its k / v
  // rows
  int fuse;
  const void* q_new;  // [B, n_new, H_q, 128] bf16
  const void* k_new;  // [B, n_new, H_kv, 128] bf16
  const void* v_new;
  const int32_t* pos;
  float* q_rot_out;  // RoPE(q_new) [B, n_new, H_q, 128] fp32
  float2* k_sz;      // uint8 cache, fused step: where the new rows' (scale, zero point) go
  float2* v_sz;
  double theta[kMaxHalfDim];
};

struct CombineParams {
  const float* o_part;
  const float* lse_part;
  int rows;  // batch * h_q
  int num_splits, head_dim;
  void* out;
  int out_dtype;
  float* lse_out;
};

// Kernel shapes the host needs for grids, split heuristics and workspace.
struct KernelShape {
  int threads;
  int smem_bytes;
  int heads_per_cta;  // query heads one block serves
  int max_ctas_per_sm;  // > 0: blocks per SM beyond this slow the kernel down (measured)
};

KernelShape append_rope_shape();
cudaError_t launch_append_rope(const AppendParams& p, cudaStream_t stream);

KernelShape decode_fma_shape(int cache_dtype, int head_dim, int group);
cudaError_t launch_decode_fma(const DecodeParams& p, cudaStream_t stream);

// rows = query rows per kv head (group x new tokens)
KernelShape decode_mma_shape(int head_dim, int rows);
cudaError_t launch_decode_mma(const DecodeParams& p, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                              cudaStream_t stream);

// Paged 16-token pages, head_dim 128, G <= 16: kv heads per block of the
// head-slice kernel (4 or 2), or 0 when it does not apply.
int decode_mma_heads_group(const DecodeParams& p);
KernelShape decode_mma_heads_shape(int heads_per_block);
cudaError_t launch_decode_mma_heads(const DecodeParams& p, int heads_per_block, const CUtensorMap& tmap_k,
                                    const CUtensorMap& tmap_v, cudaStream_t stream);

// uint8 cache (codes + per-row scale and zero point), tensor cores; maps =
// {K codes, V codes, K (scale, zero), V (scale, zero)}. The same kernels read
// an fp8 e5m2 cache (p.cache_dtype == kDtypeF8, f8): codes only, maps[2] and
// maps[3] unused.
KernelShape decode_u8_shape(int head_dim, int group, bool f8);
cudaError_t launch_decode_u8(const DecodeParams& p, const CUtensorMap* maps, cudaStream_t stream);
// Paged 16- or 32-token pages, G <= 16: kv heads per block of the head-group
// uint8 kernel (4 or 2), or 0 when it does not apply. Its maps box `hg` heads.
int decode_u8_heads_group(const DecodeParams& p);
cudaError_t launch_decode_u8_heads(const DecodeParams& p, int hg, const CUtensorMap* maps, cudaStream_t stream);

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream);

// tmap_k / tmap_v: the merged-halves bf16 maps with 128-row boxes.
KernelShape tc05_shape();
// uint8 cache, one new token, 16 < G <= 32, contiguous, head_dim 128: keys on
// the MMA rows (attn_tc05_keys.cu; launched for uint8 only, an e5m2 cache
// takes attn_tc05_widen.cu). maps: K codes, V codes (128-row boxes), K and V
// (scale, zero) rows, as make_u8_maps builds them; Tc05Params without the
// fused fields. tc05_keys_applies covers both byte caches (the shape both
// MQA kernels take).
KernelShape tc05_keys_shape();
bool tc05_keys_applies(int group, int n_new, int head_dim, bool paged);
cudaError_t launch_tc05_keys_attention(const Tc05Params& p, int cache_dtype, const CUtensorMap* maps,
                                       cudaStream_t stream);
// the same step over an e5m2 cache with the heads on the MMA rows
// (attn_tc05_widen.cu): converter warps widen the code tiles. maps: the K and
// V code maps of make_u8_maps. With two splits the two blocks of a kv head
// merge in a cluster (no combine: tc05_widen_merges_splits).
KernelShape tc05_widen_shape();
bool tc05_widen_merges_splits(const Tc05Params& p);
cudaError_t launch_tc05_widen_attention(const Tc05Params& p, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                                        cudaStream_t stream);
// tmap_q (used when p.q_tma is set): q_rot as [B n_new tokens][H_q][128]
// fp32, box 128 x group x (64 / group).
cudaError_t launch_tc05_attention(const Tc05Params& p, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                                  const CUtensorMap* tmap_q, cudaStream_t stream);
// Prefill over a bf16 cache (contiguous or paged): blocks of
// tc05_prefill_rows_per_block() rows (two 128-row query tiles); p.row_blocks
// counts those blocks.
int tc05_prefill_rows_per_block();
// tmap_q: q_rot as [B n_new tokens][H_q][128] fp32, box 128 x group x
// (256 / group), used when p.q_tma is set.
cudaError_t launch_tc05_prefill(const Tc05Params& p, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                                const CUtensorMap& tmap_q, cudaStream_t stream);
// true when launch_tc05_attention merges the splits itself (two splits, R <=
// 64 rows in one row block: each pair of split blocks is a two-block cluster
// that writes out and lse_out directly): no combine follows, and o_part /
// lse_part are not written
bool tc05_merges_splits(const Tc05Params& p);
// rows of the TMA box (keys per load) the tcgen05 kernel expects for an fp8
// e5m2 cache
int tc05_f8_box_rows();

}  // namespace mqa
