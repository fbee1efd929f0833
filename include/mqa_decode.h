/*
 * mqa_decode.h -- C ABI of the GB300 decode-step attention library
 * (libmqa_decode.so, sm_103a).
 *
 * One autoregressive decode step of grouped-query attention over a KV cache:
 *
 *   1. kv_append_rope        RoPE on the new token's q and k; append the
 *                            rotated k and the v into the cache.
 *   2. gqa_decode_attention  O_h = softmax(Q_h K_g(h)^T / sqrt(d)) V_g(h),
 *                            g(h) = floor(h / G), G = H_q / H_kv, over every
 *                            cached token of the sequence.
 *   3. splitkv_combine       log-sum-exp merge of split-KV partial results
 *                            (called by 2 itself when it splits).
 *
 * Sources: "Grouped-query attention: berbagi KV head di antara grup query"
 * (nalar.dev), section "Jumlah head menentukan batas grup" (G, g(h), A_h,
 * O_h) and "GQA berada di antara MHA dan MQA" (H_kv = H_q is MHA, H_kv = 1
 * is MQA); "KV Cache" explainer (lensaml.com), Langkah 3 (cache pair
 * [batch, kv_heads, tokens, head_dim], one slice written per decode step,
 * keys rotated by position once and stored rotated); "KV Cache 최적화 심층
 * 분석" (youngju.dev), class PagedKVCache (block = pos / block_size,
 * offset = pos % block_size); "Arsitektur Inferensi LLM" (tveniu.com),
 * section 4 PagedAttention (16-token blocks behind a page table) and section
 * 5 FlashAttention (online softmax, no score matrix in HBM).
 *
 * Conventions for every call
 *  - All pointers to tensors are DEVICE pointers unless stated otherwise;
 *    the layout struct itself is a HOST pointer, read during the call only.
 *    The new-token inputs (q_new, k_new, v_new, pos, seq_lens) and the
 *    output `out` may instead be pinned host memory that the device reaches
 *    through unified addressing (cudaHostAlloc / pinned tensors): the kernels
 *    then read and write them across the CPU-GPU link, with no copy launch.
 *    Caches, block tables, q_rot, workspaces and err_word stay in device
 *    memory.
 *  - The caller owns every buffer. The library never allocates device memory,
 *    never synchronises, and keeps no pointer after a call returns.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *    stream) and runs asynchronously; a host-side status says only that the
 *    arguments were accepted and the launches were enqueued.
 *  - Argument errors are found on the host and returned BEFORE anything is
 *    launched (MQA_ERR_INVALID_ARG / MQA_ERR_UNSUPPORTED). Errors that only
 *    the data can show (a position, length or block-table entry out of
 *    range) are found on the device: the kernel ORs an MQA_DEVERR_* bit into
 *    the caller's `err_word` (device int32, zeroed by the caller) and skips
 *    that sequence's work; it never traps.
 *  - Tensors are dense row-major with the stated shapes; every base pointer
 *    must be 16-byte aligned.
 */
#ifndef MQA_DECODE_H
#define MQA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MQA_API __attribute__((visibility("default")))
#else
#define MQA_API
#endif

struct CUstream_st;
typedef struct CUstream_st* mqa_stream_t; /* same type as cudaStream_t */

typedef enum mqa_status {
  MQA_OK = 0,
  MQA_ERR_INVALID_ARG = 1, /* null pointer, bad shape, misaligned pointer */
  MQA_ERR_UNSUPPORTED = 2, /* valid but not built: head_dim, dtype, variant */
  MQA_ERR_CUDA = 3,        /* a CUDA runtime call or a launch failed */
  MQA_ERR_WORKSPACE = 4    /* workspace missing or smaller than needed */
} mqa_status;

typedef enum mqa_dtype {
  MQA_BF16 = 0,
  MQA_F32 = 1,
  MQA_U8 = 2, /* cache only: uint8 codes + (scale, zero point) per cached (token, kv head); q/k/v new in bf16 */
  MQA_FP8_E5M2 = 3 /* cache only: fp8 e5m2 values, one byte per element; q/k/v new in bf16 */
} mqa_dtype;

/* Which decode-attention kernel to run (gqa_decode_attention `variant`). */
typedef enum mqa_variant {
  MQA_VARIANT_AUTO = 0,        /* tensor cores for a bf16 cache, else CUDA cores */
  MQA_VARIANT_CUDA_CORE = 1,   /* fp32 FMA on CUDA cores; bf16 and f32 caches */
  MQA_VARIANT_TENSOR_CORE = 2  /* bf16 tensor-core MMA; bf16 cache only */
} mqa_variant;

/* Bits a kernel ORs into the caller's device error word. */
#define MQA_DEVERR_POS_RANGE 0x1u  /* append position < 0, >= capacity, or past the block table */
#define MQA_DEVERR_PAGE_RANGE 0x2u /* a block-table entry in use lies outside [0, num_pages) */
#define MQA_DEVERR_SEQ_LEN 0x4u    /* seq_len < 1, > capacity, > max_seq_len or past the block table */
#define MQA_DEVERR_TIMEOUT 0x8u    /* a bounded wait inside a kernel ran out (the result is invalid) */
#define MQA_DEVERR_U8_SCALE 0x10u  /* MQA_U8: a V scale above 1023 was read; those output rows are invalid */

/*
 * Where the KV cache of one layer lives.
 *
 * Contiguous (paged == 0): k_cache and v_cache are each
 *     [batch, h_kv, capacity, head_dim]   (the pages' [batch, kv_heads, tokens, head_dim])
 * Paged (paged == 1): k_cache and v_cache are each a page pool
 *     [num_pages, h_kv, page_size, head_dim]
 *   and block_table is a device int32 [batch, max_pages_per_seq]: token t of
 *   sequence b lives in page block_table[b * max_pages_per_seq + t / page_size]
 *   at row t % page_size. Entries past a sequence's last page are not read.
 *   Several sequences may share a page (read path only).
 *
 * cache_dtype applies to both caches and to q_new / k_new / v_new.
 * Requirements: h_q % h_kv == 0; head_dim in {64, 128}; batch >= 1;
 * page_size a power of two in [16, 256] (paged).
 *
 * MQA_U8 cache ("KV Cache 최적화 심층 분석", QuantizedKVCache): each cached
 * (token, kv head) row of head_dim values is stored as uint8 codes with a
 * float32 (scale, zero_point) pair in k_scale_zero / v_scale_zero
 * ([batch, h_kv, capacity, 2] contiguous, [num_pages, h_kv, page_size, 2]
 * paged); the value is (code - zero_point) * scale. kv_append_rope quantises
 * the new row: scale = (max - min) / 255 (1 if max == min), zero_point =
 * round(-min / scale) clamped to [0, 255], code = round(x / scale +
 * zero_point) clamped to [0, 255], in float32, rounding half to even; the
 * key is quantised after its fp64 rotation, rounded to float32. q_new,
 * k_new and v_new are bf16. Attention over a MQA_U8 cache runs on tensor
 * cores only.
 *
 * MQA_FP8_E5M2 cache (the fp8_e5m2 KV-cache dtype of the pages' vLLM
 * serving examples): one byte per element, 1 sign, 5 exponent (bias 15) and
 * 2 mantissa bits, no scale; k_scale_zero / v_scale_zero are unused.
 * kv_append_rope rounds the new row to nearest (ties to even) -- the key
 * once, from its fp64 rotation -- and saturates magnitudes beyond 57344 to
 * it. q_new, k_new and v_new are bf16; attention on tensor cores only. One
 * new token per sequence runs on the warp-MMA kernels (codes widened to fp16,
 * fp16 query) or, for 16 < G <= 32 contiguous at head_dim 128, the MQA
 * tcgen05 kernel. Several new tokens with 32 or more query rows per kv head
 * over a contiguous cache at head_dim 128 (multi-token calls, prefill) run
 * on the tcgen05 kernel's fp8 form: the code tiles are the MMA's B operand as
 * they sit in memory, the query and the probabilities enter as two e4m3
 * parts each (hi + lo, the query scaled by 64 first), so q and P keep about 8
 * significant bits of precision beyond a single e4m3 rounding; fewer rows, or
 * a paged pool, take the warp-MMA kernels.
 *
 * Bounded waits: inside the attention kernels every wait for another warp's
 * progress (a tile landing, a tile freed, a product done) gives up after
 * wait_limit_ns nanoseconds (0 selects the default, one second). The kernel
 * then ORs MQA_DEVERR_TIMEOUT into err_word, lets its own copies and tensor
 * core products still in flight complete (those waits keep the one-second
 * limit), releases what it holds and returns; its outputs are then invalid,
 * and the next call on the stream runs normally. A healthy wait lasts
 * microseconds: a short limit only serves to exercise this path (below one
 * second the waits poll instead of letting the hardware suspend the warp,
 * which could outlast the limit). (The
 * one-token MQA kernels over a one-byte cache -- 16 < G <= 32 over MQA_U8
 * or MQA_FP8_E5M2, contiguous, head_dim 128 -- always use one second.)
 *
 * window: 0 = the attention reads every cached token [0, L); W > 0 = a
 * sliding window: only the last W tokens [max(0, L - W), L) are read
 * ("KV Cache 최적화 심층 분석", SlidingWindowAttention keeps the cache's last
 * window_size tokens). Rows and pages wholly before the window are never
 * read, so a paged cache may release them (table entries -1).
 */
typedef struct mqa_kv_layout {
  int32_t cache_dtype; /* mqa_dtype */
  int32_t batch;
  int32_t h_q;
  int32_t h_kv;
  int32_t head_dim;
  int32_t paged;
  void* k_cache;
  void* v_cache;
  int64_t capacity; /* contiguous: tokens per (sequence, kv head) row; unused when paged */
  int32_t page_size;
  int32_t num_pages;
  int32_t max_pages_per_seq;
  int32_t window; /* 0: full context; W > 0: sliding window of the last W tokens */
  const int32_t* block_table;
  void* k_scale_zero; /* MQA_U8 only: float32 (scale, zero_point) per cached row of K */
  void* v_scale_zero; /* MQA_U8 only: same for V */
  uint64_t wait_limit_ns; /* 0: 1 s; see "Bounded waits" above */
} mqa_kv_layout;

/*
 * kv_append_rope -- steps 1-2 of the decode step for every sequence b:
 * p = pos[b] (the new token's 0-based position = its sequence length after
 * the append minus one).
 *   q_rot[b, h, :]  = RoPE(q_new[b, h, :], p)               (fp32 out)
 *   cache K at (b, j, p) = round(RoPE(k_new[b, j, :], p))   (cache dtype)
 *   cache V at (b, j, p) = v_new[b, j, :]                   (bit copy)
 * RoPE rotates adjacent pairs (x[2i], x[2i+1]) by angle p * theta_i,
 * theta_i = rope_base^(-2i/head_dim): (x cos - y sin, x sin + y cos). The
 * angle and the key's rotation are evaluated in fp64 and the key is rounded
 * once (nearest, ties to even) to the cache dtype; the query is rotated in
 * fp32. ("KV Cache" explainer, Langkah 3: each key is rotated by its
 * position once and stored rotated; only the newest token is projected.)
 *
 * q_new [batch, h_q, head_dim], k_new / v_new [batch, h_kv, head_dim]
 * (cache dtype), pos [batch] int32, q_rot [batch, h_q, head_dim] fp32 output.
 * A paged layout needs the page of position p already in the block table.
 * A sequence whose p or page is out of range sets MQA_DEVERR_POS_RANGE /
 * MQA_DEVERR_PAGE_RANGE and its cache is left untouched (q_rot is written).
 */
MQA_API mqa_status kv_append_rope(const mqa_kv_layout* layout, const void* q_new, const void* k_new, const void* v_new,
                          const int32_t* pos, double rope_base, float* q_rot, int32_t* err_word,
                          mqa_stream_t stream);

/*
 * gqa_decode_attention -- step 3: for every sequence b and query head h,
 *   O[b, h, :] = sum_t softmax_t(scale * q_rot[b, h, :] . K[b, g(h), t, :]) V[b, g(h), t, :]
 * over tokens t in [0, seq_lens[b]) (with layout->window = W > 0: t in
 * [max(0, seq_lens[b] - W), seq_lens[b])), g(h) = floor(h / (h_q / h_kv)).
 * Each kernel block streams the K/V tiles of one (sequence, kv head) token
 * range from HBM once and serves all G query heads of the group from that
 * load, with an fp32 online softmax (FlashAttention's running max and sum,
 * "Arsitektur Inferensi LLM", section 5).
 *
 * q_rot       [batch, h_q, head_dim] fp32 (output of kv_append_rope)
 * seq_lens    [batch] int32 device, lengths after the append (>= 1)
 * max_seq_len host upper bound of every seq_lens[b]; sizes the grid and the split
 * scale       score scale, normally 1/sqrt(head_dim)
 * num_splits  1 = no split; > 1 = split the token axis into that many equal
 *             chunks (rounded up to 64 tokens) and merge them with
 *             splitkv_combine; 0 = let the library choose (mqa_choose_splits)
 * out         [batch, h_q, head_dim] in out_dtype (mqa_dtype)
 * lse_out     optional [batch, h_q] fp32: natural-log sum of exp(scaled score)
 * workspace   device scratch of at least mqa_workspace_size(...) bytes when the
 *             call splits (may be NULL when it does not); 256-byte aligned
 * variant     mqa_variant
 * A sequence with an out-of-range length or block-table entry sets its
 * MQA_DEVERR_* bit; its output rows are then unspecified.
 */
MQA_API mqa_status gqa_decode_attention(const mqa_kv_layout* layout, const float* q_rot, const int32_t* seq_lens,
                                int32_t max_seq_len, float scale, int32_t num_splits, void* out,
                                int32_t out_dtype, float* lse_out, void* workspace, size_t workspace_bytes,
                                int32_t variant, int32_t* err_word, mqa_stream_t stream);

/*
 * splitkv_combine -- merge per-split results of disjoint token ranges:
 *   LSE = log sum_s exp(lse_part[b, h, s]),
 *   out[b, h, :] = sum_s exp(lse_part[b, h, s] - LSE) * o_part[b, h, s, :].
 * o_part [batch, h_q, num_splits, head_dim] fp32 holds each split's
 * NORMALISED output; lse_part [batch, h_q, num_splits] fp32 its natural-log
 * sum of exp(score). A split with no tokens has lse = -inf and is ignored;
 * at least one split per row must be non-empty. out is [batch, h_q,
 * head_dim] in out_dtype; lse_out (optional) [batch, h_q] fp32.
 */
MQA_API mqa_status splitkv_combine(const float* o_part, const float* lse_part, int32_t batch, int32_t h_q,
                           int32_t num_splits, int32_t head_dim, void* out, int32_t out_dtype, float* lse_out,
                           mqa_stream_t stream);

/*
 * mqa_decode_step -- the whole decode step in one call: kv_append_rope, then
 * gqa_decode_attention (and the combine when it splits), on one stream. The
 * arguments mean what they mean in those two calls; q_rot is the caller's
 * fp32 [batch, h_q, head_dim] scratch that carries the rotated query from the
 * first launch to the second. Every argument of both calls is checked before
 * the first launch. On the tensor-core path the step is ONE launch (plus the
 * combine when it splits; two splits of the bf16 and e5m2 tcgen05 one-token
 * kernels merge inside the launch) when one block serves all query heads of a
 * kv head -- at most 32 of them on the warp-MMA kernels, 32 to 128 on the bf16
 * tcgen05 kernel (contiguous cache, head_dim 128), 17 to 32 on the
 * one-byte-cache tcgen05 kernels: the attention kernel rotates q and k_new
 * itself, writes the new token's slot (quantised, for a uint8 or e5m2 cache,
 * exactly as kv_append_rope writes it) and q_rot, and then reads that slot
 * back. Otherwise the attention launch directly follows the append launch and
 * is allowed to start while the append is still running: it streams every
 * cached row except the appended one, the lengths and the block table early,
 * and waits for the append before it reads q_rot or the new token's row.
 */
MQA_API mqa_status mqa_decode_step(const mqa_kv_layout* layout, const void* q_new, const void* k_new,
                                   const void* v_new, const int32_t* pos, const int32_t* seq_lens,
                                   int32_t max_seq_len, double rope_base, float scale, int32_t num_splits,
                                   float* q_rot, void* out, int32_t out_dtype, float* lse_out, void* workspace,
                                   size_t workspace_bytes, int32_t variant, int32_t* err_word, mqa_stream_t stream);

/*
 * gqa_decode_attention_noalloc -- gqa_decode_attention for callers that cannot
 * allocate device memory (the pages have no counterpart of this call).
 *
 * A split run needs scratch for its per-split partial results; normally the
 * caller allocates it and passes it as `workspace`. Callers that own no
 * device allocator -- for instance a plugin loaded into a process whose
 * framework has reserved the device memory for its own pool, or a serving
 * loop that must not take cudaMalloc's implicit device synchronisation --
 * use this call instead: the scratch is a fixed 32 MiB array inside the
 * library, which every GPU that loads the library holds until the process
 * exits. The call itself allocates nothing and frees nothing.
 *
 * Arguments as in gqa_decode_attention, without workspace. Returns
 * MQA_ERR_WORKSPACE when mqa_workspace_size(layout, max_seq_len, num_splits,
 * variant) exceeds 32 MiB.
 * The first call in each CUDA context (per device; again after the context is
 * destroyed and created anew, e.g. by cudaDeviceReset) looks up the scratch's
 * device address with that device current; make that first call before any
 * stream capture. A failed lookup returns MQA_ERR_CUDA with its text in
 * mqa_last_cuda_error.
 * All calls share the one scratch array and it keeps the last call's
 * contents; nothing in it needs clearing, since every call rewrites each
 * partial result it reads. Calls whose work overlaps on the GPU (two streams,
 * or two host threads on different streams) race on the scratch and must be
 * serialised by the caller.
 */
MQA_API mqa_status gqa_decode_attention_noalloc(const mqa_kv_layout* layout, const float* q_rot,
                                                const int32_t* seq_lens, int32_t max_seq_len, float scale,
                                                int32_t num_splits, void* out, int32_t out_dtype, float* lse_out,
                                                int32_t variant, int32_t* err_word, mqa_stream_t stream);

/*
 * Multi-token decode: n_new query tokens per sequence in one pass -- the
 * target model's verification of drafted tokens in speculative decoding
 * ("Arsitektur Inferensi LLM", section 7: the gamma drafted tokens are
 * checked in parallel, and the result must equal decoding them one by one).
 *
 * kv_append_rope_multi: q_new [batch, n_new, h_q, head_dim], k_new / v_new
 *   [batch, n_new, h_kv, head_dim] (cache dtype); new token i of sequence b
 *   is rotated by and stored at position pos[b] + i; q_rot [batch, n_new, h_q,
 *   head_dim] fp32 output. Same arithmetic and device errors as kv_append_rope.
 * gqa_decode_attention_multi: seq_lens[b] = length after the append; query
 *   token i of sequence b (position L - n_new + i) attends to the tokens
 *   [0, L - n_new + i] (with a window W: the last W of them) -- causal among
 *   the new tokens. out [batch, n_new, h_q, head_dim], lse_out [batch, n_new,
 *   h_q]. max_seq_len >= n_new; a sequence with L < n_new sets
 *   MQA_DEVERR_SEQ_LEN. The (token, query head) pairs of a kv head are the
 *   rows of one MMA tile set, so the K/V bytes are read once for all n_new
 *   tokens.
 * mqa_decode_step_multi: the two calls on one stream, pos[b] = L - n_new; ONE
 *   launch (plus the combine when it splits and does not merge in a cluster)
 *   when the attention kernel takes the append over -- bf16 cache, one block
 *   for all (token, head) rows of a kv head: the warp-MMA kernel with n_new
 *   <= 8 and G n_new <= 32, the tcgen05 kernel with n_new <= 16 and G n_new
 *   <= 128 -- with the cache rows bit for bit those of the two calls.
 * 1 <= n_new <= 32 for the attention (kv_append_rope_multi takes any n_new;
 * longer runs of new tokens go to gqa_prefill_attention). n_new > 1 runs on
 * tensor cores only (MQA_ERR_UNSUPPORTED on CUDA cores): over a bf16 cache,
 * contiguous or paged (32 or more query rows per kv head on the tcgen05
 * kernel, which gathers a paged key tile page by page); over a MQA_FP8_E5M2
 * cache (contiguous with head_dim 128 and (h_q / h_kv) * n_new >= 32: the
 * tcgen05 kernel's fp8 form; otherwise the one-byte warp-MMA kernel); over a
 * MQA_U8 cache (the one-byte warp-MMA kernel, contiguous or paged). Over a
 * one-byte cache the append is always its own launch. n_new = 1 is exactly
 * the single-token call.
 */
MQA_API mqa_status kv_append_rope_multi(const mqa_kv_layout* layout, int32_t n_new, const void* q_new,
                                        const void* k_new, const void* v_new, const int32_t* pos, double rope_base,
                                        float* q_rot, int32_t* err_word, mqa_stream_t stream);
MQA_API mqa_status gqa_decode_attention_multi(const mqa_kv_layout* layout, int32_t n_new, const float* q_rot,
                                              const int32_t* seq_lens, int32_t max_seq_len, float scale,
                                              int32_t num_splits, void* out, int32_t out_dtype, float* lse_out,
                                              void* workspace, size_t workspace_bytes, int32_t variant,
                                              int32_t* err_word, mqa_stream_t stream);
MQA_API mqa_status mqa_decode_step_multi(const mqa_kv_layout* layout, int32_t n_new, const void* q_new,
                                         const void* k_new, const void* v_new, const int32_t* pos,
                                         const int32_t* seq_lens, int32_t max_seq_len, double rope_base, float scale,
                                         int32_t num_splits, float* q_rot, void* out, int32_t out_dtype,
                                         float* lse_out, void* workspace, size_t workspace_bytes, int32_t variant,
                                         int32_t* err_word, mqa_stream_t stream);
/* Split count / workspace bytes of gqa_decode_attention_multi (as the
 * single-token queries below; -1 / 0 for invalid arguments). */
MQA_API int32_t mqa_choose_splits_multi(const mqa_kv_layout* layout, int32_t n_new, int32_t max_seq_len,
                                        int32_t variant);
MQA_API size_t mqa_workspace_size_multi(const mqa_kv_layout* layout, int32_t n_new, int32_t max_seq_len,
                                        int32_t num_splits, int32_t variant);

/*
 * Prefill: the prompt's n_new tokens of every sequence appended and attended
 * causally in one pass ("KV Cache" explainer, Langkah 1 and 4: the prompt's
 * keys and values are computed in one pass and stored; prefill is
 * compute-bound). The arithmetic is that of the multi-token calls above --
 * query token i of sequence b (position L - n_new + i) attends to the keys
 * [0, L - n_new + i] (or the last W of them) -- on the tensor-memory tensor
 * cores (tcgen05): one block per (sequence, kv head, 256 (token, query head)
 * rows as two 128-row query tiles), S and O accumulated in tensor memory.
 *
 * gqa_prefill_attention: q_rot [batch, n_new, h_q, 128] fp32 (from
 *   kv_append_rope_multi), seq_lens[b] = L after the append (>= n_new; L > n_new
 *   means a cached prefix of L - n_new tokens), out [batch, n_new, h_q, 128],
 *   lse_out optional [batch, n_new, h_q].
 * mqa_prefill_step: kv_append_rope_multi (pos[b] = L - n_new), then
 *   gqa_prefill_attention, on one stream.
 * head_dim 128 with a bf16 cache, contiguous or paged (a key tile gathered
 * page by page from the pool the block table names, the prompt's rows
 * appended into its pages), or a contiguous MQA_FP8_E5M2 cache (the kernel's
 * fp8 form described with MQA_FP8_E5M2). A MQA_U8 cache (contiguous or paged)
 * and a paged MQA_FP8_E5M2 pool, head_dim 64 or 128, take the one-byte
 * warp-MMA kernel's multi-token form over the whole prompt instead (32 rows per
 * block; correct, not tuned for prompts). MQA_ERR_UNSUPPORTED otherwise. No
 * workspace. A block-table entry outside the pool for a page the prompt
 * attends or is appended to sets MQA_DEVERR_PAGE_RANGE (that page reads as
 * zeros). A bounded wait that runs out sets
 * MQA_DEVERR_TIMEOUT and every later block of the launch returns at once.
 */
MQA_API mqa_status gqa_prefill_attention(const mqa_kv_layout* layout, int32_t n_new, const float* q_rot,
                                         const int32_t* seq_lens, int32_t max_seq_len, float scale, void* out,
                                         int32_t out_dtype, float* lse_out, int32_t* err_word, mqa_stream_t stream);
MQA_API mqa_status mqa_prefill_step(const mqa_kv_layout* layout, int32_t n_new, const void* q_new, const void* k_new,
                                    const void* v_new, const int32_t* pos, const int32_t* seq_lens,
                                    int32_t max_seq_len, double rope_base, float scale, float* q_rot, void* out,
                                    int32_t out_dtype, float* lse_out, int32_t* err_word, mqa_stream_t stream);

/* Split count gqa_decode_attention uses for num_splits = 0 on the current device
 * (>= 1), or -1 if the layout is invalid. */
MQA_API int32_t mqa_choose_splits(const mqa_kv_layout* layout, int32_t max_seq_len, int32_t variant);

/* Workspace bytes gqa_decode_attention needs for this layout, bound and split
 * count (num_splits = 0: the count mqa_choose_splits returns); 0 when the call
 * does not split. */
MQA_API size_t mqa_workspace_size(const mqa_kv_layout* layout, int32_t max_seq_len, int32_t num_splits, int32_t variant);

/* Kernel launches one mqa_decode_step_multi call (n_new = 1: mqa_decode_step)
 * makes for these arguments: 1 when the attention kernel appends the new
 * tokens itself and needs no combine, 2 for append + attention or attention +
 * combine, 3 for all three; -1 when the call would be refused. If
 * fused_append is not NULL it receives 1 when the append runs inside the
 * attention launch. Host only, no device work. (The library's own routing,
 * not an operation of the pages.) */
MQA_API int32_t mqa_step_launches(const mqa_kv_layout* layout, int32_t n_new, int32_t max_seq_len, int32_t num_splits,
                                  int32_t variant, int32_t* fused_append);

/* Static description of a status code. */
MQA_API const char* mqa_status_string(mqa_status status);

/* Text of the last CUDA error seen by this thread's calls ("" if none). */
MQA_API const char* mqa_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MQA_DECODE_H */
