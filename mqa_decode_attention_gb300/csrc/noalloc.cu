// gqa_decode_attention_noalloc: decode attention for callers that cannot
// allocate device memory.
//
// When the token axis is split, gqa_decode_attention needs a scratch buffer
// for the per-split partial outputs, which its caller normally allocates.
// Some callers have no way to do that: a plugin loaded into a process whose
// framework has already reserved the device memory for its own pool, code
// written against a runtime that exposes no device allocator, or a serving
// loop that must not pay for cudaMalloc's implicit device synchronisation.
// This entry point keeps the scratch in a fixed array inside the library
// instead, so the caller passes only inputs and outputs.
//
// The array is a file-scope __device__ variable: every GPU on which the
// library is loaded holds it (kScratchBytes) until the process exits. Its
// device address is looked up once per device, on that device's first call,
// with the device current.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/mqa_decode.h"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;  // 32 MiB

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;

// Device address of g_scratch on `dev`, looked up on first use.
void* scratch_on(int dev) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" mqa_status gqa_decode_attention_noalloc(const mqa_kv_layout* layout, const float* q_rot,
                                                   const int32_t* seq_lens, int32_t max_seq_len, float scale,
                                                   int32_t num_splits, void* out, int32_t out_dtype,
                                                   float* lse_out, int32_t variant, int32_t* err_word,
                                                   mqa_stream_t stream) {
  const size_t need = mqa_workspace_size(layout, max_seq_len, num_splits, variant);
  if (need > kScratchBytes) return MQA_ERR_WORKSPACE;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MQA_ERR_CUDA;
  void* ws = scratch_on(dev);
  if (ws == nullptr) return MQA_ERR_CUDA;
  return gqa_decode_attention(layout, q_rot, seq_lens, max_seq_len, scale, num_splits, out, out_dtype, lse_out, ws,
                              kScratchBytes, variant, err_word, stream);
}
