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
// device address is looked up with the device current, on the first call in
// each CUDA context: the cached address is keyed by the context's unique id,
// so a context torn down and created again (cudaDeviceReset, or a driver-API
// caller releasing the primary context) gets the new address, never a stale
// one.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/mqa_decode.h"
#include "launch.h"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;  // 32 MiB

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

template <class F>
F driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return reinterpret_cast<F>(p);
}

// Unique id of the calling thread's current context; false when there is none
// (or the driver entry points are unavailable).
bool current_context_id(unsigned long long* id) {
  static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  if (get_current == nullptr || get_id == nullptr) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_scratch on `dev` (the current device) in the current
// context. The address is cached per device with the id of the context it
// was found in and looked up again whenever that id differs.
cudaError_t scratch_on(int dev, void** out) {
  struct Slot {
    unsigned long long ctx_id;
    void* addr;
  };
  static std::mutex mu;
  static Slot slot[kMaxDevices] = {};
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  unsigned long long id = 0;
  if (current_context_id(&id) && slot[dev].addr != nullptr && slot[dev].ctx_id == id) {
    *out = slot[dev].addr;
    return cudaSuccess;
  }
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);  // makes the device's context current
  if (e != cudaSuccess) return e;
  if (current_context_id(&id)) {
    slot[dev] = Slot{id, p};
  } else {
    slot[dev] = Slot{0, nullptr};  // no id to key on: look the address up on every call
  }
  *out = p;
  return cudaSuccess;
}

mqa_status fail(cudaError_t e) {
  cudaGetLastError();  // leave no stale error for the next call to report
  mqa::record_cuda_error(e);
  return MQA_ERR_CUDA;
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
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(e);
  void* ws = nullptr;
  e = scratch_on(dev, &ws);
  if (e != cudaSuccess) return fail(e);
  return gqa_decode_attention(layout, q_rot, seq_lens, max_seq_len, scale, num_splits, out, out_dtype, lse_out, ws,
                              kScratchBytes, variant, err_word, stream);
}
