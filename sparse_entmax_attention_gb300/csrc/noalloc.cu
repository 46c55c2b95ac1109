// noalloc.cu -- a decode entry point for callers that cannot allocate device
// memory: the full-cache softmax decode with its scratch (split partials and
// "last block" counters) in a fixed array compiled into the library.
#include <mutex>
#include <string.h>

#include "common.cuh"

namespace ekv {

// The scratch every GPU that loads this library holds until the process
// exits. One decode fits when entmaxkv_workspace_bytes(cfg, n_seqs,
// ENTMAXKV_POLICY_SOFTMAX, 0) is at most this size.
constexpr size_t kNoAllocScratchBytes = 8u << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
static void* g_scratch_ptr[kMaxDevices];
static std::mutex g_scratch_mu;

// Device address of the scratch on the current device, looked up once per
// device (the symbol's host-side name is not a device address).
static cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace ekv

using namespace ekv;

extern "C" size_t entmaxkv_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

extern "C" int32_t entmaxkv_decode_softmax_noalloc(const entmaxkv_config* cfg,
                                                   const entmaxkv_cache* cache, const void* q,
                                                   const int32_t* seq_ids, int32_t n_seqs,
                                                   float* out, float* lse, void* stream) {
  if (!cfg || !cache || !q || !out || n_seqs < 0) return ENTMAXKV_ERR_INVALID_ARG;
  if (n_seqs == 0) return ENTMAXKV_OK;
  const size_t need = entmaxkv_workspace_bytes(cfg, n_seqs, ENTMAXKV_POLICY_SOFTMAX, 0);
  if (need == 0) return ENTMAXKV_ERR_INVALID_ARG;
  if (need > kNoAllocScratchBytes) return ENTMAXKV_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return ENTMAXKV_ERR_CUDA;
  // The ordinary decode path, pointed at the fixed scratch: it clears the
  // counters at the start of the call, so nothing carries over between calls.
  return entmaxkv_decode(cfg, cache, q, seq_ids, n_seqs, 2.0f, ENTMAXKV_POLICY_SOFTMAX, 0, 0.0f, 0u,
                         scratch, kNoAllocScratchBytes, out, nullptr, 0, nullptr, lse, nullptr,
                         stream);
}
