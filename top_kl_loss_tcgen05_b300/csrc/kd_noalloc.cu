// kd_noalloc.cu - the top-K cache extraction for callers that cannot allocate
// device memory.
//
// kd_topk_cache needs a small caller-provided workspace: a status word and
// counters. Some callers cannot provide one. Examples are a cache-extraction
// step running inside a host application that owns every device allocation
// through its own pool, and a latency-bound loop where cudaMalloc's implicit
// device synchronisation is not acceptable. kd_topk_cache_noalloc takes the
// same inputs and outputs but keeps its scratch in a fixed array in device
// memory that belongs to this library. It calls no cudaMalloc, cudaFree or
// allocating library routine.
//
// The array lives in every GPU that loads libkd, until the process exits. It
// is shared by all calls on that device and keeps the last call's contents.
// Each call clears it on its stream first, so calls that overlap on the GPU
// (different streams, no ordering between them) race on it.
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/kd.h"

namespace {

// Fixed scratch of the no-allocation variant: large enough for the top-K
// workspace (kd_topk_workspace_size, 256 bytes today).
constexpr size_t kNoAllocScratchBytes = 4096;
static __device__ __align__(256) unsigned char g_topk_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_topk_scratch on the current device. In host code the
// name g_topk_scratch is only a host-side stand-in, so the address must come
// from cudaGetSymbolAddress, once per device, with that device current.
int scratch_ptr(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KD_ERR_CUDA;
  std::lock_guard<std::mutex> g(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_topk_scratch);
    if (e != cudaSuccess || !p) {
      if (std::getenv("KD_DEBUG"))
        std::fprintf(stderr, "libkd: cudaGetSymbolAddress failed: %s\n", cudaGetErrorString(e));
      return KD_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return KD_OK;
}

}  // namespace

extern "C" int kd_topk_cache_noalloc(const void* logits, int32_t dtype, int64_t T, int64_t V, int64_t ld,
                                     int32_t K, int32_t* ids, float* logp, void* stream) {
  if (!logits || !ids || !logp || T <= 0 || V <= 0 || K <= 0 || K > V || ld < V) return KD_ERR_INVALID_ARG;
  if (dtype != KD_BF16 && dtype != KD_F32) return KD_ERR_INVALID_ARG;
  const size_t need = kd_topk_workspace_size(T, V, K, dtype);
  if (need > kNoAllocScratchBytes) {
    if (std::getenv("KD_DEBUG"))
      std::fprintf(stderr, "libkd: kd_topk_cache_noalloc needs %zu scratch bytes, the fixed array holds %zu\n",
                   need, kNoAllocScratchBytes);
    return KD_ERR_WORKSPACE;
  }
  void* ws = nullptr;
  const int st = scratch_ptr(&ws);
  if (st != KD_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The status word and counters must start at zero for this call.
  if (cudaMemsetAsync(ws, 0, need, s) != cudaSuccess) return KD_ERR_CUDA;
  return kd_topk_cache(logits, dtype, T, V, ld, K, ids, logp, ws, kNoAllocScratchBytes, stream);
}
