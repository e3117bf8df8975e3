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

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/kd.h"
#include "kd_internal.h"

namespace {

// Fixed scratch of the no-allocation variant: large enough for the top-K
// workspace (kd_topk_workspace_size, 256 bytes today).
constexpr size_t kNoAllocScratchBytes = 4096;
static __device__ __align__(256) unsigned char g_topk_scratch[kNoAllocScratchBytes];

// Driver calls that identify the current context, so that a cached address
// is looked up again after the device's context was torn down and recreated
// (cudaDeviceReset reloads the module, and the array may move).
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;
std::once_flag g_ctx_once;

void load_ctx_fns() {
  cudaDriverEntryPointQueryResult q;
  void* fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(fn);
  fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(fn);
  (void)cudaGetLastError();
}

// Id of the current context (unique for the life of the process), 0 if
// there is none yet or it cannot be read.
unsigned long long current_ctx_id() {
  std::call_once(g_ctx_once, load_ctx_fns);
  if (!g_ctx_get_current || !g_ctx_get_id) return 0;
  CUcontext c = nullptr;
  if (g_ctx_get_current(&c) != CUDA_SUCCESS || !c) return 0;
  unsigned long long id = 0;
  if (g_ctx_get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};
unsigned long long g_scratch_ctx[kMaxDevices] = {0};

// Device address of g_topk_scratch on the current device. In host code the
// name g_topk_scratch is only a host-side stand-in, so the address comes
// from cudaGetSymbolAddress, with the device current: on the first call on a
// device, and again whenever that device's context has changed since.
int scratch_ptr(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    (void)cudaGetLastError();
    return KD_ERR_CUDA;
  }
  std::lock_guard<std::mutex> g(g_mu);
  const unsigned long long ctx = current_ctx_id();
  if (!g_scratch_ptr[dev] || ctx == 0 || ctx != g_scratch_ctx[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_topk_scratch);
    if (e != cudaSuccess || !p) {
      if (std::getenv("KD_DEBUG"))
        std::fprintf(stderr, "libkd: cudaGetSymbolAddress failed: %s\n", cudaGetErrorString(e));
      (void)cudaGetLastError();  // do not leave the error for the caller's next CUDA call
      g_scratch_ptr[dev] = nullptr;
      return KD_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = current_ctx_id();  // the lookup made the context current if it was not
  }
  *out = g_scratch_ptr[dev];
  return KD_OK;
}

}  // namespace

extern "C" int kd_topk_cache_noalloc(const void* logits, int32_t dtype, int64_t T, int64_t V, int64_t ld,
                                     int32_t K, int32_t* ids, float* logp, void* stream) {
  // Every check of kd_topk_cache comes first, so a refused call has put
  // nothing on the stream.
  const int chk = kd::topk_check_args(logits, dtype, T, V, ld, K, ids, logp);
  if (chk != KD_OK) return chk;
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
