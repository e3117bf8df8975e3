/*
 * c_abi_example.c - the library used from plain C, with no Python: device
 * buffers from cudaMalloc, the fused KL loss (forward, backward) and the
 * top-K cache through include/kd.h. tests/test_c_abi_gpu.py builds this file
 * with gcc, runs it, and compares what it writes with the Python binding on
 * the same inputs.
 *
 * usage: c_abi_example <out_dir>
 * Writes to <out_dir>: H.bin (bf16 [T, d]), W.bin (bf16 [V, d]), ids.bin,
 * logp.bin (the cache, [T, K]), loss.bin, lse.bin, dH.bin, dW.bin, and
 * tk_ids.bin, tk_logp.bin (kd_topk_cache of fp32 logits x.bin [T, V]).
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "kd.h"

enum { T = 300, D = 128, V = 3000, K = 16, CHUNK = 64 };

static uint32_t rng_state = 12345u;
static float urand(void) { /* LCG, uniform in [-1, 1) */
  rng_state = rng_state * 1664525u + 1013904223u;
  return (float)(rng_state >> 8) / 8388608.0f - 1.0f;
}
static uint16_t to_bf16(float f) { /* round to nearest even */
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

#define CK(x)                                                           \
  do {                                                                  \
    cudaError_t e_ = (x);                                               \
    if (e_ != cudaSuccess) {                                            \
      fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));          \
      return 1;                                                         \
    }                                                                   \
  } while (0)
#define KD(x)                                                           \
  do {                                                                  \
    int s_ = (x);                                                       \
    if (s_ != KD_OK) {                                                  \
      fprintf(stderr, "%s: %s\n", #x, kd_status_string(s_));            \
      return 1;                                                         \
    }                                                                   \
  } while (0)

static int dump(const char* dir, const char* name, const void* host, size_t bytes) {
  char path[1024];
  snprintf(path, sizeof(path), "%s/%s", dir, name);
  FILE* f = fopen(path, "wb");
  if (!f || fwrite(host, 1, bytes, f) != bytes) {
    fprintf(stderr, "cannot write %s\n", path);
    if (f) fclose(f);
    return 1;
  }
  fclose(f);
  return 0;
}

static int fetch_dump(const char* dir, const char* name, const void* dev, size_t bytes) {
  void* h = malloc(bytes);
  if (!h) return 1;
  if (cudaMemcpy(h, dev, bytes, cudaMemcpyDeviceToHost) != cudaSuccess) {
    free(h);
    return 1;
  }
  int r = dump(dir, name, h, bytes);
  free(h);
  return r;
}

int main(int argc, char** argv) {
  if (argc != 2) {
    fprintf(stderr, "usage: %s <out_dir>\n", argv[0]);
    return 2;
  }
  const char* dir = argv[1];
  static uint16_t H[T * D], W[V * D];
  static int32_t ids[T * K];
  static float logp[T * K], x[T * V];
  for (int i = 0; i < T * D; ++i) H[i] = to_bf16(urand());
  for (int i = 0; i < V * D; ++i) W[i] = to_bf16(0.1f * urand());
  for (int t = 0; t < T; ++t) {
    const int a = (int)((urand() + 1.0f) * 0.5f * V) % V;
    for (int k = 0; k < K; ++k) {
      ids[t * K + k] = (a + 7 * k) % V; /* distinct: 7 k < V */
      logp[t * K + k] = -1.0f - 0.5f * (float)k + 0.1f * urand();
    }
  }
  for (int i = 0; i < T * V; ++i) x[i] = 4.0f * urand();

  void *dH_in, *dW_in, *dids, *dlogp, *dx;
  float *dloss, *dlse, *ddH, *ddW, *dtklogp;
  int32_t* dtkids;
  CK(cudaMalloc(&dH_in, sizeof(H)));
  CK(cudaMalloc(&dW_in, sizeof(W)));
  CK(cudaMalloc(&dids, sizeof(ids)));
  CK(cudaMalloc(&dlogp, sizeof(logp)));
  CK(cudaMalloc(&dx, sizeof(x)));
  CK(cudaMalloc((void**)&dloss, sizeof(float)));
  CK(cudaMalloc((void**)&dlse, T * sizeof(float)));
  CK(cudaMalloc((void**)&ddH, (size_t)T * D * sizeof(float)));
  CK(cudaMalloc((void**)&ddW, (size_t)V * D * sizeof(float)));
  CK(cudaMalloc((void**)&dtkids, (size_t)T * K * sizeof(int32_t)));
  CK(cudaMalloc((void**)&dtklogp, (size_t)T * K * sizeof(float)));
  CK(cudaMemcpy(dH_in, H, sizeof(H), cudaMemcpyHostToDevice));
  CK(cudaMemcpy(dW_in, W, sizeof(W), cudaMemcpyHostToDevice));
  CK(cudaMemcpy(dids, ids, sizeof(ids), cudaMemcpyHostToDevice));
  CK(cudaMemcpy(dlogp, logp, sizeof(logp), cudaMemcpyHostToDevice));
  CK(cudaMemcpy(dx, x, sizeof(x), cudaMemcpyHostToDevice));

  /* the loss: workspace from the size query (aligned by cudaMalloc) */
  const size_t ws_bytes = kd_fused_kl_workspace_size(D, V, K, CHUNK);
  void* ws;
  CK(cudaMalloc(&ws, ws_bytes));
  CK(cudaMemset(ws, 0, ws_bytes));
  KD(kd_fused_kl_fwd(dH_in, dW_in, (const int32_t*)dids, (const float*)dlogp, T, D, V, K, CHUNK, dloss, dlse,
                     NULL, ws, ws_bytes, NULL));
  KD(kd_fused_kl_bwd(dH_in, dW_in, (const int32_t*)dids, (const float*)dlogp, dlse, T, D, V, K, CHUNK,
                     1.0f / T, NULL, ddH, ddW, 0, ws, ws_bytes, NULL));
  /* the top-K cache of fp32 logits */
  const size_t tk_bytes = kd_topk_workspace_size(T, V, K, KD_F32);
  void* tkws;
  CK(cudaMalloc(&tkws, tk_bytes));
  CK(cudaMemset(tkws, 0, tk_bytes));
  KD(kd_topk_cache(dx, KD_F32, T, V, V, K, dtkids, dtklogp, tkws, tk_bytes, NULL));
  CK(cudaDeviceSynchronize());
  KD(kd_read_device_status(ws, NULL));
  KD(kd_read_device_status(tkws, NULL));

  if (dump(dir, "H.bin", H, sizeof(H)) || dump(dir, "W.bin", W, sizeof(W)) || dump(dir, "ids.bin", ids, sizeof(ids)) ||
      dump(dir, "logp.bin", logp, sizeof(logp)) || dump(dir, "x.bin", x, sizeof(x)) ||
      fetch_dump(dir, "loss.bin", dloss, sizeof(float)) || fetch_dump(dir, "lse.bin", dlse, T * sizeof(float)) ||
      fetch_dump(dir, "dH.bin", ddH, (size_t)T * D * sizeof(float)) ||
      fetch_dump(dir, "dW.bin", ddW, (size_t)V * D * sizeof(float)) ||
      fetch_dump(dir, "tk_ids.bin", dtkids, (size_t)T * K * sizeof(int32_t)) ||
      fetch_dump(dir, "tk_logp.bin", dtklogp, (size_t)T * K * sizeof(float)))
    return 1;
  printf("ok\n");
  return 0;
}
