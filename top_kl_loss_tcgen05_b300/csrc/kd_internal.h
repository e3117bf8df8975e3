// kd_internal.h - host-side declarations shared by the libkd translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace kd {

// Tile shape of the projection GEMMs: 128 rows of the M operand, BK = 64
// reduction elements per pipeline stage (one 128-byte swizzle row of bf16).
constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kBNLogits = 256;  // forward / recompute: N tile over the vocabulary
constexpr int kBNGrad = 256;    // dH^T / dW: N tile

// One GEMM problem of a launch: C[M, N] = sum_k A[m, k] B[n, k].
struct Problem {
  int m_blocks, n_blocks, k_blocks;
  int a_mn, b_mn;   // operand major-ness: 0 = K contiguous, 1 = M/N contiguous
  int M, N;         // valid extents (epilogue stores are clipped to them)
  int tile_begin;   // first global tile index of this problem
  int n_fastest;    // tile order: 1 = consecutive tiles walk N, 0 = walk M
  int reduce_add;   // fp32 epilogue: 1 = TMA reduce-add into C, 0 = store
  int c_trans;      // fp32 epilogue: 1 = write C^T (TMEM lanes are C's columns)
  int out_bf16;     // transposed epilogue: 1 = C is bf16 (64-byte boxes, no swizzle), 0 = fp32
  int bnh;          // wide pair tiles: N of one MMA instruction, the width of each of the
                    // tile's two halves. 256 (0 means 256), or 240 for 480-wide tiles
                    // (plain fp32 C only; the last 16 columns of a half use tmCt)
};

// Kernel parameters (passed as __grid_constant__; tensor maps live in param space).
struct GemmArgs {
  CUtensorMap tmA[2];
  CUtensorMap tmB[2];
  CUtensorMap tmC[2];
  CUtensorMap tmCt[2];    // C with 16-column boxes (no swizzle), for halves 240 wide
  Problem pr[2];
  int nprob;
  int total_tiles;
  int* tile_counter;      // dynamic tile scheduler (zeroed before each launch)
  // fused-epilogue data (chunk-local rows)
  int rows;               // rows of this chunk
  int S;                  // vocabulary tiles: row stride of the [chunk][S] partials
  int V;
  int Kp;                 // row stride of the sorted id / p / zK arrays
  const int* ids_sorted;  // [chunk][Kp], ascending, padded
  const float* p_sorted;  // [chunk][Kp]
  const int* cnt;         // [chunk] entries per row
  float* zK;              // [chunk][Kp] student logit at each sorted id
  float* part_m;          // [chunk][S] per-(row, vocab tile) max
  float* part_s;          // [chunk][S] per-(row, vocab tile) sum exp(z - max)
  const float* lse;       // [rows] chunk slice of the saved log-sum-exp
  float scale;            // dz scale
  const float* dscale;    // optional device multiplier of `scale`
  float zscale;           // logit scale 1/tau (temperature) in the loss epilogues; 1 = none
  const uint8_t* mask;    // [rows] chunk slice of the position mask (0 = excluded), or null
  int* status;            // device status word
  int cta2;               // 1: cluster-pair tiles (256 rows, tcgen05 cta_group::2)
  int wide;               // with cta2: 1 = 256 x 512 tiles, 0 = 256 x 256
};

// Rows of one GEMM tile (M extent) for the chosen tile shape; with cta2 the B
// operand's tensor map box is 128 rows (each CTA of the pair loads one such
// box per K step, two for wide tiles: one per 256-column half).
inline int gemm_tile_rows(int cta2) { return cta2 ? 2 * kBM : kBM; }
inline int gemm_b_box_rows(int cta2) { return cta2 ? kBNLogits / 2 : kBNLogits; }
// Columns of one GEMM tile (N extent): 512 for wide CTA-pair tiles, 256
// otherwise. Per-vocabulary-tile partials stay per 256 columns either way.
inline int gemm_tile_cols(int cta2, int wide) { return (cta2 && wide) ? 2 * kBNLogits : kBNLogits; }

cudaError_t encode_map_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
                          uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer);
// Same, without shared-memory swizzle (box rows land densely in smem).
cudaError_t encode_map_2d_plain(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
                                uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer);

// Launchers (kd_gemm.cu).
cudaError_t launch_logits_fwd(const GemmArgs& a, int num_sms, cudaStream_t s);
cudaError_t launch_logits_dz(const GemmArgs& a, int num_sms, cudaStream_t s);
cudaError_t launch_logits_fwd_store(const GemmArgs& a, int num_sms, cudaStream_t s);
cudaError_t launch_logits_teacher(const GemmArgs& a, int num_sms, cudaStream_t s);
cudaError_t launch_grad(const GemmArgs& a, int num_sms, cudaStream_t s);

// Small kernels (kd_loss_aux.cu).
cudaError_t launch_prep(const int32_t* ids, const float* logp, int rows, int K, int V, int Kp, float inv_tau,
                        int* ids_sorted, float* p_sorted, int* cnt, float* ent, int* status, cudaStream_t s);
cudaError_t launch_merge(const float* part_m, const float* part_s, int S, int rows, const float* ent,
                         const float* p_sorted, const float* zK, const int* cnt, int Kp, const uint8_t* mask,
                         float* lse_out, float* loss_rows_out, double* block_sums, unsigned* done, double* acc,
                         int first, cudaStream_t s);
// Per-position gradient factor s = grad_scale * (*grad_scale_dev, if any) *
// inv_tau * (mean_over_mask ? 1/N : 1), N = positions with mask != 0 (0 if
// N = 0), written to *out on the device.
cudaError_t launch_grad_scale(float grad_scale, const float* grad_scale_dev, float inv_tau, const uint8_t* mask,
                              int64_t T, int mean_over_mask, float* out, cudaStream_t s);
cudaError_t launch_dz_from_exp(__nv_bfloat16* E, int64_t ldz, int V, int S, int rows, const float* part_m,
                               const float* lse, const int* ids_sorted, const float* p_sorted, const float* zK,
                               const int* cnt, int Kp, float scale, const float* dscale, const uint8_t* mask,
                               cudaStream_t s);
// loss = acc / T, or acc / N over the mask's included positions when
// mean_over_mask (0 when N = 0).
cudaError_t launch_finalize(const double* acc, int64_t T, const uint8_t* mask, int mean_over_mask, float* loss,
                            cudaStream_t s);
cudaError_t launch_transpose(const void* src, int rows, int cols, void* dst, int ld_dst, cudaStream_t s);
cudaError_t launch_wait_timeout(uint64_t limit_ns, int* status, cudaStream_t s);

// Argument checks of kd_topk_cache apart from its workspace (kd_api.cu);
// returns a kd_status value.
int topk_check_args(const void* logits, int dtype, int64_t T, int64_t V, int64_t ld, int K, const void* ids,
                    const void* logp);

// Top-K (kd_topk.cu).
size_t topk_smem_bytes(int K);
cudaError_t launch_topk(const void* logits, int dtype, int64_t T, int64_t V, int64_t ld, int K, int32_t* ids,
                        float* logp, int* ws_words, int force_exact, int num_sms, cudaStream_t stream);
size_t tile_topk_smem_bytes(int K);
cudaError_t launch_tile_topk(const float* Z, int64_t ldz, int rows, int V, int S, const float* part_m,
                             const float* part_s, int K, int32_t* ids, float* logp, int* ws_words, int force_exact,
                             cudaStream_t stream);

}  // namespace kd
