// kd_loss_aux.cu - the per-chunk steps of the fused KL loss that are not GEMMs.
//
//  prep    teacher side of the loss for one chunk: p = softmax over the K
//          cached log-probs (renormalised over K), the entropy term
//          sum_k p log p, and the (id, p) list sorted by id with duplicates
//          summed, so that the GEMM epilogues can find the ids inside each
//          vocabulary tile.
//  merge   per position: log-sum-exp over the whole vocabulary from the
//          per-tile (max, sum) partials of the forward GEMM; the loss
//          L_t = sum p log p - sum_k p_k z_id_k + lse_t; a per-block sum.
//          The last block of a chunk adds the chunk's block sums to the
//          running fp64 total in a fixed order; finally loss = total / T.
//  dz      (single-call forward + backward) dz = s (q - p 1[j in K]) from
//          the forward GEMM's stored e = exp(z - m_tile) in bf16:
//          q_j = e_j exp(m_tile - lse) off the K ids; at the K ids q comes
//          from the fp32 logit the forward gathered, so q - p is formed
//          from unrounded values exactly as in the recompute path.
// All reductions run in a fixed order, so the loss is bitwise reproducible.
// Definition: "ทำให้ Knowledge Distillation มีประสิทธิภาพ..." (ai-thai.com),
// section "กลไก Fused Chunked KL Loss". The page states no formula: the KL
// direction (teacher to student), the renormalisation of the teacher over K
// and the mean over positions are the readings its text supports.
#include <cstdint>
#include <cuda_runtime.h>

#include "kd_internal.h"
#include "kd_ptx.cuh"

namespace kd {
namespace {

constexpr int kPrepThreads = 128;
constexpr uint64_t kDropKey = ~0ull;

__device__ float block_reduce_max(float v, float* sm) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if (lane == 0) sm[w] = v;
  __syncthreads();
  float r = sm[0];
  for (int i = 1; i < (int)(blockDim.x >> 5); ++i) r = fmaxf(r, sm[i]);
  __syncthreads();
  return r;
}

// Sum in a fixed order: per-thread strided partial, xor tree, warps in order.
__device__ float block_reduce_sum(float v, float* sm) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) sm[w] = v;
  __syncthreads();
  float r = sm[0];
  for (int i = 1; i < (int)(blockDim.x >> 5); ++i) r += sm[i];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kPrepThreads) prep_kernel(const int32_t* __restrict__ ids,
                                                            const float* __restrict__ logp, int K, int V,
                                                            int Kp, int Kpow2, float inv_tau,
                                                            int* __restrict__ ids_sorted,
                                                            float* __restrict__ p_sorted, int* __restrict__ cnt,
                                                            float* __restrict__ ent, int* status) {
  extern __shared__ uint64_t keys[];  // [Kpow2]
  __shared__ float red[kPrepThreads / 32];
  __shared__ int scan_w[kPrepThreads / 32 + 1];
  const int r = blockIdx.x, tid = threadIdx.x;
  const int32_t* rid = ids + (size_t)r * K;
  const float* rl = logp + (size_t)r * K;

  // Teacher (log-probs divided by the temperature) renormalised over its K
  // entries.
  float mx = -INFINITY;
  for (int k = tid; k < K; k += kPrepThreads) mx = fmaxf(mx, rl[k] * inv_tau);
  mx = block_reduce_max(mx, red);
  float se = 0.f;
  for (int k = tid; k < K; k += kPrepThreads) se += expf(rl[k] * inv_tau - mx);
  se = block_reduce_sum(se, red);
  const float lse_k = mx + logf(se);
  float e = 0.f;
  for (int k = tid; k < K; k += kPrepThreads) {
    const float lp = rl[k] * inv_tau - lse_k;
    e += expf(lp) * lp;
  }
  e = block_reduce_sum(e, red);
  if (tid == 0) ent[r] = e;

  // Sort (id, original slot) by id; bad ids sort last and are dropped.
  bool bad = false;
  for (int i = tid; i < Kpow2; i += kPrepThreads) {
    uint64_t key = kDropKey;
    if (i < K) {
      const int id = rid[i];
      if (id < 0 || id >= V) bad = true;
      else key = ((uint64_t)(uint32_t)id << 32) | (uint32_t)i;
    }
    keys[i] = key;
  }
  if (bad) set_status(status, ST_BAD_ID);
  __syncthreads();
  for (int k = 2; k <= Kpow2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < Kpow2; i += kPrepThreads) {
        const int p = i ^ j;
        if (p > i) {
          const uint64_t a = keys[i], b = keys[p];
          const bool up = (i & k) == 0;
          if (up ? (a > b) : (a < b)) { keys[i] = b; keys[p] = a; }
        }
      }
      __syncthreads();
    }
  }

  // Compact runs of equal ids: one output entry per distinct id with the
  // summed probability (the scatter-add of duplicates).
  int base_out = 0;
  for (int base = 0; base < Kpow2; base += kPrepThreads) {
    const int i = base + tid;
    const uint64_t key = keys[i];
    const bool valid = key != kDropKey;
    const uint32_t id = (uint32_t)(key >> 32);
    const bool head = valid && (i == 0 || (uint32_t)(keys[i - 1] >> 32) != id || keys[i - 1] == kDropKey);
    const int lane = tid & 31, w = tid >> 5;
    const unsigned bal = __ballot_sync(0xffffffffu, head);
    if (lane == 0) scan_w[w] = __popc(bal);
    __syncthreads();
    if (tid == 0) {
      int acc = 0;
      for (int q = 0; q < kPrepThreads / 32; ++q) { const int t = scan_w[q]; scan_w[q] = acc; acc += t; }
      scan_w[kPrepThreads / 32] = acc;
    }
    __syncthreads();
    if (head) {
      const int slot = base_out + scan_w[w] + __popc(bal & ((1u << lane) - 1u));
      float ps = 0.f;
      for (int j = i; j < Kpow2 && keys[j] != kDropKey && (uint32_t)(keys[j] >> 32) == id; ++j)
        ps += expf(rl[(uint32_t)keys[j]] * inv_tau - lse_k);
      ids_sorted[(size_t)r * Kp + slot] = (int)id;
      p_sorted[(size_t)r * Kp + slot] = ps;
    }
    base_out += scan_w[kPrepThreads / 32];
    __syncthreads();
  }
  if (tid == 0) cnt[r] = base_out;
}

// The same teacher prep with one warp per row, for K <= 128 (the cache
// sizes of the method: K = 100). Each lane holds 4 of the row's entries;
// the (id, slot) keys are sorted by a 128-element bitonic network in
// registers and shuffles (sort position = 4 * lane + q), so no block-wide
// barrier is involved and a launch takes about one row's latency.
constexpr int kPrepWarpK = 128;
constexpr int kPrepWarpRows = 8;  // rows (warps) per block

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__global__ void __launch_bounds__(32 * kPrepWarpRows) prep_warp_kernel(
    const int32_t* __restrict__ ids, const float* __restrict__ logp, int rows, int K, int V, int Kp, float inv_tau,
    int* __restrict__ ids_sorted, float* __restrict__ p_sorted, int* __restrict__ cnt, float* __restrict__ ent,
    int* status) {
  __shared__ uint64_t skeys[kPrepWarpRows][kPrepWarpK];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * kPrepWarpRows + w;
  if (r >= rows) return;  // whole warps only; nothing below synchronises the block
  const int32_t* rid = ids + (size_t)r * K;
  const float* rl = logp + (size_t)r * K;

  float lv[4];
  uint64_t key[4];
  bool bad = false;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int i = lane + 32 * q;  // original slot of this register
    lv[q] = -INFINITY;
    key[q] = kDropKey;
    if (i < K) {
      lv[q] = __ldg(rl + i) * inv_tau;
      const int id = __ldg(rid + i);
      if (id < 0 || id >= V) bad = true;
      else key[q] = ((uint64_t)(uint32_t)id << 32) | (uint32_t)i;
    }
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) set_status(status, ST_BAD_ID);

  // Teacher renormalised over its K entries, and sum p log p.
  float mx = -INFINITY;
#pragma unroll
  for (int q = 0; q < 4; ++q) mx = fmaxf(mx, lv[q]);
  mx = warp_max(mx);
  float se = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q) if (lane + 32 * q < K) se += expf(lv[q] - mx);
  se = warp_sum(se);
  const float lse_k = mx + logf(se);
  float e = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (lane + 32 * q < K) {
      const float lp = lv[q] - lse_k;
      e += expf(lp) * lp;
    }
  }
  e = warp_sum(e);
  if (lane == 0) ent[r] = e;

  // Ascending bitonic sort of the 128 keys; position 4 * lane + q.
#pragma unroll
  for (int k = 2; k <= kPrepWarpK; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j >= 4) {
        const int lj = j >> 2;
        const bool lower = (lane & lj) == 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint64_t o = __shfl_xor_sync(0xffffffffu, key[q], lj);
          const bool up = (((lane << 2) | q) & k) == 0;
          const uint64_t lo = key[q] < o ? key[q] : o, hi = key[q] < o ? o : key[q];
          key[q] = (lower == up) ? lo : hi;
        }
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (q & j) continue;
          const int p = q | j;
          const bool up = (((lane << 2) | q) & k) == 0;
          const uint64_t a = key[q], b = key[p];
          if (up ? (a > b) : (a < b)) { key[q] = b; key[p] = a; }
        }
      }
    }
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) skeys[w][(lane << 2) | q] = key[q];
  __syncwarp();

  // One output entry per distinct id (a run of equal ids), with the summed
  // probability (the scatter-add of duplicates); slots in id order.
  bool head[4];
  int hc = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int pos = (lane << 2) | q;
    const uint64_t kq = key[q];
    head[q] = kq != kDropKey &&
              (pos == 0 || skeys[w][pos - 1] == kDropKey || (uint32_t)(skeys[w][pos - 1] >> 32) != (uint32_t)(kq >> 32));
    hc += head[q] ? 1 : 0;
  }
  int incl = hc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  int slot = incl - hc;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (!head[q]) continue;
    const int pos = (lane << 2) | q;
    const uint32_t id = (uint32_t)(key[q] >> 32);
    float ps = 0.f;
    for (int j = pos; j < kPrepWarpK && skeys[w][j] != kDropKey && (uint32_t)(skeys[w][j] >> 32) == id; ++j)
      ps += expf(__ldg(rl + (uint32_t)skeys[w][j]) * inv_tau - lse_k);
    ids_sorted[(size_t)r * Kp + slot] = (int)id;
    p_sorted[(size_t)r * Kp + slot] = ps;
    ++slot;
  }
  if (lane == 31) cnt[r] = incl;
}

// One warp per position, 8 positions per block. Each lane takes every 32nd
// vocabulary-tile partial of the row (a coalesced read of the row's [S]
// partials), and the lanes are combined by xor-shuffle trees, after which
// every lane holds the same value. The block sum of its 8 losses is taken in
// a fixed order, so the result is deterministic.
__global__ void __launch_bounds__(256) merge_kernel(const float* __restrict__ part_m,
                                                    const float* __restrict__ part_s, int S, int rows,
                                                    const float* __restrict__ ent,
                                                    const float* __restrict__ p_sorted,
                                                    const float* __restrict__ zK, const int* __restrict__ cnt,
                                                    int Kp, const uint8_t* __restrict__ mask,
                                                    float* __restrict__ lse_out,
                                                    float* __restrict__ loss_rows_out,
                                                    double* __restrict__ block_sums, unsigned* done,
                                                    double* acc, int first) {
  __shared__ float sl[8];
  __shared__ bool last_block;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int row = blockIdx.x * 8 + w;
  float L = 0.f;
  if (row < rows) {
    const float* pm = part_m + (size_t)row * S;
    const float* ps = part_s + (size_t)row * S;
    // Two passes with independent loads (many in flight): the row maximum
    // M over the tile maxima, then sum_j s_j exp(m_j - M). Both in a fixed
    // order (per lane, then an xor tree), so the result is deterministic.
    float m = -INFINITY;
#pragma unroll 8
    for (int j = lane; j < S; j += 32) m = fmaxf(m, __ldg(pm + j));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float s = 0.f;
#pragma unroll 8
    for (int j = lane; j < S; j += 32) s += __ldg(ps + j) * expf(__ldg(pm + j) - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float lse = m + logf(s);
    const int c = cnt[row];
    float dot = 0.f;
    for (int k = lane; k < c; k += 32) dot += p_sorted[(size_t)row * Kp + k] * zK[(size_t)row * Kp + k];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    L = ent[row] - dot + lse;
    if (mask && mask[row] == 0) L = 0.f;  // excluded position
    if (lane == 0) {
      lse_out[row] = lse;
      if (loss_rows_out) loss_rows_out[row] = L;
    }
  }
  if (lane == 0) sl[w] = L;
  __syncthreads();
  if (tid == 0) {
    double a = 0.0;
    for (int i = 0; i < 8; ++i) a += (double)sl[i];
    block_sums[blockIdx.x] = a;
    __threadfence();
    last_block = atomicAdd(done, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  // The last block to finish adds the chunk's block sums to the running total,
  // in block order (lanes take contiguous runs, then a fixed shuffle tree).
  if (last_block && w == 0) {
    __threadfence();
    const int nb = gridDim.x, per = (nb + 31) / 32;
    double a = 0.0;
    for (int i = lane * per; i < (lane + 1) * per && i < nb; ++i)
      a += *reinterpret_cast<volatile double*>(&block_sums[i]);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double b = __shfl_down_sync(0xffffffffu, a, o);
      if ((lane & (2 * o - 1)) == 0) a += b;
    }
    if (lane == 0) {
      *acc = first ? a : (*acc + a);
      *done = 0u;  // ready for the next chunk
    }
  }
}

// loss = acc / T, or acc / N (N = included positions, counted here in a
// fixed order) when mean_over_mask.
__global__ void __launch_bounds__(256) finalize_kernel(const double* acc, int64_t T, const uint8_t* mask,
                                                       int mean_over_mask, float* loss) {
  __shared__ long long part[8];
  if (!(mask && mean_over_mask)) {
    if (threadIdx.x == 0) *loss = (float)(*acc / (double)T);
    return;
  }
  long long n = 0;
  for (int64_t t = threadIdx.x; t < T; t += blockDim.x) n += mask[t] != 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = n;
  __syncthreads();
  if (threadIdx.x == 0) {
    long long tot = 0;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) tot += part[i];
    *loss = tot > 0 ? (float)(*acc / (double)tot) : 0.f;
  }
}

// The backward's per-position gradient factor (see launch_grad_scale).
__global__ void __launch_bounds__(256) grad_scale_kernel(float grad_scale, const float* grad_scale_dev,
                                                         float inv_tau, const uint8_t* mask, int64_t T,
                                                         int mean_over_mask, float* out) {
  __shared__ long long part[8];
  long long n = 0;
  if (mask && mean_over_mask)
    for (int64_t t = threadIdx.x; t < T; t += blockDim.x) n += mask[t] != 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = n;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = grad_scale * (grad_scale_dev ? *grad_scale_dev : 1.f) * inv_tau;
    if (mask && mean_over_mask) {
      long long tot = 0;
      for (int i = 0; i < (int)(blockDim.x >> 5); ++i) tot += part[i];
      s = tot > 0 ? s / (float)tot : 0.f;
    }
    *out = s;
  }
}

// dst[c][r] = src[r][c] for a bf16 [rows, cols] matrix (dst row stride
// ld_dst): 32 x 32 tiles through shared memory.
__global__ void __launch_bounds__(256) transpose_kernel(const uint16_t* __restrict__ src, int rows, int cols,
                                                        uint16_t* __restrict__ dst, int ld_dst) {
  __shared__ uint16_t tile[32][34];
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  for (int j = ty; j < 32; j += 8) {
    const int r = r0 + j, c = c0 + tx;
    if (r < rows && c < cols) tile[j][tx] = src[(size_t)r * cols + c];
  }
  __syncthreads();
  for (int j = ty; j < 32; j += 8) {
    const int c = c0 + j, r = r0 + tx;
    if (c < cols && r < rows) dst[(size_t)c * ld_dst + r] = tile[tx][j];
  }
}

// Waits on an mbarrier that nothing arrives at, with a time limit, and
// records the timeout in the status word: the failure path every pipeline
// wait takes, exercised on purpose.
__global__ void wait_timeout_kernel(uint64_t limit_ns, int* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait_for(&bar, 0u, limit_ns)) set_status(status, ST_TIMEOUT);
  }
}

// One block per position, streaming its row of e in 16-byte vectors and
// rewriting it in place as dz (bf16), then the row's K entries.
constexpr int kDzThreads = 256;

__device__ __forceinline__ uint32_t scale_bf16x2(uint32_t u, float f) {
  const float lo = __uint_as_float(u << 16) * f;
  const float hi = __uint_as_float(u & 0xFFFF0000u) * f;
  return pack_bf16x2(lo, hi);
}

__global__ void __launch_bounds__(kDzThreads) dz_from_exp_kernel(uint16_t* __restrict__ E, int64_t ldz, int V, int S,
                                                                const float* __restrict__ part_m,
                                                                const float* __restrict__ lse,
                                                                const int* __restrict__ ids_sorted,
                                                                const float* __restrict__ p_sorted,
                                                                const float* __restrict__ zK,
                                                                const int* __restrict__ cnt, int Kp, float scale,
                                                                const float* __restrict__ dscale,
                                                                const uint8_t* __restrict__ mask) {
  const int r = blockIdx.x;
  const float sc = scale * (dscale ? __ldg(dscale) : 1.f) * ((mask && mask[r] == 0) ? 0.f : 1.f);
  const float l2 = __ldg(lse + r) * kLog2e;
  uint16_t* row = E + (size_t)r * ldz;
  const float* pm = part_m + (size_t)r * S;
  uint4* rv = reinterpret_cast<uint4*>(row);
  const int nvec = V >> 3;  // 8 columns per vector, never straddling a 256-column tile
  for (int v = threadIdx.x; v < nvec; v += kDzThreads) {
    const float f = sc * ex2(fmaf(__ldg(pm + ((v << 3) / kBNLogits)), kLog2e, -l2));
    uint4 x = rv[v];
    x.x = scale_bf16x2(x.x, f);
    x.y = scale_bf16x2(x.y, f);
    x.z = scale_bf16x2(x.z, f);
    x.w = scale_bf16x2(x.w, f);
    rv[v] = x;
  }
  for (int j = (nvec << 3) + threadIdx.x; j < V; j += kDzThreads) {
    const float f = sc * ex2(fmaf(__ldg(pm + j / kBNLogits), kLog2e, -l2));
    const __nv_bfloat16 h = __float2bfloat16_rn(__uint_as_float((uint32_t)row[j] << 16) * f);
    row[j] = *reinterpret_cast<const uint16_t*>(&h);
  }
  __syncthreads();  // the row's bulk writes land before its K entries are overwritten
  const int c = __ldg(cnt + r);
  for (int k = threadIdx.x; k < c; k += kDzThreads) {
    const size_t o = (size_t)r * Kp + k;
    const int j = __ldg(ids_sorted + o);
    const float q = ex2(fmaf(__ldg(zK + o), kLog2e, -l2));
    const __nv_bfloat16 h = __float2bfloat16_rn(sc * (q - __ldg(p_sorted + o)));
    row[j] = *reinterpret_cast<const uint16_t*>(&h);
  }
}

}  // namespace

cudaError_t launch_dz_from_exp(__nv_bfloat16* E, int64_t ldz, int V, int S, int rows, const float* part_m,
                               const float* lse, const int* ids_sorted, const float* p_sorted, const float* zK,
                               const int* cnt, int Kp, float scale, const float* dscale, const uint8_t* mask,
                               cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  dz_from_exp_kernel<<<rows, kDzThreads, 0, s>>>(reinterpret_cast<uint16_t*>(E), ldz, V, S, part_m, lse, ids_sorted,
                                                p_sorted, zK, cnt, Kp, scale, dscale, mask);
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout(uint64_t limit_ns, int* status, cudaStream_t s) {
  wait_timeout_kernel<<<1, 32, 0, s>>>(limit_ns, status);
  return cudaGetLastError();
}

cudaError_t launch_transpose(const void* src, int rows, int cols, void* dst, int ld_dst, cudaStream_t s) {
  dim3 grid((cols + 31) / 32, (rows + 31) / 32);
  transpose_kernel<<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(src), rows, cols, static_cast<uint16_t*>(dst),
                                        ld_dst);
  return cudaGetLastError();
}

cudaError_t launch_prep(const int32_t* ids, const float* logp, int rows, int K, int V, int Kp, float inv_tau,
                        int* ids_sorted, float* p_sorted, int* cnt, float* ent, int* status, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (K <= kPrepWarpK) {
    prep_warp_kernel<<<(rows + kPrepWarpRows - 1) / kPrepWarpRows, 32 * kPrepWarpRows, 0, s>>>(
        ids, logp, rows, K, V, Kp, inv_tau, ids_sorted, p_sorted, cnt, ent, status);
    return cudaGetLastError();
  }
  int Kpow2 = 1;
  while (Kpow2 < K) Kpow2 <<= 1;
  if (Kpow2 < kPrepThreads) Kpow2 = kPrepThreads;
  const size_t smem = (size_t)Kpow2 * sizeof(uint64_t);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  prep_kernel<<<rows, kPrepThreads, smem, s>>>(ids, logp, K, V, Kp, Kpow2, inv_tau, ids_sorted, p_sorted, cnt,
                                              ent, status);
  return cudaGetLastError();
}

cudaError_t launch_merge(const float* part_m, const float* part_s, int S, int rows, const float* ent,
                         const float* p_sorted, const float* zK, const int* cnt, int Kp, const uint8_t* mask,
                         float* lse_out, float* loss_rows_out, double* block_sums, unsigned* done, double* acc,
                         int first, cudaStream_t s) {
  const int nb = (rows + 7) / 8;
  merge_kernel<<<nb, 256, 0, s>>>(part_m, part_s, S, rows, ent, p_sorted, zK, cnt, Kp, mask, lse_out, loss_rows_out,
                                  block_sums, done, acc, first);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const double* acc, int64_t T, const uint8_t* mask, int mean_over_mask, float* loss,
                            cudaStream_t s) {
  finalize_kernel<<<1, 256, 0, s>>>(acc, T, mask, mean_over_mask, loss);
  return cudaGetLastError();
}

cudaError_t launch_grad_scale(float grad_scale, const float* grad_scale_dev, float inv_tau, const uint8_t* mask,
                              int64_t T, int mean_over_mask, float* out, cudaStream_t s) {
  grad_scale_kernel<<<1, 256, 0, s>>>(grad_scale, grad_scale_dev, inv_tau, mask, T, mean_over_mask, out);
  return cudaGetLastError();
}

}  // namespace kd
