// kd_topk.cu - offline teacher cache: logits [T, V] -> top-K ids + log-softmax.
//
// The cache step of the offline distillation ("ทำให้ Knowledge Distillation มี
// ประสิทธิภาพ..." (ai-thai.com), section "การทำ Distillation แบบ Offline": the
// teacher runs once and only its K most probable tokens per position are
// kept). Selection order: value descending, then id ascending; -0.0 == +0.0.
//
// One CTA streams one row from HBM exactly once with 16-byte loads. In that
// single pass it computes
//   * the row's log-sum-exp: an online (max, sum of exp) per thread, merged in
//     a fixed order, so the result is deterministic;
//   * the top-K candidates: each thread keeps its own best 8 (value, id)
//     pairs in registers. A vector of 8 logits is skipped with one compare
//     when its maximum is below the thread's 8th best.
// The 256 x 8 candidates are sorted in shared memory and the first K taken.
// This is exact unless some thread dropped an element that ranks at or above
// the K-th pick. Each thread tracks the best element it dropped, so that case
// is detected, and then (or when K > 2048) the row is redone by an exact
// radix selection over the row in global memory (L2-resident by then).
#include <cstdint>
#include <cuda_runtime.h>

#include "kd_internal.h"
#include "kd_ptx.cuh"

namespace kd {
namespace {

constexpr int kThreads = 256;
constexpr int kList = 8;                      // per-thread candidate list
constexpr int kUnion = kThreads * kList;      // 2048 candidates per row
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Order-preserving map float -> uint32 (larger float -> larger key), with
// -0.0 mapped to the key of +0.0.
__device__ __forceinline__ uint32_t okey(float x) {
  uint32_t b = __float_as_uint(x);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float okey_to_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
// Rank key: larger = earlier in the output (value desc, then id asc).
__device__ __forceinline__ uint64_t rkey(float x, uint32_t id) {
  return ((uint64_t)okey(x) << 32) | (uint64_t)(0xFFFFFFFFu - id);
}

template <typename Tin>
struct Row;
template <>
struct Row<uint16_t> {  // bf16
  static constexpr int kVec = 8;
  __device__ static __forceinline__ float cvt(uint16_t v) { return __uint_as_float((uint32_t)v << 16); }
  __device__ static __forceinline__ void unpack(const uint4& u, float (&x)[8]) {
    x[0] = __uint_as_float(u.x << 16); x[1] = __uint_as_float(u.x & 0xFFFF0000u);
    x[2] = __uint_as_float(u.y << 16); x[3] = __uint_as_float(u.y & 0xFFFF0000u);
    x[4] = __uint_as_float(u.z << 16); x[5] = __uint_as_float(u.z & 0xFFFF0000u);
    x[6] = __uint_as_float(u.w << 16); x[7] = __uint_as_float(u.w & 0xFFFF0000u);
  }
};
template <>
struct Row<float> {
  static constexpr int kVec = 4;
  __device__ static __forceinline__ float cvt(float v) { return v; }
  __device__ static __forceinline__ void unpack(const uint4& u, float (&x)[4]) {
    x[0] = __uint_as_float(u.x); x[1] = __uint_as_float(u.y);
    x[2] = __uint_as_float(u.z); x[3] = __uint_as_float(u.w);
  }
};

// Per-thread state of the streaming pass.
struct Scan {
  float m, s;            // online log-sum-exp: max and sum of exp(x - m)
  uint64_t L[kList];     // best 8 rank keys, descending; 0 = empty
  float thr;             // value of L[7] (-inf while the list is not full)
  uint64_t drop;         // best rank key this thread dropped (exact)
  float drop_v;          // best value dropped by the one-compare skip
  __device__ void init() {
    m = -INFINITY; s = 0.f; thr = -INFINITY; drop = 0; drop_v = -INFINITY;
#pragma unroll
    for (int j = 0; j < kList; ++j) L[j] = 0;
  }
  __device__ __forceinline__ void lse_max(float vmax) {
    if (vmax > m) {
      s *= ex2((m - vmax) * kLog2e);
      m = vmax;
    }
  }
  __device__ __forceinline__ void offer(float x, uint32_t id) {
    const uint64_t k = rkey(x, id);
    if (k > L[kList - 1]) {
      if (L[kList - 1] > drop) drop = L[kList - 1];
      L[kList - 1] = k;
#pragma unroll
      for (int j = kList - 1; j > 0; --j) {
        const uint64_t a = L[j - 1], b = L[j];
        const bool sw = b > a;
        L[j - 1] = sw ? b : a;
        L[j] = sw ? a : b;
      }
      thr = L[kList - 1] ? okey_to_float((uint32_t)(L[kList - 1] >> 32)) : -INFINITY;
    } else if (k > drop) {
      drop = k;
    }
  }
  template <int N>
  __device__ __forceinline__ void vec(const float (&x)[N], uint32_t id0) {
    float vmax = x[0];
#pragma unroll
    for (int j = 1; j < N; ++j) vmax = fmaxf(vmax, x[j]);
    lse_max(vmax);
    const float mb = -m * kLog2e;
#pragma unroll
    for (int j = 0; j < N; ++j) s += ex2(fmaf(x[j], kLog2e, mb));
    if (vmax < thr) {
      drop_v = fmaxf(drop_v, vmax);
    } else {
#pragma unroll
      for (int j = 0; j < N; ++j) offer(x[j], id0 + j);
    }
  }
  __device__ __forceinline__ void one(float x, uint32_t id) {
    lse_max(x);
    s += ex2((x - m) * kLog2e);
    offer(x, id);
  }
};

// Combine two (max, sum) pairs of the online log-sum-exp. Commutative, so
// the xor-shuffle tree leaves the same value in every lane.
__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) { m = m2; s = s2; return; }
  const float mm = fmaxf(m, m2);
  s = s * ex2((m - mm) * kLog2e) + s2 * ex2((m2 - mm) * kLog2e);
  m = mm;
}

// Descending bitonic sort of n (power of two) 64-bit keys in shared memory.
__device__ void bitonic_desc(uint64_t* a, int n) {
  for (int k = 2; k <= n; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int p = i ^ j;
        if (p > i) {
          const uint64_t x = a[i], y = a[p];
          const bool desc = (i & k) == 0;
          if (desc ? (x < y) : (x > y)) { a[i] = y; a[p] = x; }
        }
      }
      __syncthreads();
    }
  }
}

// Block-wide exclusive scan of one int per thread. Returns the prefix and
// writes the total to *total.
__device__ int block_excl_scan(int v, int* sm_warp, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) sm_warp[w] = inc;
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int i = 0; i < kThreads / 32; ++i) { const int t = sm_warp[i]; sm_warp[i] = acc; acc += t; }
    sm_warp[kThreads / 32] = acc;
  }
  __syncthreads();
  const int r = sm_warp[w] + inc - v;
  *total = sm_warp[kThreads / 32];
  __syncthreads();
  return r;
}

template <typename Tin>
__device__ __forceinline__ float load_elem(const Tin* row, int64_t j) {
  return Row<Tin>::cvt(row[j]);
}

// Exact top-K by radix selection on the order keys, reading the row from
// global memory. Writes the K rank keys, sorted descending, to cand[0..K).
template <typename Tin>
__device__ void exact_select(const Tin* row, int V, int K, uint64_t* cand, int n_pow2, uint32_t* hist,
                             int* sm_scan, int* sm_misc) {
  const int tid = threadIdx.x;
  uint32_t prefix = 0, pmask = 0;
  int krem = K;
  const int last_shift = sizeof(Tin) == 2 ? 16 : 0;
  for (int shift = 24; shift >= last_shift; shift -= 8) {
    for (int i = tid; i < 256; i += kThreads) hist[i] = 0;
    __syncthreads();
    for (int j = tid; j < V; j += kThreads) {
      const uint32_t k = okey(load_elem(row, j));
      if ((k & pmask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid == 0) {
      int cum = 0, b = 255;
      for (; b > 0; --b) {
        if (cum + (int)hist[b] >= krem) break;
        cum += (int)hist[b];
      }
      sm_misc[0] = b;
      sm_misc[1] = krem - cum;
    }
    __syncthreads();
    prefix |= (uint32_t)sm_misc[0] << shift;
    pmask |= 0xFFu << shift;
    krem = sm_misc[1];
    __syncthreads();
  }
  if (sizeof(Tin) == 2) {
    // bf16 widened to fp32: the low 16 key bits follow from the sign.
    prefix |= (prefix & 0x80000000u) ? 0u : 0xFFFFu;
    pmask = 0xFFFFFFFFu;
  }
  const uint32_t kth = prefix;
  const int need_eq = krem;       // elements equal to kth to take, lowest ids first
  const int n_gt = K - need_eq;   // elements strictly above kth
  for (int i = tid; i < n_pow2; i += kThreads) cand[i] = 0;
  if (tid == 0) sm_misc[2] = 0;
  __syncthreads();
  for (int j = tid; j < V; j += kThreads) {
    const float x = load_elem(row, j);
    if (okey(x) > kth) {
      const int slot = atomicAdd(&sm_misc[2], 1);
      cand[slot] = rkey(x, (uint32_t)j);
    }
  }
  __syncthreads();
  // Equal elements in id order: 8 consecutive elements per thread per tile.
  int taken = 0;
  for (int base = 0; base < V && taken < need_eq; base += kThreads * 8) {
    const int j0 = base + tid * 8;
    int c = 0;
    for (int q = 0; q < 8; ++q) {
      const int j = j0 + q;
      if (j < V && okey(load_elem(row, j)) == kth) ++c;
    }
    int tot;
    int r = block_excl_scan(c, sm_scan, &tot);
    for (int q = 0; q < 8 && c > 0; ++q) {
      const int j = j0 + q;
      if (j < V) {
        const float x = load_elem(row, j);
        if (okey(x) == kth) {
          if (taken + r < need_eq) cand[n_gt + taken + r] = rkey(x, (uint32_t)j);
          ++r;
        }
      }
    }
    taken += tot;  // block-uniform
  }
  __syncthreads();
  bitonic_desc(cand, n_pow2);
}

template <typename Tin>
__global__ void __launch_bounds__(kThreads) topk_kernel(const Tin* __restrict__ logits, int64_t T, int V,
                                                        int64_t ld, int K, int cand_n, int force_exact,
                                                        int32_t* __restrict__ ids, float* __restrict__ logp,
                                                        int* __restrict__ ws_words) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint64_t* cand = reinterpret_cast<uint64_t*>(smem_raw);
  __shared__ uint32_t hist[256];
  __shared__ int sm_scan[kThreads / 32 + 1];
  __shared__ int sm_misc[4];
  __shared__ float sm_m[kThreads / 32], sm_s[kThreads / 32];
  __shared__ float sm_lse;
  __shared__ int sm_ok;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int VEC = Row<Tin>::kVec;

  for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
    const Tin* row = logits + t * ld;
    Scan st;
    st.init();
    // Head elements up to the first 16-byte boundary, then 16-byte vectors,
    // then the tail.
    const uintptr_t addr = reinterpret_cast<uintptr_t>(row);
    int head = (int)(((16u - (addr & 15u)) & 15u) / sizeof(Tin));
    if (head > V) head = V;
    const int nvec = (V - head) / VEC;
    const int tail0 = head + nvec * VEC;
    if (tid < head) st.one(Row<Tin>::cvt(row[tid]), (uint32_t)tid);
    if (tid < V - tail0) st.one(Row<Tin>::cvt(row[tail0 + tid]), (uint32_t)(tail0 + tid));
    const uint4* vrow = reinterpret_cast<const uint4*>(row + head);
    int i = tid;
    for (; i + 3 * kThreads < nvec; i += 4 * kThreads) {
      uint4 u[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) u[q] = __ldcs(vrow + i + q * kThreads);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float x[VEC];
        Row<Tin>::unpack(u[q], x);
        st.vec(x, (uint32_t)(head + (i + q * kThreads) * VEC));
      }
    }
    for (; i < nvec; i += kThreads) {
      const uint4 u = __ldcs(vrow + i);
      float x[VEC];
      Row<Tin>::unpack(u, x);
      st.vec(x, (uint32_t)(head + i * VEC));
    }

    // Row log-sum-exp, merged in a fixed order.
    float m = st.m, s = st.s;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
      lse_merge(m, s, m2, s2);
    }
    if (lane == 0) { sm_m[warp] = m; sm_s[warp] = s; }

    // Candidate union.
    bool exact = force_exact || K > kUnion;
    if (!exact) {
#pragma unroll
      for (int j = 0; j < kList; ++j) cand[tid * kList + j] = st.L[j];
    }
    __syncthreads();
    if (tid == 0) {
      float M = sm_m[0], S = sm_s[0];
      for (int w = 1; w < kThreads / 32; ++w) lse_merge(M, S, sm_m[w], sm_s[w]);
      sm_lse = M + logf(S);
    }
    if (!exact) {
      bitonic_desc(cand, kUnion);
      const uint64_t eK = cand[K - 1];
      const float eKv = okey_to_float((uint32_t)(eK >> 32));
      const bool ok = eK != 0 && st.drop < eK && st.drop_v < eKv;
      exact = !__syncthreads_and(ok);
    }
    if (exact) {
      if (tid == 0 && !force_exact && ws_words) atomicAdd(&ws_words[1], 1);
      __syncthreads();
      exact_select<Tin>(row, V, K, cand, cand_n, hist, sm_scan, sm_misc);
    }
    __syncthreads();
    const float lse = sm_lse;
    for (int k = tid; k < K; k += kThreads) {
      const uint64_t c = cand[k];
      ids[t * K + k] = (int32_t)(0xFFFFFFFFu - (uint32_t)c);
      logp[t * K + k] = okey_to_float((uint32_t)(c >> 32)) - lse;
    }
    __syncthreads();
  }
  (void)sm_ok;
}

}  // namespace

size_t topk_smem_bytes(int K) {
  int n = 1;
  while (n < K) n <<= 1;
  if (n < kUnion) n = kUnion;
  return (size_t)n * sizeof(uint64_t);
}

cudaError_t launch_topk(const void* logits, int dtype, int64_t T, int64_t V, int64_t ld, int K,
                        int32_t* ids, float* logp, int* ws_words, int force_exact, int num_sms,
                        cudaStream_t stream) {
  int n = 1;
  while (n < K) n <<= 1;
  if (n < kUnion) n = kUnion;
  const size_t smem = (size_t)n * sizeof(uint64_t);
  int blocks_per_sm = 0;
  cudaError_t e;
  if (dtype == 0) {
    e = cudaFuncSetAttribute(topk_kernel<uint16_t>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks_per_sm, topk_kernel<uint16_t>, kThreads, smem);
  } else {
    e = cudaFuncSetAttribute(topk_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks_per_sm, topk_kernel<float>, kThreads, smem);
  }
  if (e != cudaSuccess) return e;
  if (blocks_per_sm < 1) blocks_per_sm = 1;
  int64_t grid = (int64_t)num_sms * blocks_per_sm;
  if (grid > T) grid = T;
  if (dtype == 0)
    topk_kernel<uint16_t><<<(unsigned)grid, kThreads, smem, stream>>>(
        static_cast<const uint16_t*>(logits), T, (int)V, ld, K, n, force_exact, ids, logp, ws_words);
  else
    topk_kernel<float><<<(unsigned)grid, kThreads, smem, stream>>>(
        static_cast<const float*>(logits), T, (int)V, ld, K, n, force_exact, ids, logp, ws_words);
  return cudaGetLastError();
}

}  // namespace kd
