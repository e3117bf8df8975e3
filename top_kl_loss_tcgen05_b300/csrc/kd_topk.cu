// kd_topk.cu - offline teacher cache: logits [T, V] -> top-K ids + log-softmax.
//
// The cache step of the offline distillation ("ทำให้ Knowledge Distillation มี
// ประสิทธิภาพ..." (ai-thai.com), section "การทำ Distillation แบบ Offline": the
// teacher runs once and only its K most probable tokens per position are
// kept). Selection order: value descending, then id ascending; -0.0 == +0.0.
//
// Persistent CTAs (five per SM) take rows from an atomic counter; per row:
//   pass 1  stream the row from HBM with 16-byte loads (6 per thread in
//           flight). Each thread keeps an online (max, sum of exp) of its
//           elements. That is the log-sum-exp, merged in a fixed order
//           (deterministic). A full batch takes its maximum first, with
//           packed bf16x2 max on the raw words, rescales the running sum
//           once, then adds its exps two at a time (fma.rn.f32x2 for the
//           arguments, add.rn.f32x2 into a two-lane sum): fewer instructions
//           per element, for a kernel that otherwise issues on about 70% of
//           cycles. The batch maxima also go to shared memory for pass 2.
//   tau     the K-th largest of the 256 per-thread maxima, found by a
//           bisection over the value keys (one __syncthreads_count per bit).
//           The maxima are K distinct elements >= tau, so tau is a lower
//           bound of the row's K-th largest value. On the pages' workload only
//           about 200 elements of a 201088-wide row are >= tau.
//   pass 2  each thread re-reads only its batches of 8 vectors whose maximum
//           (recorded in pass 1) is >= tau, about 6% of the row, and appends
//           every element >= tau to a shared buffer. The buffer holds every
//           top-K element, ties included.
//   select  sort the buffer by (value desc, id asc); its first K entries are
//           the cache row.
// If the buffer overflows (massive ties) or K > 1024, the row is redone by an
// exact radix selection over the row in global memory.
//
// tile_topk_kernel makes the same selection from the fp32 logits that the
// teacher GEMM wrote, using the per-(row, 256-column tile) maxima and sums
// of exp that the GEMM epilogue produced: the log-sum-exp is merged from
// them, tau is the K-th largest tile maximum (again K actual elements, so a
// lower bound of the K-th value), and only tiles whose maximum reaches tau
// are read: about K of the row's ceil(V/256) tiles.
#include <cstdint>
#include <cuda_runtime.h>

#include "kd_internal.h"
#include "kd_ptx.cuh"

namespace kd {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kCandCap = 2048;   // candidate buffer entries (fast path)
constexpr int kFastMaxK = 1024;  // larger K goes to the exact path
constexpr int kBatch = 6;        // 16-byte loads per thread in flight in pass 1
constexpr int kSlots = 16;       // per-thread batch-maximum slots kept for pass 2


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

// Split of a row into scalar head, 16-byte-aligned body and scalar tail.
template <typename Tin>
struct RowSplit {
  int head, nvec, tail0, tail;
  __device__ RowSplit(const Tin* row, int V) {
    const uintptr_t addr = reinterpret_cast<uintptr_t>(row);
    head = (int)(((16u - (addr & 15u)) & 15u) / sizeof(Tin));
    if (head > V) head = V;
    nvec = (V - head) / Row<Tin>::kVec;
    tail0 = head + nvec * Row<Tin>::kVec;
    tail = V - tail0;
  }
};

// Maximum of the elements of a full batch of 16-byte vectors. bf16: packed
// max.bf16x2 over the raw words, then the larger half (exact: the bf16 values
// widen to fp32 without rounding). fp32: fmaxf over the elements.
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
template <typename Tin, int N>
__device__ __forceinline__ float batch_max(const uint4 (&u)[N]) {
  if constexpr (sizeof(Tin) == 2) {
    uint32_t w = bf16x2_max(bf16x2_max(u[0].x, u[0].y), bf16x2_max(u[0].z, u[0].w));
#pragma unroll
    for (int q = 1; q < N; ++q)
      w = bf16x2_max(w, bf16x2_max(bf16x2_max(u[q].x, u[q].y), bf16x2_max(u[q].z, u[q].w)));
    return fmaxf(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  } else {
    float m = -INFINITY;
#pragma unroll
    for (int q = 0; q < N; ++q)
      m = fmaxf(fmaxf(m, fmaxf(__uint_as_float(u[q].x), __uint_as_float(u[q].y))),
                fmaxf(__uint_as_float(u[q].z), __uint_as_float(u[q].w)));
    return m;
  }
}

// Sum-of-exp step for one bf16x2 word w: acc (two fp32 lanes, packed in a
// 64-bit register) += (exp2(lo * c + mb), exp2(hi * c + mb)), with one
// fma.rn.f32x2 and one add.rn.f32x2 for the pair.
__device__ __forceinline__ void sumexp_bf16x2(uint64_t& acc, uint32_t w, uint64_t c2, uint64_t mb2) {
  asm("{.reg .b32 lo, hi, a, b;\n\t"
      ".reg .b64 x, r;\n\t"
      "shl.b32 lo, %1, 16;\n\t"
      "and.b32 hi, %1, 0xFFFF0000;\n\t"
      "mov.b64 x, {lo, hi};\n\t"
      "fma.rn.f32x2 r, x, %2, %3;\n\t"
      "mov.b64 {a, b}, r;\n\t"
      "ex2.approx.ftz.f32 a, a;\n\t"
      "ex2.approx.ftz.f32 b, b;\n\t"
      "mov.b64 r, {a, b};\n\t"
      "add.rn.f32x2 %0, %0, r;}"
      : "+l"(acc)
      : "r"(w), "l"(c2), "l"(mb2));
}
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  return ((uint64_t)__float_as_uint(hi) << 32) | (uint64_t)__float_as_uint(lo);
}

// Per-thread online log-sum-exp.
struct Lse {
  float m, s;  // max and sum of exp(x - m)
  __device__ __forceinline__ void init() { m = -INFINITY; s = 0.f; }
  __device__ __forceinline__ void max_to(float vmax) {
    if (vmax > m) {
      s *= ex2((m - vmax) * kLog2e);
      m = vmax;
    }
  }
  template <int N>
  __device__ __forceinline__ void add(const float (&x)[N], float vmax) {
    max_to(vmax);
    const float mb = -m * kLog2e;
#pragma unroll
    for (int j = 0; j < N; ++j) s += ex2(fmaf(x[j], kLog2e, mb));
  }
  // Sum only; the caller has already raised m to at least every element.
  template <int N>
  __device__ __forceinline__ void add_sum(const float (&x)[N], float mb) {
#pragma unroll
    for (int j = 0; j < N; ++j) s += ex2(fmaf(x[j], kLog2e, mb));
  }
  __device__ __forceinline__ void one(float x) {
    max_to(x);
    s += ex2((x - m) * kLog2e);
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
    for (int i = 0; i < kWarps; ++i) { const int t = sm_warp[i]; sm_warp[i] = acc; acc += t; }
    sm_warp[kWarps] = acc;
  }
  __syncthreads();
  const int r = sm_warp[w] + inc - v;
  *total = sm_warp[kWarps];
  __syncthreads();
  return r;
}

// Loads the 8 (bf16) or 4 (fp32) elements of body vector i of a row.
template <typename Tin>
__device__ __forceinline__ void load_vec(const Tin* row, const RowSplit<Tin>& rs, int i,
                                         float (&x)[Row<Tin>::kVec]) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(row + rs.head) + i);
  Row<Tin>::unpack(u, x);
}

// Exact top-K by radix selection on the order keys, reading the row from
// global memory (it is usually still in L2). Writes the K rank keys, sorted
// descending, to cand[0..K) (cand holds n_pow2 >= K entries).
template <typename Tin>
__device__ void exact_select(const Tin* row, int V, int K, uint64_t* cand, int n_pow2, uint32_t* hist,
                             int* sm_scan, int* sm_misc) {
  constexpr int VEC = Row<Tin>::kVec;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const RowSplit<Tin> rs(row, V);
  uint32_t prefix = 0, pmask = 0;
  int krem = K;
  const int last_shift = sizeof(Tin) == 2 ? 16 : 0;
  for (int shift = 24; shift >= last_shift; shift -= 8) {
    for (int i = tid; i < 256; i += kThreads) hist[i] = 0;
    __syncthreads();
    // scalar head and tail
    for (int j = tid; j < rs.head; j += kThreads) {
      const uint32_t k = okey(Row<Tin>::cvt(row[j]));
      if ((k & pmask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1u);
    }
    for (int j = tid; j < rs.tail; j += kThreads) {
      const uint32_t k = okey(Row<Tin>::cvt(row[rs.tail0 + j]));
      if ((k & pmask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1u);
    }
    // body: warp-uniform trip count, warp-aggregated increments
    for (int b = warp * 32; b < rs.nvec; b += kThreads) {
      const int i = b + lane;
      float x[VEC];
      if (i < rs.nvec) load_vec(row, rs, i, x);
#pragma unroll
      for (int j = 0; j < VEC; ++j) {
        uint32_t dig = 256u;
        if (i < rs.nvec) {
          const uint32_t k = okey(x[j]);
          if ((k & pmask) == prefix) dig = (k >> shift) & 255u;
        }
        const unsigned peers = __match_any_sync(0xffffffffu, dig);
        if (dig < 256u && lane == __ffs(peers) - 1) atomicAdd(&hist[dig], (uint32_t)__popc(peers));
      }
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
  // elements strictly above the K-th value (order does not matter here)
  for (int j = tid; j < rs.head; j += kThreads) {
    const float x = Row<Tin>::cvt(row[j]);
    if (okey(x) > kth) cand[atomicAdd(&sm_misc[2], 1)] = rkey(x, (uint32_t)j);
  }
  for (int j = tid; j < rs.tail; j += kThreads) {
    const float x = Row<Tin>::cvt(row[rs.tail0 + j]);
    if (okey(x) > kth) cand[atomicAdd(&sm_misc[2], 1)] = rkey(x, (uint32_t)(rs.tail0 + j));
  }
  for (int i = tid; i < rs.nvec; i += kThreads) {
    float x[VEC];
    load_vec(row, rs, i, x);
#pragma unroll
    for (int j = 0; j < VEC; ++j)
      if (okey(x[j]) > kth) cand[atomicAdd(&sm_misc[2], 1)] = rkey(x[j], (uint32_t)(rs.head + i * VEC + j));
  }
  __syncthreads();
  // elements equal to the K-th value, in id order: head, body vectors, tail
  int taken = 0;
  {
    int c = 0;
    float xh = 0.f;
    if (tid < rs.head) { xh = Row<Tin>::cvt(row[tid]); c = okey(xh) == kth; }
    int tot;
    const int r = block_excl_scan(c, sm_scan, &tot);
    if (c && taken + r < need_eq) cand[n_gt + taken + r] = rkey(xh, (uint32_t)tid);
    taken += tot;
  }
  for (int base = 0; base < rs.nvec && taken < need_eq; base += kThreads) {
    const int i = base + tid;
    float x[VEC];
    int c = 0;
    if (i < rs.nvec) {
      load_vec(row, rs, i, x);
#pragma unroll
      for (int j = 0; j < VEC; ++j) c += okey(x[j]) == kth;
    }
    int tot;
    int r = block_excl_scan(c, sm_scan, &tot);
    if (c) {
#pragma unroll
      for (int j = 0; j < VEC; ++j) {
        if (okey(x[j]) == kth) {
          if (taken + r < need_eq) cand[n_gt + taken + r] = rkey(x[j], (uint32_t)(rs.head + i * VEC + j));
          ++r;
        }
      }
    }
    taken += tot;  // block-uniform
  }
  if (taken < need_eq) {
    int c = 0;
    float xt = 0.f;
    if (tid < rs.tail) { xt = Row<Tin>::cvt(row[rs.tail0 + tid]); c = okey(xt) == kth; }
    int tot;
    const int r = block_excl_scan(c, sm_scan, &tot);
    if (c && taken + r < need_eq) cand[n_gt + taken + r] = rkey(xt, (uint32_t)(rs.tail0 + tid));
  }
  __syncthreads();
  bitonic_desc(cand, n_pow2);
}

// Five CTAs per SM (48 registers): the row stream is latency-bound, and on
// B300 five resident CTAs with 6 loads per thread in flight outrun three
// with 8 (0.62 vs 0.71 ms on the [8192, 201088] bf16 workload, identical
// output).
template <typename Tin>
__global__ void __launch_bounds__(kThreads, 5) topk_kernel(const Tin* __restrict__ logits, int64_t T, int V,
                                                           int64_t ld, int K, int force_exact,
                                                           int32_t* __restrict__ ids, float* __restrict__ logp,
                                                           int* __restrict__ ws_words) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  uint64_t* cand = reinterpret_cast<uint64_t*>(smem_raw);  // sel_entries(K) entries
  __shared__ uint32_t hist[256];
  __shared__ int sm_scan[kWarps + 1];
  __shared__ int sm_misc[4];
  __shared__ float sm_m[kWarps], sm_s[kWarps];
  __shared__ float sm_lse;
  __shared__ int sm_n;
  __shared__ int sm_next;
  __shared__ float bmax[kSlots][kThreads];  // per-thread batch maxima (batch b in slot b % kSlots)

  constexpr int VEC = Row<Tin>::kVec;
  constexpr int kLoBits = sizeof(Tin) == 2 ? 16 : 0;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int* row_counter = ws_words + 2;
  const bool fast = !force_exact && K <= kFastMaxK;

  if (tid == 0) sm_next = atomicAdd(row_counter, 1);
  __syncthreads();
  int row = sm_next;
  __syncthreads();
  while (row < T) {
    if (tid == 0) sm_next = atomicAdd(row_counter, 1);  // read after this row's barriers
    const Tin* rp = logits + (int64_t)row * ld;
    const RowSplit<Tin> rs(rp, V);
    const uint4* vr = reinterpret_cast<const uint4*>(rp + rs.head);
    const int nv = rs.nvec;

    // ---- pass 1: log-sum-exp and per-thread maximum
    Lse st;
    st.init();
    if (tid < rs.head) st.one(Row<Tin>::cvt(rp[tid]));
    if (tid < rs.tail) st.one(Row<Tin>::cvt(rp[rs.tail0 + tid]));
#pragma unroll
    for (int q = 0; q < kSlots; ++q) bmax[q][tid] = -INFINITY;
    int nb = 0;  // batches of this thread
    for (int i0 = tid; i0 < nv; i0 += kBatch * kThreads, ++nb) {
      uint4 u[kBatch];
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        const int i = i0 + q * kThreads;
        u[q] = i < nv ? __ldcs(vr + i) : make_uint4(0u, 0u, 0u, 0u);
      }
      float bm = -INFINITY;
      if (i0 + (kBatch - 1) * kThreads < nv) {
        // full batch: its maximum first (packed), one rescale, then the sums
        bm = batch_max<Tin>(u);
        st.max_to(bm);
        const float mb = -st.m * kLog2e;
        if constexpr (sizeof(Tin) == 2) {
          const uint64_t c2 = pack_f32x2(kLog2e, kLog2e), mb2 = pack_f32x2(mb, mb);
          uint64_t acc = 0;  // two fp32 lanes of 0.0
#pragma unroll
          for (int q = 0; q < kBatch; ++q) {
            sumexp_bf16x2(acc, u[q].x, c2, mb2);
            sumexp_bf16x2(acc, u[q].y, c2, mb2);
            sumexp_bf16x2(acc, u[q].z, c2, mb2);
            sumexp_bf16x2(acc, u[q].w, c2, mb2);
          }
          st.s += __uint_as_float((uint32_t)acc) + __uint_as_float((uint32_t)(acc >> 32));
        } else {
#pragma unroll
          for (int q = 0; q < kBatch; ++q) {
            float x[VEC];
            Row<Tin>::unpack(u[q], x);
            st.add_sum(x, mb);
          }
        }
      } else {
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
          if (i0 + q * kThreads < nv) {
            float x[VEC];
            Row<Tin>::unpack(u[q], x);
            float vmax = x[0];
#pragma unroll
            for (int j = 1; j < VEC; ++j) vmax = fmaxf(vmax, x[j]);
            st.add(x, vmax);
            bm = fmaxf(bm, vmax);
          }
        }
      }
      const int slot = nb % kSlots;
      bmax[slot][tid] = fmaxf(bmax[slot][tid], bm);
    }
    float m = st.m, sum = st.s;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, sum, o);
      lse_merge(m, sum, m2, s2);
    }
    if (lane == 0) { sm_m[warp] = m; sm_s[warp] = sum; }
    if (tid == 0) sm_n = 0;
    __syncthreads();
    if (tid == 0) {
      float M = sm_m[0], Sm = sm_s[0];
      for (int w = 1; w < kWarps; ++w) lse_merge(M, Sm, sm_m[w], sm_s[w]);
      sm_lse = M + logf(Sm);
    }

    bool exact = !fast;
    if (fast) {
      // ---- tau: K-th largest of the per-thread maxima (key 0 = no element)
      const uint32_t mykey = st.m == -INFINITY ? 0u : okey(st.m);
      uint32_t kth = 0;
      for (int b = 31; b >= kLoBits; --b) {
        const uint32_t c = kth | (1u << b);
        if (__syncthreads_count(mykey >= c) >= K) kth = c;
      }
      if (kLoBits && kth) kth |= (kth & 0x80000000u) ? 0u : ((1u << kLoBits) - 1u);
      const float tau = kth ? okey_to_float(kth) : -INFINITY;

      // ---- pass 2: every element >= tau into the candidate buffer
      if (tid < rs.head) {
        const float x = Row<Tin>::cvt(rp[tid]);
        if (x >= tau) {
          const int p = atomicAdd(&sm_n, 1);
          if (p < kCandCap) cand[p] = rkey(x, (uint32_t)tid);
        }
      }
      if (tid < rs.tail) {
        const float x = Row<Tin>::cvt(rp[rs.tail0 + tid]);
        if (x >= tau) {
          const int p = atomicAdd(&sm_n, 1);
          if (p < kCandCap) cand[p] = rkey(x, (uint32_t)(rs.tail0 + tid));
        }
      }
      // only batches whose recorded maximum reaches tau (threads whose
      // maximum is below tau read nothing)
      for (int bi = 0, i0 = tid; st.m >= tau && i0 < nv; i0 += kBatch * kThreads, ++bi) {
        if (bmax[bi % kSlots][tid] < tau) continue;
        uint4 u[kBatch];
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
          const int i = i0 + q * kThreads;
          u[q] = i < nv ? __ldcs(vr + i) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
          const int i = i0 + q * kThreads;
          if (i < nv) {
            float x[VEC];
            Row<Tin>::unpack(u[q], x);
            float vmax = x[0];
#pragma unroll
            for (int j = 1; j < VEC; ++j) vmax = fmaxf(vmax, x[j]);
            if (vmax >= tau) {
#pragma unroll
              for (int j = 0; j < VEC; ++j) {
                if (x[j] >= tau) {
                  const int p = atomicAdd(&sm_n, 1);
                  if (p < kCandCap) cand[p] = rkey(x[j], (uint32_t)(rs.head + i * VEC + j));
                }
              }
            }
          }
        }
      }
      __syncthreads();
      const int n = sm_n;
      if (n > kCandCap || n < K) {
        exact = true;
      } else {
        int n2 = 1;
        while (n2 < n) n2 <<= 1;
        for (int i = n + tid; i < n2; i += kThreads) cand[i] = 0;
        __syncthreads();
        bitonic_desc(cand, n2);
      }
    }
    if (exact) {
      if (tid == 0 && !force_exact) atomicAdd(&ws_words[1], 1);
      __syncthreads();
      int kp2 = 1;
      while (kp2 < K) kp2 <<= 1;  // <= sel_entries(K)
      exact_select<Tin>(rp, V, K, cand, kp2, hist, sm_scan, sm_misc);
    }
    __syncthreads();
    const float lse = sm_lse;
    for (int k = tid; k < K; k += kThreads) {
      const uint64_t c = cand[k];
      ids[(int64_t)row * K + k] = (int32_t)(0xFFFFFFFFu - (uint32_t)c);
      logp[(int64_t)row * K + k] = okey_to_float((uint32_t)(c >> 32)) - lse;
    }
    __syncthreads();
    row = sm_next;
    __syncthreads();
  }
}

constexpr int kTileW = kBNLogits;     // columns per tile of the teacher GEMM
constexpr int kTileListCap = 1024;    // tiles at or above tau read by the fast path
constexpr int kTauKeysPerLane = 32;   // warp-held tile-maximum keys (up to 1024 tiles)

__device__ __forceinline__ float block_max_f(float v, float* red) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if (lane == 0) red[w] = v;
  __syncthreads();
  float r = red[0];
  for (int i = 1; i < kWarps; ++i) r = fmaxf(r, red[i]);
  __syncthreads();
  return r;
}
// Sum in a fixed order (lanes by xor tree, then warps in index order).
__device__ __forceinline__ float block_sum_f(float v, float* red) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) red[w] = v;
  __syncthreads();
  float r = red[0];
  for (int i = 1; i < kWarps; ++i) r += red[i];
  __syncthreads();
  return r;
}
__device__ __forceinline__ int block_sum_i(int v, int* red) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) red[w] = v;
  __syncthreads();
  int r = 0;
  for (int i = 0; i < kWarps; ++i) r += red[i];
  __syncthreads();
  return r;
}

// One block per row of the chunk.
__global__ void __launch_bounds__(kThreads, 4) tile_topk_kernel(const float* __restrict__ Z, int64_t ldz, int V, int S,
                                                            const float* __restrict__ part_m,
                                                            const float* __restrict__ part_s, int K,
                                                            int force_exact, int32_t* __restrict__ ids,
                                                            float* __restrict__ logp, int* __restrict__ ws_words) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  uint64_t* cand = reinterpret_cast<uint64_t*>(smem_raw);  // sel_entries(K) entries
  __shared__ uint32_t hist[256];
  __shared__ int sm_scan[kWarps + 1];
  __shared__ int sm_misc[4];
  __shared__ float sm_red[kWarps];
  __shared__ int sm_ired[kWarps];
  __shared__ int tiles[kTileListCap];
  __shared__ int sm_nt, sm_n;
  __shared__ uint32_t sm_tau;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x;
  const float* pm = part_m + (size_t)row * S;
  const float* ps = part_s + (size_t)row * S;
  const float* zr = Z + (size_t)row * ldz;

  // log-sum-exp of the row from the tile partials
  float M = -INFINITY;
  for (int j = tid; j < S; j += kThreads) M = fmaxf(M, __ldg(pm + j));
  M = block_max_f(M, sm_red);
  float sum = 0.f;
  for (int j = tid; j < S; j += kThreads) sum += __ldg(ps + j) * ex2((__ldg(pm + j) - M) * kLog2e);
  sum = block_sum_f(sum, sm_red);
  const float lse = M + logf(sum);

  bool exact = force_exact || K > kFastMaxK;
  if (!exact) {
    // tau: the K-th largest tile maximum (key 0 = take every tile), by
    // bisection on the order keys. Up to 1024 tiles (V <= 262144), one warp
    // holds every key in registers and counts with warp reductions, so the
    // block waits at a single barrier; larger rows count block-wide.
    uint32_t kth = 0;
    if (S > K && S <= 32 * kTauKeysPerLane) {
      if (warp == 0) {
        uint32_t key[kTauKeysPerLane];
#pragma unroll
        for (int i = 0; i < kTauKeysPerLane; ++i) {
          const int j = lane + 32 * i;
          key[i] = j < S ? okey(__ldg(pm + j)) : 0u;  // key 0 never reaches c >= 1
        }
        for (int b = 31; b >= 0; --b) {
          const uint32_t c = kth | (1u << b);
          uint32_t cnt = 0;
#pragma unroll
          for (int i = 0; i < kTauKeysPerLane; ++i) cnt += key[i] >= c;
          if ((int)__reduce_add_sync(0xffffffffu, cnt) >= K) kth = c;
        }
        if (lane == 0) sm_tau = kth;
      }
      __syncthreads();
      kth = sm_tau;
    } else if (S > K) {
      for (int b = 31; b >= 0; --b) {
        const uint32_t c = kth | (1u << b);
        int cnt = 0;
        for (int j = tid; j < S; j += kThreads) cnt += okey(__ldg(pm + j)) >= c;
        if (block_sum_i(cnt, sm_ired) >= K) kth = c;
      }
    }
    if (tid == 0) { sm_nt = 0; sm_n = 0; }
    __syncthreads();
    for (int j = tid; j < S; j += kThreads) {
      if (okey(__ldg(pm + j)) >= kth) {
        const int p = atomicAdd(&sm_nt, 1);
        if (p < kTileListCap) tiles[p] = j;
      }
    }
    __syncthreads();
    const int nt = sm_nt;
    if (nt > kTileListCap) {
      exact = true;
    } else {
      // a warp per listed tile (32 lanes x 8 consecutive columns), four
      // tiles' loads in flight per warp before any is processed
      constexpr int kTilesInFlight = 4;
      for (int i0 = warp; i0 < nt; i0 += kWarps * kTilesInFlight) {
        float x[kTilesInFlight][8];
        int c0[kTilesInFlight];
#pragma unroll
        for (int u = 0; u < kTilesInFlight; ++u) {
          const int i = i0 + u * kWarps;
          c0[u] = i < nt ? tiles[i] * kTileW + lane * 8 : V;  // V: nothing to read
          if (c0[u] + 8 <= V) {
            const float4 a = __ldg(reinterpret_cast<const float4*>(zr + c0[u]));
            const float4 b = __ldg(reinterpret_cast<const float4*>(zr + c0[u] + 4));
            x[u][0] = a.x; x[u][1] = a.y; x[u][2] = a.z; x[u][3] = a.w;
            x[u][4] = b.x; x[u][5] = b.y; x[u][6] = b.z; x[u][7] = b.w;
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) x[u][j] = c0[u] + j < V ? __ldg(zr + c0[u] + j) : -INFINITY;
          }
        }
#pragma unroll
        for (int u = 0; u < kTilesInFlight; ++u) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (c0[u] + j < V && okey(x[u][j]) >= kth) {
              const int p = atomicAdd(&sm_n, 1);
              if (p < kCandCap) cand[p] = rkey(x[u][j], (uint32_t)(c0[u] + j));
            }
          }
        }
      }
      __syncthreads();
      const int n = sm_n;
      if (n > kCandCap || n < K) {
        exact = true;
      } else {
        int n2 = 1;
        while (n2 < n) n2 <<= 1;
        for (int i = n + tid; i < n2; i += kThreads) cand[i] = 0;
        __syncthreads();
        bitonic_desc(cand, n2);
      }
    }
  }
  if (exact) {
    if (tid == 0 && !force_exact) atomicAdd(&ws_words[1], 1);
    __syncthreads();
    int kp2 = 1;
    while (kp2 < K) kp2 <<= 1;
    exact_select<float>(zr, V, K, cand, kp2, hist, sm_scan, sm_misc);
  }
  __syncthreads();
  for (int k = tid; k < K; k += kThreads) {
    const uint64_t c = cand[k];
    ids[(int64_t)row * K + k] = (int32_t)(0xFFFFFFFFu - (uint32_t)c);
    logp[(int64_t)row * K + k] = okey_to_float((uint32_t)(c >> 32)) - lse;
  }
}

}  // namespace

// Entries of the candidate / exact-path buffer: the fast path's candidate
// buffer, or a power of two >= K for the exact path if larger.
static int sel_entries(int K) {
  int n = 1;
  while (n < K) n <<= 1;
  return n < kCandCap ? kCandCap : n;
}

size_t topk_smem_bytes(int K) { return (size_t)sel_entries(K) * sizeof(uint64_t); }
size_t tile_topk_smem_bytes(int K) { return topk_smem_bytes(K); }

cudaError_t launch_tile_topk(const float* Z, int64_t ldz, int rows, int V, int S, const float* part_m,
                             const float* part_s, int K, int32_t* ids, float* logp, int* ws_words, int force_exact,
                             cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const size_t smem = tile_topk_smem_bytes(K);
  cudaError_t e = cudaFuncSetAttribute(tile_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  tile_topk_kernel<<<rows, kThreads, smem, stream>>>(Z, ldz, V, S, part_m, part_s, K, force_exact, ids, logp,
                                                    ws_words);
  return cudaGetLastError();
}

cudaError_t launch_topk(const void* logits, int dtype, int64_t T, int64_t V, int64_t ld, int K,
                        int32_t* ids, float* logp, int* ws_words, int force_exact, int num_sms,
                        cudaStream_t stream) {
  const size_t smem = topk_smem_bytes(K);
  int blocks_per_sm = 0;
  cudaError_t e = cudaMemsetAsync(ws_words + 2, 0, sizeof(int), stream);  // row counter
  if (e != cudaSuccess) return e;
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
        static_cast<const uint16_t*>(logits), T, (int)V, ld, K, force_exact, ids, logp, ws_words);
  else
    topk_kernel<float><<<(unsigned)grid, kThreads, smem, stream>>>(
        static_cast<const float*>(logits), T, (int)V, ld, K, force_exact, ids, logp, ws_words);
  return cudaGetLastError();
}

}  // namespace kd
