// kd_gemm.cu - the projection GEMMs of the fused chunked KL loss on tcgen05.
//
// The three GEMM shapes of the method ("ทำให้ Knowledge Distillation มี
// ประสิทธิภาพ..." (ai-thai.com), section "กลไก Fused Chunked KL Loss": hidden
// states -> logits per chunk, loss accumulated, chunk discarded; backward
// recomputes each chunk):
//   logits  z = H_c W^T    A = H_c [c, d] K-major, B = W [V, d] K-major
//   dH^T    W^T dz^T       A = W [V, d] M-major,   B = dz [c, V] K-major
//           (stored transposed by the epilogue, so dH lands row-major)
//   dW      dz^T H_c       A = dz [c, V] M-major,  B = H_c^T [d, c] K-major
// These are the operand layouts the tensor core reads at full rate (an
// N-major B costs 15-28% on B300; an M-major A costs nothing).
// All run in one persistent, warp-specialised kernel template:
//   warp 0     TMA producer: takes the next tile from a global counter
//              (dynamic scheduling), passes its id to the other roles through
//              a 4-deep shared-memory queue, and streams the tile's A/B
//              blocks into a ring of shared-memory stages (128-byte swizzle).
//   warp 1     MMA issuer: one thread issues tcgen05.mma (K = 16 per
//              instruction) into one of two 256-column TMEM accumulators, or
//              (wide tiles) into one 512-column accumulator, two MMAs per K
//              step that share their A operand: the first keeps A in the
//              tensor core's collector buffer, the second reads it from
//              there, so A leaves shared memory once per K step.
//              tcgen05.commit frees the smem stage, and then signals the
//              finished accumulator.
//   warps 2+   epilogue: tcgen05.ld the accumulator (a warp may read only
//              its quadrant of 32 TMEM lanes = 32 rows; see the widths below
//              for how many warps share a quadrant). While the MMA warp fills
//              the other accumulator (narrow tiles) or after it finished
//              (wide tiles), they run the fused math:
//     EPI_FWD   online (max, sum exp) per row over the tile's vocabulary
//               slice, and the logits at the teacher ids that fall in it;
//     EPI_DZ    dz = s (exp(z - lse) - p [j in K]) -> bf16 -> TMA store;
//     EPI_GRAD  fp32 tile -> TMA store or TMA reduce-add (dW += ...),
//               optionally transposed (dH);
//     EPI_FWDST the EPI_FWD results, with the tile's maximum m as the
//               reference, plus e = exp(z - m) -> bf16 -> TMA store, from
//               which the single-call forward + backward forms dz without
//               recomputing the logits;
//     EPI_TEACHER the teacher's logits: per (row, tile) max and sum of exp
//               (for its log-sum-exp), and the fp32 tile -> TMA store, from
//               which the teacher top-K selection reads only the tiles that
//               can hold a top-K element.
// Two tile shapes:
//   C2 = false  one CTA per 128 x 256 tile (tcgen05 cta_group::1, M = 128).
//   C2 = true   a cluster of two CTAs per tile (cta_group::2, M = 256);
//               the even CTA issues the MMAs, which read both CTAs' shared
//               memory and write both CTAs' TMEM (each CTA holds its own 128
//               rows of the accumulator). B must be K-major. Two widths:
//     WIDE = false  256 x 256: each CTA loads 128 rows of A and a 128-row
//               half of B per K step; two 256-column accumulators let the
//               epilogue of one tile overlap the MMAs of the next.
//     WIDE = true   256 x 512: two N = 256 instructions per K step, each CTA
//               loads 256 rows of B (two 128-row boxes). Per SM that moves
//               48 bytes of operands per 1024 MMA cycles instead of 64, and
//               operand supply is what limits the narrow tile on B300
//               (8192^3: 1643 vs 1480 TF/s). The 512-column accumulator
//               fills TMEM, so the epilogue runs between tiles. Sixteen
//               epilogue warps (four per TMEM lane quadrant, 128 columns
//               each) keep it short for the forward, dz and store-exp
//               epilogues; the pair of warps on one 256-column half merge
//               their row statistics through shared memory. The fp32-store
//               epilogues (dH / dW, teacher logits) use eight warps with two
//               staging buffers each. Measured per GEMM, the wide tile pays
//               off for all of them, the dz recompute included.
// The logits tile therefore never leaves the chip in the forward pass. In
// backward, only the chunk's dz (bf16, c x V) goes to HBM.
#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "kd_internal.h"
#include "kd_ptx.cuh"

namespace kd {
namespace {

constexpr int EPI_FWD = 0, EPI_DZ = 1, EPI_GRAD = 2, EPI_FWDST = 3, EPI_TEACHER = 4;
constexpr int BN = kBNLogits;  // columns one epilogue warp covers per tile (a vocabulary tile)
static_assert(kBNLogits == kBNGrad, "one N tile for all GEMMs");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kStageBytesStaging = 4096;  // one 32-row x 128-byte staging buffer
constexpr uint32_t kNone = 0xFFFFFFFFu;


template <int NS, int EPI, bool C2, bool WIDE>
struct Cfg {
  static constexpr bool W = C2 && WIDE;               // 256 x 512 pair tiles
  static constexpr int TM = C2 ? 2 * kBM : kBM;       // rows of a tile
  static constexpr int TN = W ? 2 * BN : BN;          // columns of a tile
  static constexpr int NACC = W ? 1 : 2;              // TMEM accumulators (512 columns in all)
  // Epilogue warps. Wide tiles: four per TMEM lane quadrant (each on 128 of
  // the tile's 512 columns, one staging buffer each) for the epilogues that
  // keep statistics or store bf16 (forward, dz, store-exp); two per quadrant
  // (each on a 256-column half, two staging buffers each) for the ones that
  // store the fp32 tile (dH / dW, teacher logits), which lose more to single
  // buffering than they gain from more warps. One per quadrant otherwise.
  static constexpr int EPI_WARPS = W ? ((EPI == EPI_GRAD || EPI == EPI_TEACHER) ? 8 : 16) : 4;
  static constexpr int SUBS = W ? EPI_WARPS / 8 : 1;  // warps per 256-column half and quadrant
  static constexpr int SW = BN / SUBS;                // accumulator columns per warp and half
  static constexpr uint32_t NBUF = SUBS == 2 ? 1u : 2u;  // staging buffers per epilogue warp
  static constexpr bool DB = EPI_WARPS < 16;          // double-buffered TMEM loads (registers allow)
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;  // producer + MMA + epilogue warps
  static constexpr int BNL = (C2 && !WIDE) ? 128 : 256;  // B rows held by one CTA per K step
  static constexpr uint32_t A_BYTES = kBM * kBK * 2;  // this CTA's A block
  static constexpr uint32_t B_BYTES = BNL * kBK * 2;  // this CTA's B block
  static constexpr uint32_t STAGE = A_BYTES + B_BYTES;
  static constexpr uint32_t TX = C2 ? 2 * STAGE : STAGE;  // bytes that complete one full-barrier phase
  static constexpr uint32_t STG = (EPI == EPI_FWD) ? 0u : (uint32_t)EPI_WARPS * NBUF * kStageBytesStaging;
  static constexpr uint32_t BAR_OFF = NS * STAGE + STG;
  // With four warps per quadrant, the two warps that share a 256-column half
  // combine their per-row statistics through XCH: 16 pair barriers
  // [kind][half][quadrant], then [kind][half][quadrant][warp][2][32] floats.
  static constexpr uint32_t XCH_OFF = BAR_OFF + 256;
  static constexpr uint32_t XCH = SUBS == 2 ? 128u + 2u * 2u * 4u * 2u * 64u * 4u : 0u;
  static constexpr uint32_t SMEM = XCH_OFF + XCH + 1024;  // + alignment slack
  static_assert((2 * NS + 13) * 8 + 24 <= 256, "barrier block");
};

struct Tile {
  int prob, mb, nb;
};

__device__ __forceinline__ Tile decode(const GemmArgs& g, int t) {
  Tile r;
  r.prob = (g.nprob > 1 && t >= g.pr[1].tile_begin) ? 1 : 0;
  const Problem& P = g.pr[r.prob];
  const int i = t - P.tile_begin;
  if (P.n_fastest) {
    r.nb = i % P.n_blocks;
    r.mb = i / P.n_blocks;
  } else {
    r.mb = i % P.m_blocks;
    r.nb = i / P.m_blocks;
  }
  return r;
}

// First index k in the ascending list rid[0..cnt) with rid[k] >= x.
__device__ __forceinline__ int lower_bound(const int* rid, int cnt, int x) {
  int lo = 0, hi = cnt;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(rid + mid) < x) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// Runs f(v, c0) over columns [0, ncols) of a warp's TMEM rows, 32 columns
// at a time (v: lane i holds row i's 32 fp32 values at columns c0 ...
// c0 + 31). The load of the next 32 columns is in flight while f works on
// the current ones (two register buffers). ncols is warp-uniform.
// done() runs once, as soon as the last load has completed (before f works
// on those columns; at once if there are none): from then on the sweep
// reads only registers, so the caller may hand the accumulator back there.
template <bool DB = true, typename F, typename D>
__device__ __forceinline__ void tmem_sweep(uint32_t taddr, int ncols, F&& f, D&& done) {
  const int nch = (ncols + 31) >> 5;
  if (nch <= 0) {
    done();
    return;
  }
  if (!DB) {  // one register buffer (for register-tight launches)
    uint32_t v[32];
    for (int c = 0; c < nch; ++c) {
      tmem_ld32(taddr + (uint32_t)c * 32u, v);
      tmem_wait_ld_r(v);
      if (c + 1 == nch) done();
      f(v, c * 32);
    }
    return;
  }
  uint32_t va[32], vb[32];
  tmem_ld32(taddr, va);
  tmem_wait_ld_r(va);
  if (nch == 1) done();
  for (int c = 0; c < nch; c += 2) {
    const bool nb = c + 1 < nch;
    if (nb) tmem_ld32(taddr + (uint32_t)(c + 1) * 32u, vb);
    f(va, c * 32);
    if (nb) {
      tmem_wait_ld_r(vb);
      const bool na = c + 2 < nch;
      if (!na) done();
      if (na) tmem_ld32(taddr + (uint32_t)(c + 2) * 32u, va);
      f(vb, (c + 1) * 32);
      if (na) {
        tmem_wait_ld_r(va);
        if (c + 3 == nch) done();
      }
    }
  }
}
template <bool DB = true, typename F>
__device__ __forceinline__ void tmem_sweep(uint32_t taddr, int ncols, F&& f) {
  tmem_sweep<DB>(taddr, ncols, f, [] {});
}

// Maximum of the first lim (>= 1) of the 32 values.
__device__ __forceinline__ float max32_lim(const uint32_t (&v)[32], int lim) {
  if (lim >= 32) return max32(v);
  float m = -INFINITY;
#pragma unroll
  for (int j = 0; j < 32; ++j)
    if (j < lim) m = fmaxf(m, u2f(v[j]));
  return m;
}

// sum_j exp2(v_j * a + b) over the first lim of the 32 values, in four
// independent partial sums.
__device__ __forceinline__ float sumexp32_lim(const uint32_t (&v)[32], int lim, float a, float b) {
  float s4[4] = {0.f, 0.f, 0.f, 0.f};
  if (lim >= 32) {
#pragma unroll
    for (int j = 0; j < 32; ++j) s4[j & 3] += ex2(fmaf(u2f(v[j]), a, b));
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < lim) s4[j & 3] += ex2(fmaf(u2f(v[j]), a, b));
  }
  return (s4[0] + s4[1]) + (s4[2] + s4[3]);
}

// ------------------------------------------------------------ cluster helpers
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of the same shared-memory location in cluster CTA `rank`.
__device__ __forceinline__ uint32_t mapa(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_remote(uint64_t* local_bar, uint32_t rank) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(mapa(smem_u32(local_bar), rank))
               : "memory");
}
__device__ __forceinline__ void st_remote_u32(const volatile int* local, uint32_t rank, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(mapa(smem_u32((const void*)local), rank)), "r"(v)
               : "memory");
}
// Pair TMA load: the bytes land in this CTA's smem and complete on the
// barrier at cluster address `bar_c` (the even CTA's full barrier).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* m, uint32_t bar_c, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(m), "r"(bar_c), "r"(x), "r"(y)
      : "memory");
}

template <bool C2>
__device__ __forceinline__ void tmem_alloc_x(uint32_t* slot) {
  if (C2) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  } else {
    tmem_alloc(slot, kTmemCols);
    tmem_relinquish();
  }
}
template <bool C2>
__device__ __forceinline__ void tmem_dealloc_x(uint32_t taddr) {
  if (C2)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(kTmemCols) : "memory");
  else
    tmem_dealloc(taddr, kTmemCols);
}
// A-operand collector use of one MMA: none, fill (read A from shared memory
// and keep it), or lastuse (take A kept by the previous MMA, then drop it).
enum class CollA { kNone, kFill, kLastUse };
template <bool C2, CollA CA = CollA::kNone>
__device__ __forceinline__ void mma_x(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accum) {
  if (C2 && CA == CollA::kFill)
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16.collector::a::fill [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(accum)
        : "memory");
  else if (C2 && CA == CollA::kLastUse)
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16.collector::a::lastuse [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(accum)
        : "memory");
  else if (C2)
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(accum)
        : "memory");
  else
    tc_mma_f16(d, a, b, idesc, accum);
}
// Arrives on `bar` once the MMAs issued so far are complete; with C2 also on
// the barrier at the same offset in the other CTA of the pair.
template <bool C2>
__device__ __forceinline__ void commit_x(uint64_t* bar) {
  if (C2) {
    const uint16_t mask = 3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(mask)
        : "memory");
  } else {
    tc_commit(bar);
  }
}

template <int NS, int EPI, bool C2, bool WIDE>
__global__ void __launch_bounds__(Cfg<NS, EPI, C2, WIDE>::THREADS, 1)
    gemm_kernel(const __grid_constant__ GemmArgs g) {
  using C = Cfg<NS, EPI, C2, WIDE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* full = bars;                 // [NS] TMA -> MMA (C2: the even CTA's count both halves)
  uint64_t* empty = bars + NS;           // [NS] MMA -> TMA
  uint64_t* tfull = bars + 2 * NS;       // [2]  MMA -> epilogue
  uint64_t* tempty = bars + 2 * NS + 2;  // [2]  epilogue -> MMA (C2: the even CTA's count both CTAs)
  uint64_t* drain = bars + 2 * NS + 4;   // all issued MMAs done, before TMEM is released
  uint64_t* tqf = bars + 2 * NS + 5;     // [4] tile queue: id published
  uint64_t* tqe = bars + 2 * NS + 9;     // [4] tile queue: slot free again (C2: in the even CTA)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * NS + 13);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* tq = reinterpret_cast<volatile int*>(tmem_slot + 2);  // [4] tile ids

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = C2 ? cluster_rank() : 0u;
  const bool leader = rank == 0;
  // Readers that release a queue slot: the MMA thread and the epilogue
  // warps, plus (C2) the odd CTA's producer and epilogue warps.
  constexpr uint32_t kQueueReaders = C2 ? 2u * (1u + C::EPI_WARPS) : 1u + C::EPI_WARPS;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], (C2 ? 2 : 1) * C::EPI_WARPS);
    }
    mbar_init(drain, 1);
    for (int q = 0; q < 4; ++q) { mbar_init(&tqf[q], 1); mbar_init(&tqe[q], kQueueReaders); }
    if (C::SUBS == 2)
      for (int q = 0; q < 16; ++q) mbar_init(reinterpret_cast<uint64_t*>(smem + C::XCH_OFF) + q, 2);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int p = 0; p < g.nprob; ++p) {
      tma_prefetch_desc(&g.tmA[p]);
      tma_prefetch_desc(&g.tmB[p]);
      if (EPI != EPI_FWD) tma_prefetch_desc(&g.tmC[p]);
      if (EPI == EPI_GRAD && g.pr[p].bnh == 240) tma_prefetch_desc(&g.tmCt[p]);
    }
  }
  if (warp == 1) tmem_alloc_x<C2>(tmem_slot);
  tc_fence_before();
  __syncwarp();            // the cluster barrier is .aligned: whole warps arrive together
  if (C2) cluster_sync();  // barriers of both CTAs initialised before any remote arrive
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, ipar = 0;  // per-stage bit: load issued / its phase parity
      bool ok = true;
      const uint32_t full0_c = C2 ? mapa(smem_u32(full), 0) : 0u;
      for (int j = 0; ok; ++j) {
        const int qs = j & 3;
        const uint32_t qpar = (uint32_t)(j >> 2) & 1u;
        int t;
        if (leader) {
          // Tiles are handed out in index order by a global counter: a CTA
          // (pair) takes the next tile when it starts one, so long and short
          // tiles balance.
          t = atomicAdd(g.tile_counter, 1);
          if (t >= g.total_tiles) t = -1;
          if (!mbar_wait<C2>(&tqe[qs], qpar ^ 1u, abort_flag)) { ok = false; break; }
          tq[qs] = t;
          if (C2) {
            st_remote_u32(&tq[qs], 1, (uint32_t)t);
            mbar_arrive_remote(&tqf[qs], 1);
          }
          mbar_arrive(&tqf[qs]);
        } else {
          if (!mbar_wait<true>(&tqf[qs], qpar, abort_flag)) { ok = false; break; }
          t = tq[qs];
          mbar_arrive_remote(&tqe[qs], 0);
        }
        if (t < 0) break;
        const Tile tl = decode(g, t);
        const Problem& P = g.pr[tl.prob];
        const CUtensorMap* mA = &g.tmA[tl.prob];
        const CUtensorMap* mB = &g.tmB[tl.prob];
        const int am = tl.mb * C::TM + (int)rank * kBM;  // this CTA's first A row (M)
        // N of one MMA: wide pair tiles run two of them, bnh columns apart
        // (each CTA loads bnh / 2 B rows for each); 256 otherwise
        const int bnh = (C::W && P.bnh) ? P.bnh : BN;
        // this CTA's first B row (N); wide pair tiles load a second box bnh
        // rows further
        const int bn = C2 ? (C::W ? tl.nb * 2 * bnh + (int)rank * (bnh / 2) : tl.nb * C::TN + (int)rank * 128)
                          : tl.nb * C::TN;
        const uint32_t tx = C::W ? 2u * (C::A_BYTES + 2u * (uint32_t)(bnh / 2) * 128u) : C::TX;
        for (int kb = 0; kb < P.k_blocks; ++kb) {
          if (!mbar_wait<C2>(&empty[stage], phase ^ 1u, abort_flag)) { ok = false; break; }
          const uint32_t sA = smem_u32(smem + stage * C::STAGE);
          const uint32_t sB = sA + C::A_BYTES;
          if (C2) {
            const uint32_t fb = full0_c + (uint32_t)stage * 8u;
            if (leader) mbar_arrive_expect_tx(&full[stage], tx);
            if (!P.a_mn) {
              tma_load_2d_pair(sA, mA, fb, kb * kBK, am);
            } else {
#pragma unroll
              for (int q = 0; q < kBM / 64; ++q) tma_load_2d_pair(sA + q * 8192, mA, fb, am + q * 64, kb * kBK);
            }
            tma_load_2d_pair(sB, mB, fb, kb * kBK, bn);  // (wide: N half 0)
            if (C::W) tma_load_2d_pair(sB + 16384, mB, fb, kb * kBK, bn + bnh);  // N half 1
          } else {
            mbar_arrive_expect_tx(&full[stage], C::TX);
            if (!P.a_mn) {
              tma_load_2d(sA, mA, &full[stage], kb * kBK, am);
            } else {
#pragma unroll
              for (int q = 0; q < kBM / 64; ++q) tma_load_2d(sA + q * 8192, mA, &full[stage], am + q * 64, kb * kBK);
            }
            if (!P.b_mn) {
              tma_load_2d(sB, mB, &full[stage], kb * kBK, bn);
            } else {
#pragma unroll
              for (int q = 0; q < BN / 64; ++q) tma_load_2d(sB + q * 8192, mB, &full[stage], bn + q * 64, kb * kBK);
            }
          }
          issued |= 1u << stage;
          ipar = (ipar & ~(1u << stage)) | (phase << stage);
          if (++stage == NS) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        set_status(g.status, ST_TIMEOUT);
        *abort_flag = 1;
      }
      // Never leave while a TMA load may still write shared memory: wait
      // (bounded) until the last load issued into each stage has landed.
      // Nothing else arrives on full[s] afterwards, so the phase it completes
      // stays the most recent one and the parity wait returns at once on the
      // normal path. With C2 the even CTA's barriers also count the odd
      // CTA's bytes, and the odd CTA leaves only after the final cluster
      // barrier, i.e. after this wait.
      if (leader) {
        for (int st = 0; st < NS; ++st) {
          if (!((issued >> st) & 1u)) continue;
          const uint32_t a = smem_u32(&full[st]);
          const uint64_t t0 = globaltimer();
          while (!mbar_try_wait(a, (ipar >> st) & 1u)) {
            if (globaltimer() - t0 > kWaitLimitNs) break;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int j = 0; ok; ++j) {
        const int qs = j & 3;
        if (!mbar_wait<C2>(&tqf[qs], (uint32_t)(j >> 2) & 1u, abort_flag)) { ok = false; break; }
        const int t = tq[qs];
        mbar_arrive(&tqe[qs]);
        if (t < 0) break;
        const Tile tl = decode(g, t);
        const Problem& P = g.pr[tl.prob];
        if (!mbar_wait<C2>(&tempty[acc], acc_phase ^ 1u, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);  // wide: acc = 0, columns [0, 512)
        const int b_mn = C2 ? 0 : P.b_mn;
        const uint32_t idesc = idesc_bf16_f32(C::TM, (C::W && P.bnh) ? P.bnh : BN, P.a_mn, b_mn);
        for (int kb = 0; kb < P.k_blocks; ++kb) {
          if (!mbar_wait<C2>(&full[stage], phase, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sA = smem_u32(smem + stage * C::STAGE);
          const uint32_t sB = sA + C::A_BYTES;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint64_t ad = P.a_mn ? sdesc_sw128(sA + k * 2048, 8192, 1024) : sdesc_sw128(sA + k * 32, 16, 1024);
            const uint64_t bd = b_mn ? sdesc_sw128(sB + k * 2048, 8192, 1024) : sdesc_sw128(sB + k * 32, 16, 1024);
            if (C::W) {
              // The two N halves share A: the first MMA keeps it in the
              // collector, the second (B rows 256 further in smem, TMEM
              // columns 256 further) reads it from there instead of smem.
              mma_x<C2, CollA::kFill>(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
              mma_x<C2, CollA::kLastUse>(d_tmem + 256, ad, sdesc_sw128(sB + 16384 + k * 32, 16, 1024), idesc,
                                         (kb | k) != 0 ? 1u : 0u);
            } else {
              mma_x<C2>(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
            }
          }
          commit_x<C2>(&empty[stage]);
          if (++stage == NS) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        commit_x<C2>(&tfull[acc]);
        if (++acc == C::NACC) { acc = 0; acc_phase ^= 1u; }
      }
      if (!ok) {
        set_status(g.status, ST_TIMEOUT);
        *abort_flag = 1;
      }
      // Let every MMA already issued finish before TMEM is released (with
      // C2 the arrival reaches the drain barrier of both CTAs).
      commit_x<C2>(drain);
    }
    if (lane == 0) {
      const uint32_t a = smem_u32(drain);
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(a, 0u)) {
        if (globaltimer() - t0 > kWaitLimitNs) break;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int wq = warp & 3;        // TMEM lane quadrant this warp may access
    const int ew = warp - 2;        // epilogue warp index
    // Column block of this warp: wide tiles give each quadrant four warps,
    // one per 128 columns (hc = which 256-column half, sub = which 128
    // columns of it); otherwise one warp covers the 256-column tile.
    const int hc = (ew >> 2) / C::SUBS;
    const int sub = (ew >> 2) % C::SUBS;
    int acc = 0;
    uint32_t acc_phase = 0;
    int buf = 0, nstore = 0;
    bool ok = true;
    uint8_t* stg = smem + NS * C::STAGE + (uint32_t)ew * C::NBUF * kStageBytesStaging;
    // The staging buffer for the next TMA store box, once the store that last
    // used it has finished reading it.
    auto stage_buf = [&]() -> uint32_t {
      if (nstore >= (int)C::NBUF) {
        if (lane == 0) {
          if (C::NBUF == 2) bulk_wait_read<1>();
          else bulk_wait_read<0>();
        }
        __syncwarp();
      }
      return smem_u32(stg + buf * kStageBytesStaging);
    };
    auto stage_issued = [&]() {
      ++nstore;
      buf = (buf + 1) % (int)C::NBUF;
    };
    uint64_t* pbar = reinterpret_cast<uint64_t*>(smem + C::XCH_OFF);  // [kind][half][quadrant]
    float* xch = reinterpret_cast<float*>(smem + C::XCH_OFF + 128);    // [kind][half][quadrant][warp][2][32]
    // Wide tiles: hand two values of this row to the other warp of the same
    // quadrant and half, and take its two (po). `kind` selects one of two
    // barriers and buffers, so a tile can exchange twice. Bounded: false on
    // a timeout or an abort.
    auto pair_exchange = [&](int kind, float a, float b, float* po) -> bool {
      float* base = xch + ((kind * 2 + hc) * 4 + wq) * 2 * 64;
      float* mine = base + sub * 64;
      const float* other = base + (sub ^ 1) * 64;
      mine[lane] = a;
      mine[32 + lane] = b;
      __syncwarp();
      uint64_t* bar = pbar + (kind * 2 + hc) * 4 + wq;
      if (lane == 0) mbar_arrive(bar);
      const bool w = mbar_wait<false>(bar, acc_phase, abort_flag);
      po[0] = other[lane];
      po[1] = other[32 + lane];
      return w;
    };
    for (int j = 0;; ++j) {
      const int qs = j & 3;
      if (!mbar_wait<C2>(&tqf[qs], (uint32_t)(j >> 2) & 1u, abort_flag)) ok = false;
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      const int t = tq[qs];
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(&tqe[qs]);
        else mbar_arrive_remote(&tqe[qs], 0);
      }
      if (t < 0) break;
      const Tile tl = decode(g, t);
      const Problem& P = g.pr[tl.prob];
      const int m0 = tl.mb * C::TM + (int)rank * kBM;  // first tile row held in this CTA's TMEM
      const int row = m0 + 32 * wq + lane;
      const int vt = tl.nb * (C::TN / BN) + hc;  // the 256-column block (vocabulary tile) of this warp
      const int bnh = (C::W && P.bnh) ? P.bnh : BN;  // columns of this warp's half (256, or 240)
      const int n0 = vt * bnh;                       // first column of the half
      const int c_sub = sub * C::SW;                 // this warp's first column within the half
      const int nw0 = n0 + c_sub;                    // ... and in C
      const int sw = min(C::SW, bnh - c_sub);        // this warp's columns of the half

      // Teacher-id cursor of this row for the warp's vocabulary columns.
      int cnt = 0, k = 0;
      const int* rid = nullptr;
      int nvalid = 0;
      if (EPI != EPI_GRAD) {
        nvalid = min(sw, g.V - nw0);
        if (row < g.rows) {
          cnt = __ldg(g.cnt + row);
          rid = g.ids_sorted + (size_t)row * g.Kp;
          k = lower_bound(rid, cnt, nw0);
        }
      }

      if (!mbar_wait<C2>(&tfull[acc], acc_phase, abort_flag)) { ok = false; }
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t taddr =
          tmem_base + ((uint32_t)(32 * wq) << 16) + (uint32_t)((acc + hc) * BN) + (uint32_t)c_sub;
      // Hands the accumulator back to the MMA warp (C2: the even CTA's
      // barrier counts both CTAs). The sweeps call it once their last
      // TMEM load has completed, so the next tile's MMAs run while this
      // warp finishes its last columns from registers.
      bool released = false;
      auto release = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (leader) mbar_arrive(&tempty[acc]);
          else mbar_arrive_remote(&tempty[acc], 0);
        }
        released = true;
      };
      // The loss epilogues work on z / tau: exp arguments use zl2 = log2(e) / tau
      // and the values they keep (tile maxima, logits at teacher ids) are
      // scaled by zscale = 1 / tau. With tau = 1 this is the plain logit.
      const float zscale = g.zscale, zl2 = zscale * kLog2e;

      // Next teacher id of this row inside the warp's columns (kNone if none).
      const uint32_t hiend = (uint32_t)(nw0 + nvalid);
      auto next_id = [&]() -> uint32_t {
        return (k < cnt && (uint32_t)__ldg(rid + k) < hiend) ? (uint32_t)__ldg(rid + k) : kNone;
      };
      // Per-(row, vocabulary tile) statistics: m in units of z and s = sum
      // exp2((z - m) * l2). Wide tiles first combine the two warps of the
      // half (the one with sub = 0 writes).
      auto write_stats = [&](float m, float s, float l2, float mscale) -> bool {
        if (C::SUBS == 2) {
          float po[2];
          const bool w = pair_exchange(1, m, s, po);
          if (!__all_sync(0xffffffffu, w)) return false;
          if (sub != 0) return true;
          const float M = fmaxf(m, po[0]);
          float S = 0.f;
          if (m > -INFINITY) S += s * ex2((m - M) * l2);
          if (po[0] > -INFINITY) S += po[1] * ex2((po[0] - M) * l2);
          m = M;
          s = S;
        }
        if (row < g.rows && n0 < g.V) {
          g.part_m[(size_t)row * g.S + vt] = m * mscale;
          g.part_s[(size_t)row * g.S + vt] = s;
        }
        return true;
      };

      if (EPI == EPI_TEACHER) {
        // Online (max, sum exp) over the valid columns, 32 at a time, and
        // each 32 x 32 fp32 block stored as it is read.
        float m = -INFINITY, s = 0.f;
        const bool box_live = m0 + 32 * wq < g.rows;
        tmem_sweep<C::DB>(taddr, nvalid, [&](uint32_t (&v)[32], int c0) {
          const uint32_t sb = stage_buf();
          const int lim = nvalid - c0;
          const float mn = fmaxf(m, max32_lim(v, lim));
          const float acc_s = sumexp32_lim(v, lim, kLog2e, -mn * kLog2e);
          s = s * ex2((m - mn) * kLog2e) + acc_s;
          m = mn;
#pragma unroll
          for (int q = 0; q < 8; ++q)
            st_shared_v4(sb + lane * 128 + ((q ^ (lane & 7)) << 4), v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && box_live) tma_store_2d(&g.tmC[0], sb, nw0 + c0, m0 + 32 * wq);
          if (lane == 0) bulk_commit();
          stage_issued();
        }, release);
        if (!write_stats(m, s, kLog2e, 1.f)) { ok = false; break; }
      } else if (EPI == EPI_FWDST || EPI == EPI_DZ) {
        // Pass over the warp's columns storing bf16 values, 64 columns per
        // TMA box (columns past V are clipped by the store):
        //   EPI_FWDST  e = exp((z - m) / tau), m = the row's maximum over the
        //              256-column tile (a first pass; on wide tiles over both
        //              warps of the half), summed in fp32; and z at the
        //              teacher ids (fp32, from the registers);
        //   EPI_DZ     dz = s (exp(z / tau - lse) - p [j in K]); at a teacher
        //              id the difference is formed in fp32 and rounded once.
        float m = -INFINITY;
        if (EPI == EPI_FWDST) {
          tmem_sweep<C::DB>(taddr, nvalid,
                            [&](uint32_t (&v)[32], int c0) { m = fmaxf(m, max32_lim(v, nvalid - c0)); });
          if (C::SUBS == 2) {
            float po[2];
            const bool w = pair_exchange(0, m, 0.f, po);
            if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
            m = fmaxf(m, po[0]);
          }
        }
        float sc = 0.f, nb = 0.f;
        if (EPI == EPI_DZ) {
          const float lse_r = (row < g.rows) ? __ldg(g.lse + row) : 0.f;
          const bool excluded = g.mask && row < g.rows && g.mask[row] == 0;
          sc = excluded ? 0.f : g.scale * (g.dscale ? __ldg(g.dscale) : 1.f);
          nb = -lse_r * kLog2e;
        } else {
          nb = -m * zl2;
        }
        float s4[4] = {0.f, 0.f, 0.f, 0.f};
        const bool box_live = m0 + 32 * wq < g.rows;
        uint32_t want = next_id();
        uint32_t sb = 0;
        tmem_sweep<C::DB>(taddr, nvalid, [&](uint32_t (&v)[32], int c0) {
          const int h = (c0 >> 5) & 1;  // which half of the 64-column box
          if (h == 0) sb = stage_buf();
          const int lim = nvalid - c0;
          uint32_t pk[16];
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            float e0 = ex2(fmaf(u2f(v[2 * jj]), zl2, nb));
            float e1 = ex2(fmaf(u2f(v[2 * jj + 1]), zl2, nb));
            if (EPI == EPI_DZ) {
              e0 *= sc;
              e1 *= sc;
            } else if (lim >= 32) {
              s4[jj & 3] += e0 + e1;
            } else {
              if (2 * jj < lim) s4[jj & 3] += e0;
              if (2 * jj + 1 < lim) s4[jj & 3] += e1;
            }
            pk[jj] = pack_bf16x2(e0, e1);
          }
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            const int q = h * 4 + qq;
            st_shared_v4(sb + lane * 128 + ((q ^ (lane & 7)) << 4), pk[4 * qq], pk[4 * qq + 1], pk[4 * qq + 2],
                         pk[4 * qq + 3]);
          }
          // Teacher ids in these 32 columns, from the fp32 logits in registers.
          const uint32_t lo = (uint32_t)(nw0 + c0);
          bool mine = want < lo + 32u;
          while (__any_sync(0xffffffffu, mine)) {
            if (mine) {
              const uint32_t jj = want - lo;
              const float z = u2f(select32(v, jj));
              if (EPI == EPI_DZ) {
                const float q = ex2(fmaf(z, zl2, nb));
                const float dz = sc * (q - __ldg(g.p_sorted + (size_t)row * g.Kp + k));
                const int col = h * 32 + (int)jj;
                const __nv_bfloat16 hb = __float2bfloat16_rn(dz);
                st_shared_u16(sb + lane * 128 + (((col >> 3) ^ (lane & 7)) << 4) + ((col & 7) << 1),
                              *reinterpret_cast<const uint16_t*>(&hb));
              } else {
                g.zK[(size_t)row * g.Kp + k] = z * zscale;
              }
              ++k;
              want = next_id();
              mine = want < lo + 32u;
            }
          }
          if (h == 1 || c0 + 32 >= nvalid) {  // the 64-column box is complete
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && box_live) tma_store_2d(&g.tmC[0], sb, nw0 + c0 - 32 * h, m0 + 32 * wq);
            if (lane == 0) bulk_commit();
            stage_issued();
          }
        }, release);
        if (EPI == EPI_FWDST) {
          // the sums are relative to the common maximum m: the pair just adds
          float s = (s4[0] + s4[1]) + (s4[2] + s4[3]);
          bool write = true;
          if (C::SUBS == 2) {
            float po[2];
            const bool w = pair_exchange(1, s, 0.f, po);
            if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
            s += po[0];
            write = sub == 0;
          }
          if (write && row < g.rows && n0 < g.V) {
            g.part_m[(size_t)row * g.S + vt] = m * zscale;
            g.part_s[(size_t)row * g.S + vt] = s;
          }
        }
      } else if (EPI == EPI_FWD) {
        // Online (max, sum exp) per row over the warp's columns, and the
        // logits at the teacher ids that fall in them.
        float m = -INFINITY, s = 0.f;
        uint32_t want = next_id();
        tmem_sweep<C::DB>(taddr, nvalid, [&](uint32_t (&v)[32], int c0) {
          const int lim = nvalid - c0;
          const float mn = fmaxf(m, max32_lim(v, lim));
          const float acc_s = sumexp32_lim(v, lim, zl2, -mn * zl2);
          s = s * ex2((m - mn) * zl2) + acc_s;
          m = mn;
          const uint32_t lo = (uint32_t)(nw0 + c0);
          bool mine = want < lo + 32u;
          while (__any_sync(0xffffffffu, mine)) {
            if (mine) {
              g.zK[(size_t)row * g.Kp + k] = u2f(select32(v, want - lo)) * zscale;
              ++k;
              want = next_id();
              mine = want < lo + 32u;
            }
          }
        }, release);
        if (!write_stats(m, s, zl2, zscale)) { ok = false; break; }
      } else {
        // EPI_GRAD: the fp32 tile, 32 columns per TMA box, stored or
        // reduce-added into C, or written as C^T (TMEM lanes are then C's
        // columns): fp32, or bf16 in 64-byte rows without swizzle.
        const CUtensorMap* mC = &g.tmC[tl.prob];
        const bool box_live = m0 + 32 * wq < P.M;
        const int ncols = min(sw, P.N - nw0);
        tmem_sweep<C::DB>(taddr, ncols, [&](uint32_t (&v)[32], int c0) {
          const uint32_t sb = stage_buf();
          if (c_sub + c0 + 32 > bnh) {
            // the last 16 columns of a 240-wide half (plain fp32 C): a 16-column
            // box, so nothing is stored into the neighbouring tile's columns
#pragma unroll
            for (int q = 0; q < 4; ++q)
              st_shared_v4(sb + lane * 64 + q * 16, v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && box_live) {
              if (P.reduce_add) tma_reduce_add_2d(&g.tmCt[tl.prob], sb, nw0 + c0, m0 + 32 * wq);
              else tma_store_2d(&g.tmCt[tl.prob], sb, nw0 + c0, m0 + 32 * wq);
            }
            if (lane == 0) bulk_commit();
            stage_issued();
            return;
          }
          if (P.c_trans && P.out_bf16) {
            // a warp's 32 lanes fill one 64-byte row: conflict-free
#pragma unroll
            for (int r = 0; r < 32; ++r) {
              const __nv_bfloat16 hv = __float2bfloat16_rn(u2f(v[r]));
              st_shared_u16(sb + r * 64 + lane * 2, *reinterpret_cast<const uint16_t*>(&hv));
            }
          } else if (P.c_trans) {
            // [C row][C column], one 4-byte store per element, conflict-free
            // under the 128-byte swizzle
#pragma unroll
            for (int r = 0; r < 32; ++r)
              st_shared_b32(sb + r * 128 + ((((uint32_t)lane >> 2) ^ (uint32_t)(r & 7)) << 4) + ((lane & 3) << 2), v[r]);
          } else {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              st_shared_v4(sb + lane * 128 + ((q ^ (lane & 7)) << 4), v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && box_live) {
            if (P.c_trans && P.out_bf16) tma_store_2d(mC, sb, m0 + 32 * wq, nw0 + c0);
            else if (P.c_trans && P.reduce_add) tma_reduce_add_2d(mC, sb, m0 + 32 * wq, nw0 + c0);
            else if (P.c_trans) tma_store_2d(mC, sb, m0 + 32 * wq, nw0 + c0);
            else if (P.reduce_add) tma_reduce_add_2d(mC, sb, nw0 + c0, m0 + 32 * wq);
            else tma_store_2d(mC, sb, nw0 + c0, m0 + 32 * wq);
          }
          if (lane == 0) bulk_commit();
          stage_issued();
        }, release);
      }
      if (!released) release();  // (every sweep releases; kept as a guard)
      if (++acc == C::NACC) { acc = 0; acc_phase ^= 1u; }
    }
    if (!ok) {
      if (lane == 0) { set_status(g.status, ST_TIMEOUT); *abort_flag = 1; }
    }
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
  }

  tc_fence_before();
  __syncwarp();
  if (C2) cluster_sync();  // neither CTA leaves while the other may still touch its smem or TMEM
  else __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_x<C2>(tmem_base);
  }
}

// Clusters of the pair kernel that fit on the device at once (cached per
// device and instantiation).
template <typename KernelT>
int max_pair_clusters(KernelT k, int threads, uint32_t smem) {
  // Atomic: launches on distinct workspaces may come from several host
  // threads; every thread computes the same value, so the first store wins.
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const int cached = cache[dev].load(std::memory_order_relaxed);
  if (cached > 0) return cached;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess || n <= 0) {
    (void)cudaGetLastError();
    return 0;
  }
  cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

template <int NS, int EPI, bool C2, bool WIDE = false>
cudaError_t launch(const GemmArgs& a, int num_sms, cudaStream_t s) {
  using C = Cfg<NS, EPI, C2, WIDE>;
  static_assert(C::SMEM <= 232448, "shared memory budget");
  auto k = gemm_kernel<NS, EPI, C2, WIDE>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
  if (e != cudaSuccess) return e;
  int units = num_sms;  // CTAs, or CTA pairs, resident at once
  if (C2) {
    units = max_pair_clusters(k, C::THREADS, C::SMEM);
    if (units <= 0) units = num_sms / 2;
  }
  if (a.total_tiles < units) units = a.total_tiles;
  if (units < 1) return cudaSuccess;
  e = cudaMemsetAsync(a.tile_counter, 0, sizeof(int), s);
  if (e != cudaSuccess) return e;
  if (!C2) {
    k<<<units, C::THREADS, C::SMEM, s>>>(a);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(units * 2), 1, 1);
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, a);
}

}  // namespace

// Stages per width: narrow pair tiles 6 x 32 KB (7 without epilogue
// staging), wide pair tiles 3 x 48 KB with 64 KB of staging for eight
// epilogue warps (4 without), one CTA per tile 4 x 48 KB.
#define KD_GEMM_DISPATCH(EPI, NS_NARROW, NS_WIDE)                 \
  if (a.cta2 && a.wide) return launch<NS_WIDE, EPI, true, true>(a, num_sms, s); \
  if (a.cta2) return launch<NS_NARROW, EPI, true, false>(a, num_sms, s);        \
  return launch<4, EPI, false, false>(a, num_sms, s);

cudaError_t launch_logits_fwd(const GemmArgs& a, int num_sms, cudaStream_t s) { KD_GEMM_DISPATCH(EPI_FWD, 7, 4) }
cudaError_t launch_logits_dz(const GemmArgs& a, int num_sms, cudaStream_t s) { KD_GEMM_DISPATCH(EPI_DZ, 6, 3) }
cudaError_t launch_logits_fwd_store(const GemmArgs& a, int num_sms, cudaStream_t s) {
  KD_GEMM_DISPATCH(EPI_FWDST, 6, 3)
}
cudaError_t launch_logits_teacher(const GemmArgs& a, int num_sms, cudaStream_t s) {
  KD_GEMM_DISPATCH(EPI_TEACHER, 6, 3)
}
cudaError_t launch_grad(const GemmArgs& a, int num_sms, cudaStream_t s) { KD_GEMM_DISPATCH(EPI_GRAD, 6, 3) }

#undef KD_GEMM_DISPATCH

}  // namespace kd
