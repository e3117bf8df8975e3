// kd_api.cu - the C ABI of libkd: argument checks, workspace layout, the
// chunk loop of the fused KL loss, and the launches.
//
// The chunk loop is the structure of the "Fused chunked KL" variant ("ทำให้
// Knowledge Distillation มีประสิทธิภาพ..." (ai-thai.com), section "กลไก Fused
// Chunked KL Loss"; "Multiverse Computing сократила видеопамять..."
// (iitog.ru), fourth paragraph). Positions are processed one group of G
// chunks at a time (G = clamp(4096 / chunk, 1, 4), see bwd_group):
//   forward : prep -> logits GEMM with (max, sum, gather) epilogue -> merge
//   backward: prep -> logits GEMM recompute with dz epilogue -> dH + dW GEMMs
//   fwdbwd  : prep -> logits GEMM storing exp(z - m_tile) -> merge -> dz pass
//             -> dH + dW GEMMs
// The only per-group buffers (in the caller's workspace) are O(G * chunk * V):
// the bf16 dz of one group and the per-tile partials. Nothing grows with T
// apart from the caller's own inputs and outputs.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <mutex>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <nvtx3/nvToolsExt.h>

#include "../../include/kd.h"
#include "../../include/kd_profile.h"
#include "../../include/kd_testing.h"
#include "kd_internal.h"

namespace kd {

namespace {

constexpr size_t kHeader = 256;  // status word, counters, fp64 loss accumulator
constexpr size_t kCounterOffset = 64;  // int: tile counter of the GEMM launches
constexpr size_t kAccOffset = 128;
constexpr size_t kDoneOffset = 136;    // unsigned: blocks of the current merge launch that finished
constexpr size_t kScaleOffset = 144;   // float: the backward's per-position gradient factor

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

void load_encode() {
  cudaDriverEntryPointQueryResult q;
  void* fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
          cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

int num_sms_current() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// GEMM tile shape: 1 = CTA-pair tiles (tcgen05 cta_group::2; 256 x 512 or
// 256 x 256, see gemm_wide), 0 = one CTA per 128 x 256 tile.
constexpr int kDefaultCta2 = 1;

// Process-wide switches for tests and measurements (kd_testing.h). -1 keeps
// the default. They are read on the host when a call sets up its launches;
// nothing in the environment changes which kernels a call runs.
std::atomic<int> g_test_cta2{-1};
std::atomic<int> g_test_wide{-1};
std::atomic<int> g_test_force_exact{0};

int gemm_cta2() {
  const int v = g_test_cta2.load(std::memory_order_relaxed);
  return v < 0 ? kDefaultCta2 : v;
}

// Width of the CTA-pair tiles per GEMM, chosen by measurement on B300: wide
// (256 x 512, one accumulator) for every GEMM. The narrow form (256 x 256,
// double-buffered accumulators, so the epilogue overlaps the next tile)
// starves for operands; with the epilogue's TMEM loads double-buffered, the
// wide dz recompute is about 2% faster than the narrow one.
int gemm_wide(int dflt) {
  const int v = g_test_wide.load(std::memory_order_relaxed);
  return v < 0 ? dflt : v;
}

int topk_force_exact() { return g_test_force_exact.load(std::memory_order_relaxed) ? 1 : 0; }

// Chunks per GEMM group. By default up to 4 chunks and about 4096 positions
// per group: the dW tiles then run over a long contraction (G * chunk), so
// their epilogue (the fp32 read-modify-write of the tile, 8 V d bytes per
// group in all) is paid once per group, not once per chunk. A caller that
// sizes `chunk` to bound memory passes group = 1 (kd_kl_options.group). The
// workspace holds the group's dz: O(group * chunk * V).
int64_t bwd_group(int64_t chunk, int64_t group) {
  if (group > 0) return group;
  const int64_t g = 4096 / chunk;
  return g < 1 ? 1 : (g > 4 ? 4 : g);
}

// Fused-loss workspace layout (all offsets 256-byte aligned; dz 1024). One
// layout serves the forward, the backward and the single-call forward +
// backward: the per-position arrays hold one group of chunks (G * chunk
// rows; the separate calls use the first chunk rows of them).
struct Layout {
  int Kp;
  int64_t G;    // chunks per dH/dW group (backward)
  int64_t S;    // vocabulary tiles of the forward GEMM
  int64_t ldz;  // dz row stride in elements
  int64_t ldt;  // row stride of the transposed hidden-state chunk
  size_t ids_sorted, p_sorted, cnt, ent, zK, block_sums, part_m, part_s, hct, dz, total;
};

Layout fused_layout(int64_t d, int64_t V, int K, int64_t chunk, int64_t group) {
  Layout L;
  L.Kp = (K + 3) / 4 * 4;
  L.S = ceil_div(V, kBNLogits);
  L.ldz = align_up((size_t)V, 64);
  L.G = bwd_group(chunk, group);
  L.ldt = align_up((size_t)(L.G * chunk), 64);
  const int64_t prow = L.G * chunk;
  size_t o = kHeader;
  auto take = [&](size_t bytes, size_t al) {
    o = align_up(o, al);
    const size_t r = o;
    o += bytes;
    return r;
  };
  L.ids_sorted = take((size_t)prow * L.Kp * 4, 256);
  L.p_sorted = take((size_t)prow * L.Kp * 4, 256);
  L.cnt = take((size_t)prow * 4, 256);
  L.ent = take((size_t)prow * 4, 256);
  L.zK = take((size_t)prow * L.Kp * 4, 256);
  L.block_sums = take((size_t)ceil_div(prow, 8) * 8, 256);
  L.part_m = take((size_t)L.S * prow * 4, 256);
  L.part_s = take((size_t)L.S * prow * 4, 256);
  L.hct = take((size_t)d * L.ldt * 2, 1024);
  L.dz = take((size_t)(L.G * chunk) * L.ldz * 2, 1024);
  L.total = align_up(o, 256);
  return L;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Teacher-cache workspace: the header, one chunk's fp32 logits
// Z [chunk, round_up(V, 64)] and its per-(position, vocab tile) partials.
struct TeacherLayout {
  int64_t S, ldz;
  size_t z, part_m, part_s, total;
};

TeacherLayout teacher_layout(int64_t V, int64_t chunk) {
  TeacherLayout L;
  L.S = ceil_div(V, kBNLogits);
  L.ldz = align_up((size_t)V, 64);
  size_t o = kHeader;
  o = align_up(o, 1024);
  L.z = o;
  o += (size_t)chunk * L.ldz * 4;
  o = align_up(o, 256);
  L.part_m = o;
  o += (size_t)chunk * L.S * 4;
  o = align_up(o, 256);
  L.part_s = o;
  o += (size_t)chunk * L.S * 4;
  L.total = align_up(o, 256);
  return L;
}

// ------------------------------------------------------------------ profiling
// Kernel names reported by kd_profile_end, indexed by KernelId.
enum KernelId {
  K_TOPK, K_PREP, K_LOGITS_FWD, K_MERGE, K_FINALIZE, K_LOGITS_DZ, K_TRANSPOSE, K_GRAD, K_TEST, K_LOGITS_FWD_STORE,
  K_DZ_FROM_EXP, K_TEACHER_GEMM, K_TILE_TOPK, K_GRAD_SCALE, K_COUNT
};
const char* const kKernelNames[K_COUNT] = {"topk_cache", "teacher_prep", "logits_fwd_lse_gather", "lse_merge_loss",
                                           "loss_finalize", "logits_dz", "hidden_transpose", "grad_dH_dW",
                                           "test_gemm", "logits_fwd_store_exp", "dz_from_exp",
                                           "teacher_logits_gemm", "teacher_tile_topk", "grad_scale"};
struct ProfRec {
  int kid;
  cudaEvent_t a, b;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRec> g_prof_recs;
std::vector<cudaEvent_t> g_prof_pool;

cudaEvent_t prof_event() {
  if (!g_prof_pool.empty()) {
    cudaEvent_t e = g_prof_pool.back();
    g_prof_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Brackets one kernel launch: an NVTX range named after the kernel (a
// pointer check when no tool is attached), and, while profiling is on, an
// event recorded on the launch stream before the launch (constructor) and
// after it (destructor).
struct ProfScope {
  int kid;
  cudaStream_t s;
  cudaEvent_t a = nullptr;
  ProfScope(int k, cudaStream_t st) : kid(k), s(st) {
    nvtxRangePushA(kKernelNames[k]);
    std::lock_guard<std::mutex> g(g_prof_mu);
    if (!g_prof_on) return;
    a = prof_event();
    if (a && cudaEventRecord(a, s) != cudaSuccess) a = nullptr;
  }
  ~ProfScope() {
    if (a) {
      std::lock_guard<std::mutex> g(g_prof_mu);
      cudaEvent_t b = prof_event();
      if (b && cudaEventRecord(b, s) == cudaSuccess) g_prof_recs.push_back({kid, a, b});
    }
    nvtxRangePop();
  }
};

// NVTX range around one call of the C ABI, named after it; the launches of
// the call nest inside it.
struct CallRange {
  explicit CallRange(const char* name) { nvtxRangePushA(name); }
  ~CallRange() { nvtxRangePop(); }
  CallRange(const CallRange&) = delete;
  CallRange& operator=(const CallRange&) = delete;
};

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return KD_OK;
  if (std::getenv("KD_DEBUG")) std::fprintf(stderr, "libkd: CUDA error %s\n", cudaGetErrorString(e));
  return KD_ERR_CUDA;
}

int check_fused_args(const void* H, const void* W, const int32_t* ids, const float* logp, int64_t T, int64_t d,
                     int64_t V, int32_t K, int64_t chunk, int64_t group, void* ws, size_t ws_bytes) {
  if (!H || !W || !ids || !logp || T <= 0 || d <= 0 || V <= 0 || K <= 0 || chunk <= 0) return KD_ERR_INVALID_ARG;
  if (K > V) return KD_ERR_INVALID_ARG;
  if (K > 4096 || V >= (int64_t(1) << 31) || d % 8 != 0 || d > (int64_t(1) << 24) || chunk > (int64_t(1) << 24))
    return KD_ERR_UNSUPPORTED;
  if (bwd_group(chunk, group) * chunk > (int64_t(1) << 24)) return KD_ERR_UNSUPPORTED;
  if (!aligned(H, 16) || !aligned(W, 16)) return KD_ERR_UNSUPPORTED;
  const Layout L = fused_layout(d, V, K, chunk, group);
  if (!ws || !aligned(ws, 256) || ws_bytes < L.total) return KD_ERR_WORKSPACE;
  return KD_OK;
}

}  // namespace

namespace {
cudaError_t encode_map(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                       uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  std::call_once(g_encode_once, load_encode);
  if (!g_encode) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}
}  // namespace

cudaError_t encode_map_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
                          uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  return encode_map(map, dt, base, inner, outer, row_bytes, box_inner, box_outer, CU_TENSOR_MAP_SWIZZLE_128B);
}
cudaError_t encode_map_2d_plain(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
                                uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  return encode_map(map, dt, base, inner, outer, row_bytes, box_inner, box_outer, CU_TENSOR_MAP_SWIZZLE_NONE);
}

namespace {

// dH and dW of one group of positions [g0, g0 + grows) from the group's dz
// (bf16, [grows, ldz] in the workspace): H_g^T into the workspace, then one
// GEMM launch with two problems,
//   dH_g^T = W^T dz^T (stored transposed into dH) and
//   dW (+)= dz^T H_g.
// `ag` carries the tensor maps of W (tmA[0]) and dW (tmC[1]) set up once
// per call. Either output may be absent (dH == NULL, or want_dW == 0): its
// problem then has no tiles (no dW also means no H_g^T).
int grad_group(GemmArgs& ag, const Layout& L, const __nv_bfloat16* Hb, const __nv_bfloat16* dz,
               __nv_bfloat16* hct, void* dH, int dH_bf16, int want_dW, int64_t g0, int grows, int64_t d,
               int64_t V, int reduce_add, int sms, cudaStream_t s) {
  const int TR = gemm_tile_rows(ag.cta2), BR = gemm_b_box_rows(ag.cta2);
  // dW's N runs over d. With wide pair tiles and d a multiple of 480 but not
  // of 512 (d = 2880 at the GPT-OSS shapes), 480-wide tiles (two N = 240
  // MMAs) cover d exactly; 512-wide ones would spend 6.25% of dW's MMAs on
  // padding.
  const bool dw480 = ag.cta2 && ag.wide && d % 512 != 0 && d % 480 == 0;
  cudaError_t e;
  if (want_dW) {
    ProfScope ps(K_TRANSPOSE, s);
    e = launch_transpose(Hb + g0 * d, grows, (int)d, hct, (int)L.ldt, s);
    if (e != cudaSuccess) return cuda_status(e);
  }
  const cudaError_t eh =
      !dH ? cudaSuccess
      : dH_bf16 ? encode_map_2d_plain(&ag.tmC[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                      static_cast<__nv_bfloat16*>(dH) + g0 * d, (uint64_t)d, (uint64_t)grows,
                                      (uint64_t)d * 2, 32, 32)
                : encode_map_2d(&ag.tmC[0], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, static_cast<float*>(dH) + g0 * d,
                                (uint64_t)d, (uint64_t)grows, (uint64_t)d * 4, 32, 32);
  if (eh != cudaSuccess ||
      encode_map_2d(&ag.tmB[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dz, (uint64_t)V, (uint64_t)grows,
                    (uint64_t)L.ldz * 2, kBK, BR) != cudaSuccess ||
      encode_map_2d(&ag.tmA[1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dz, (uint64_t)V, (uint64_t)grows,
                    (uint64_t)L.ldz * 2, 64, 64) != cudaSuccess ||
      encode_map_2d(&ag.tmB[1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, hct, (uint64_t)grows, (uint64_t)d,
                    (uint64_t)L.ldt * 2, kBK, dw480 ? 120 : BR) != cudaSuccess)
    return KD_ERR_UNSUPPORTED;
  Problem& P0 = ag.pr[0];
  P0.m_blocks = dH ? (int)ceil_div(d, TR) : 0;  // no dH: no tiles of this problem
  P0.n_blocks = (int)ceil_div(grows, gemm_tile_cols(ag.cta2, ag.wide));
  P0.k_blocks = (int)ceil_div(V, kBK);
  P0.a_mn = 1; P0.b_mn = 0; P0.M = (int)d; P0.N = grows;
  P0.tile_begin = 0; P0.n_fastest = 0; P0.reduce_add = 0; P0.c_trans = 1; P0.out_bf16 = dH_bf16;
  P0.bnh = 256;
  Problem& P1 = ag.pr[1];
  P1.m_blocks = (int)ceil_div(V, TR);
  P1.n_blocks = (int)(dw480 ? d / 480 : ceil_div(d, gemm_tile_cols(ag.cta2, ag.wide)));
  P1.bnh = dw480 ? 240 : 256;
  P1.k_blocks = (int)ceil_div(grows, kBK);
  P1.a_mn = 1; P1.b_mn = 0; P1.M = (int)V; P1.N = (int)d;
  P1.tile_begin = P0.m_blocks * P0.n_blocks; P1.n_fastest = 1;
  P1.reduce_add = reduce_add;
  P1.c_trans = 0; P1.out_bf16 = 0;
  ag.nprob = want_dW ? 2 : 1;
  ag.total_tiles = want_dW ? P1.tile_begin + P1.m_blocks * P1.n_blocks : P1.tile_begin;
  {
    ProfScope ps(K_GRAD, s);
    e = launch_grad(ag, sms, s);
  }
  return cuda_status(e);
}

// Tensor maps of W (M-major A of the dH^T problem) and dW (C of the dW
// problem; none when dW is not wanted), shared by every group of a call.
int grad_setup(GemmArgs& ag, const void* W, float* dW, int64_t d, int64_t V, int* status, int* counter) {
  std::memset(&ag, 0, sizeof(ag));
  ag.cta2 = gemm_cta2();
  ag.wide = gemm_wide(1);
  ag.status = status;
  ag.tile_counter = counter;
  if (encode_map_2d(&ag.tmA[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, (uint64_t)d, (uint64_t)V, (uint64_t)d * 2, 64,
                    64) != cudaSuccess)
    return KD_ERR_UNSUPPORTED;
  if (dW && (encode_map_2d(&ag.tmC[1], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dW, (uint64_t)d, (uint64_t)V, (uint64_t)d * 4,
                           32, 32) != cudaSuccess ||
             encode_map_2d_plain(&ag.tmCt[1], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dW, (uint64_t)d, (uint64_t)V,
                                 (uint64_t)d * 4, 16, 32) != cudaSuccess))
    return KD_ERR_UNSUPPORTED;
  return KD_OK;
}

// Loss options of the _ex calls, validated (NULL = the plain calls).
struct LossOpts {
  float inv_tau = 1.f;
  const uint8_t* mask = nullptr;
  int mean_over_mask = 0;
  int dH_bf16 = 0;
  int64_t group = 0;  // chunks per GEMM group; 0 = the default rule (bwd_group)
};

int parse_opts(const kd_kl_options* o, LossOpts* out) {
  LossOpts r;
  if (o) {
    if (!(o->temperature > 0.f) || !std::isfinite(o->temperature) || !std::isfinite(1.f / o->temperature))
      return KD_ERR_INVALID_ARG;
    if ((o->mean_over_mask != 0 && o->mean_over_mask != 1) || (o->dH_bf16 != 0 && o->dH_bf16 != 1) ||
        o->group < 0)
      return KD_ERR_INVALID_ARG;
    r.inv_tau = 1.f / o->temperature;
    r.mask = o->mask;
    r.mean_over_mask = o->mean_over_mask;
    r.dH_bf16 = o->dH_bf16;
    r.group = o->group;
  }
  *out = r;
  return KD_OK;
}

const uint8_t* mask_at(const LossOpts& o, int64_t row0) { return o.mask ? o.mask + row0 : nullptr; }

// Typed views of the fused-loss workspace (header words and the per-group
// buffers of fused_layout).
struct FusedWs {
  int* status;
  int* counter;   // tile counter of the GEMM launches
  double* acc;    // fp64 loss accumulator
  unsigned* done; // finished blocks of the current merge launch
  float* scale;   // the backward's per-position gradient factor
  int* ids_sorted;
  float* p_sorted;
  int* cnt;
  float* ent;
  float* zK;
  double* bsum;
  float* part_m;
  float* part_s;
  __nv_bfloat16* dz;
  __nv_bfloat16* hct;
};

FusedWs fused_ws(void* ws, const Layout& L) {
  uint8_t* w = static_cast<uint8_t*>(ws);
  FusedWs f;
  f.status = reinterpret_cast<int*>(w);
  f.counter = reinterpret_cast<int*>(w + kCounterOffset);
  f.acc = reinterpret_cast<double*>(w + kAccOffset);
  f.done = reinterpret_cast<unsigned*>(w + kDoneOffset);
  f.scale = reinterpret_cast<float*>(w + kScaleOffset);
  f.ids_sorted = reinterpret_cast<int*>(w + L.ids_sorted);
  f.p_sorted = reinterpret_cast<float*>(w + L.p_sorted);
  f.cnt = reinterpret_cast<int*>(w + L.cnt);
  f.ent = reinterpret_cast<float*>(w + L.ent);
  f.zK = reinterpret_cast<float*>(w + L.zK);
  f.bsum = reinterpret_cast<double*>(w + L.block_sums);
  f.part_m = reinterpret_cast<float*>(w + L.part_m);
  f.part_s = reinterpret_cast<float*>(w + L.part_s);
  f.dz = reinterpret_cast<__nv_bfloat16*>(w + L.dz);
  f.hct = reinterpret_cast<__nv_bfloat16*>(w + L.hct);
  return f;
}

// The logits GEMM z = H_g W^T of a call: tile shape and width (the default
// for this GEMM, unless KD_GEMM_WIDE forces one), 1/tau for the epilogue,
// and the tensor map of W (K-major B), shared by every group.
int logits_setup(GemmArgs& a, int wide_default, float inv_tau, const void* W, int64_t d, int64_t V) {
  std::memset(&a, 0, sizeof(a));
  a.cta2 = gemm_cta2();
  a.wide = gemm_wide(wide_default);
  a.zscale = inv_tau;
  if (encode_map_2d(&a.tmB[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, (uint64_t)d, (uint64_t)V, (uint64_t)d * 2, kBK,
                    gemm_b_box_rows(a.cta2)) != cudaSuccess)
    return KD_ERR_UNSUPPORTED;
  return KD_OK;
}

// The logits GEMM of one group of positions [g0, g0 + rows): the tensor map
// of the group's H rows (K-major A), that of the dz buffer when the epilogue
// stores a tile (store_dz), the problem shape, and the teacher-side arrays
// and partial-statistics buffers the epilogues read or write.
int logits_group(GemmArgs& a, const Layout& L, const FusedWs& f, const __nv_bfloat16* Hb, int64_t g0, int rows,
                 int64_t d, int64_t V, bool store_dz) {
  if (encode_map_2d(&a.tmA[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Hb + g0 * d, (uint64_t)d, (uint64_t)rows,
                    (uint64_t)d * 2, kBK, kBM) != cudaSuccess)
    return KD_ERR_UNSUPPORTED;
  if (store_dz && encode_map_2d(&a.tmC[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, f.dz, (uint64_t)V, (uint64_t)rows,
                                (uint64_t)L.ldz * 2, 64, 32) != cudaSuccess)
    return KD_ERR_UNSUPPORTED;
  Problem& P = a.pr[0];
  P.m_blocks = (int)ceil_div(rows, gemm_tile_rows(a.cta2));
  P.n_blocks = (int)ceil_div(V, gemm_tile_cols(a.cta2, a.wide));
  P.k_blocks = (int)ceil_div(d, kBK);
  P.a_mn = 0; P.b_mn = 0; P.M = rows; P.N = (int)V;
  P.tile_begin = 0; P.n_fastest = 0; P.reduce_add = 0; P.c_trans = 0;
  a.nprob = 1;
  a.total_tiles = P.m_blocks * P.n_blocks;
  a.rows = rows; a.S = (int)L.S; a.V = (int)V; a.Kp = L.Kp;
  a.ids_sorted = f.ids_sorted; a.p_sorted = f.p_sorted; a.cnt = f.cnt;
  a.zK = f.zK; a.part_m = f.part_m; a.part_s = f.part_s;
  a.status = f.status;
  a.tile_counter = f.counter;
  return KD_OK;
}

// Teacher side of one group: p renormalised over K (with 1/tau), entropy,
// and the (id, p) list sorted by id.
cudaError_t prep_group(const int32_t* ids, const float* logp, int64_t g0, int rows, int32_t K, int64_t V,
                       const Layout& L, float inv_tau, const FusedWs& f, cudaStream_t s) {
  ProfScope ps(K_PREP, s);
  return launch_prep(ids + g0 * K, logp + g0 * K, rows, K, (int)V, L.Kp, inv_tau, f.ids_sorted, f.p_sorted, f.cnt,
                     f.ent, f.status, s);
}

}  // namespace

// Argument checks of kd_topk_cache other than the workspace: null pointers,
// sizes, dtype, alignment and the kernel's shared-memory limit.
int topk_check_args(const void* logits, int dtype, int64_t T, int64_t V, int64_t ld, int K, const void* ids,
                    const void* logp) {
  if (!logits || !ids || !logp || T <= 0 || V <= 0 || K <= 0 || K > V || ld < V) return KD_ERR_INVALID_ARG;
  if (dtype != KD_BF16 && dtype != KD_F32) return KD_ERR_INVALID_ARG;
  if (V >= (int64_t(1) << 31) || K > 65536) return KD_ERR_UNSUPPORTED;
  if (!aligned(logits, dtype == KD_BF16 ? 2 : 4)) return KD_ERR_UNSUPPORTED;
  if (topk_smem_bytes(K) > 200 * 1024) return KD_ERR_UNSUPPORTED;
  return KD_OK;
}

}  // namespace kd

using namespace kd;

extern "C" {

const char* kd_status_string(int status) {
  switch (status) {
    case KD_OK: return "KD_OK";
    case KD_ERR_INVALID_ARG: return "KD_ERR_INVALID_ARG";
    case KD_ERR_UNSUPPORTED: return "KD_ERR_UNSUPPORTED";
    case KD_ERR_WORKSPACE: return "KD_ERR_WORKSPACE";
    case KD_ERR_CUDA: return "KD_ERR_CUDA";
    case KD_ERR_DEVICE_TIMEOUT: return "KD_ERR_DEVICE_TIMEOUT";
    case KD_ERR_BAD_ID: return "KD_ERR_BAD_ID";
    case KD_ERR_IO: return "KD_ERR_IO";
    case KD_ERR_FORMAT: return "KD_ERR_FORMAT";
    default: return "KD_ERR_UNKNOWN";
  }
}

int kd_version(void) { return 110; }

size_t kd_topk_workspace_size(int64_t T, int64_t V, int32_t K, int32_t dtype) {
  (void)T; (void)V; (void)K; (void)dtype;
  return kHeader;
}

int kd_topk_cache(const void* logits, int32_t dtype, int64_t T, int64_t V, int64_t ld, int32_t K, int32_t* ids,
                  float* logp, void* ws, size_t ws_bytes, void* stream) {
  CallRange call_range("kd_topk_cache");
  const int chk = topk_check_args(logits, dtype, T, V, ld, K, ids, logp);
  if (chk != KD_OK) return chk;
  if (!ws || !aligned(ws, 256) || ws_bytes < kHeader) return KD_ERR_WORKSPACE;
  const int sms = num_sms_current();
  if (sms <= 0) return KD_ERR_CUDA;
  const int force = topk_force_exact();
  ProfScope ps(K_TOPK, static_cast<cudaStream_t>(stream));
  return cuda_status(launch_topk(logits, dtype, T, V, ld, K, ids, logp, static_cast<int*>(ws), force, sms,
                                 static_cast<cudaStream_t>(stream)));
}

size_t kd_fused_kl_workspace_size_ex(int64_t d, int64_t V, int32_t K, int64_t chunk, int32_t group) {
  if (d <= 0 || V <= 0 || K <= 0 || chunk <= 0 || group < 0) return 0;
  // Sizes the calls refuse get no workspace size either (and the layout
  // arithmetic stays far from overflow).
  if (K > 4096 || K > V || V >= (int64_t(1) << 31) || d > (int64_t(1) << 24) || chunk > (int64_t(1) << 24) ||
      bwd_group(chunk, group) * chunk > (int64_t(1) << 24))
    return 0;
  return fused_layout(d, V, K, chunk, group).total;
}

size_t kd_fused_kl_workspace_size(int64_t d, int64_t V, int32_t K, int64_t chunk) {
  return kd_fused_kl_workspace_size_ex(d, V, K, chunk, 0);
}

int kd_fused_kl_fwd_ex(const void* H, const void* W, const int32_t* ids, const float* logp, int64_t T, int64_t d,
                       int64_t V, int32_t K, int64_t chunk, float* loss, float* lse, float* loss_rows,
                       const kd_kl_options* opt, void* ws, size_t ws_bytes, void* stream) {
  CallRange call_range("kd_fused_kl_fwd");
  LossOpts o;
  int st = parse_opts(opt, &o);
  if (st != KD_OK) return st;
  st = check_fused_args(H, W, ids, logp, T, d, V, K, chunk, o.group, ws, ws_bytes);
  if (st != KD_OK) return st;
  if (!loss || !lse) return KD_ERR_INVALID_ARG;
  const int sms = num_sms_current();
  if (sms <= 0) return KD_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Layout L = fused_layout(d, V, K, chunk, o.group);
  const FusedWs f = fused_ws(ws, L);
  const __nv_bfloat16* Hb = static_cast<const __nv_bfloat16*>(H);
  // The merge kernels count finished blocks in the workspace header; the
  // count returns to 0 after every launch, and starts there for this call.
  cudaError_t e = cudaMemsetAsync(f.done, 0, sizeof(unsigned), s);
  if (e != cudaSuccess) return cuda_status(e);

  GemmArgs a;
  if ((st = logits_setup(a, 1, o.inv_tau, W, d, V)) != KD_OK) return st;
  // Positions go through in groups of G chunks (one GEMM launch per group:
  // more tiles per launch, fewer launches; the group is the unit the
  // workspace is sized for).
  const int64_t gchunk = L.G * chunk;
  for (int64_t c0 = 0; c0 < T; c0 += gchunk) {
    const int rows = (int)((T - c0) < gchunk ? (T - c0) : gchunk);
    e = prep_group(ids, logp, c0, rows, K, V, L, o.inv_tau, f, s);
    if (e != cudaSuccess) return cuda_status(e);
    if ((st = logits_group(a, L, f, Hb, c0, rows, d, V, false)) != KD_OK) return st;
    {
      ProfScope ps(K_LOGITS_FWD, s);
      e = launch_logits_fwd(a, sms, s);
    }
    if (e != cudaSuccess) return cuda_status(e);
    {
      ProfScope ps(K_MERGE, s);
      e = launch_merge(f.part_m, f.part_s, (int)L.S, rows, f.ent, f.p_sorted, f.zK, f.cnt, L.Kp, mask_at(o, c0),
                       lse + c0, loss_rows ? loss_rows + c0 : nullptr, f.bsum, f.done, f.acc, c0 == 0, s);
    }
    if (e != cudaSuccess) return cuda_status(e);
  }
  ProfScope ps(K_FINALIZE, s);
  return cuda_status(launch_finalize(f.acc, T, o.mask, o.mean_over_mask, loss, s));
}

int kd_fused_kl_fwd(const void* H, const void* W, const int32_t* ids, const float* logp, int64_t T, int64_t d,
                    int64_t V, int32_t K, int64_t chunk, float* loss, float* lse, float* loss_rows, void* ws,
                    size_t ws_bytes, void* stream) {
  return kd_fused_kl_fwd_ex(H, W, ids, logp, T, d, V, K, chunk, loss, lse, loss_rows, nullptr, ws, ws_bytes, stream);
}

int kd_fused_kl_bwd_ex(const void* H, const void* W, const int32_t* ids, const float* logp, const float* lse,
                       int64_t T, int64_t d, int64_t V, int32_t K, int64_t chunk, float grad_scale,
                       const float* grad_scale_dev, void* dH, float* dW, int32_t accumulate_dW,
                       const kd_kl_options* opt, void* ws, size_t ws_bytes, void* stream) {
  CallRange call_range("kd_fused_kl_bwd");
  LossOpts o;
  int st = parse_opts(opt, &o);
  if (st != KD_OK) return st;
  st = check_fused_args(H, W, ids, logp, T, d, V, K, chunk, o.group, ws, ws_bytes);
  if (st != KD_OK) return st;
  if (!lse || (!dH && !dW)) return KD_ERR_INVALID_ARG;
  if ((dH && !aligned(dH, 16)) || (dW && !aligned(dW, 16))) return KD_ERR_UNSUPPORTED;
  const int sms = num_sms_current();
  if (sms <= 0) return KD_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Layout L = fused_layout(d, V, K, chunk, o.group);
  const FusedWs f = fused_ws(ws, L);
  const __nv_bfloat16* Hb = static_cast<const __nv_bfloat16*>(H);

  // s = grad_scale * (*grad_scale_dev) * 1/tau (* 1/N), on the device.
  cudaError_t e;
  {
    ProfScope ps(K_GRAD_SCALE, s);
    e = launch_grad_scale(grad_scale, grad_scale_dev, o.inv_tau, o.mask, T, o.mean_over_mask, f.scale, s);
  }
  if (e != cudaSuccess) return cuda_status(e);
  // W: K-major B of the logits GEMM, M-major A of the dH^T GEMM.
  GemmArgs az, ag;
  if ((st = logits_setup(az, 1, o.inv_tau, W, d, V)) != KD_OK) return st;
  if ((st = grad_setup(ag, W, dW, d, V, f.status, f.counter)) != KD_OK) return st;

  // One group of G chunks at a time: prep, the recompute GEMM writing the
  // group's dz, then dH and dW of the group.
  const int64_t gchunk = L.G * chunk;
  for (int64_t g0 = 0; g0 < T; g0 += gchunk) {
    const int grows = (int)((T - g0) < gchunk ? (T - g0) : gchunk);
    e = prep_group(ids, logp, g0, grows, K, V, L, o.inv_tau, f, s);
    if (e != cudaSuccess) return cuda_status(e);
    // Recompute the group's logits; the epilogue writes dz (bf16).
    if ((st = logits_group(az, L, f, Hb, g0, grows, d, V, true)) != KD_OK) return st;
    az.lse = lse + g0; az.scale = 1.f; az.dscale = f.scale;
    az.mask = mask_at(o, g0);
    {
      ProfScope ps(K_LOGITS_DZ, s);
      e = launch_logits_dz(az, sms, s);
    }
    if (e != cudaSuccess) return cuda_status(e);
    st = grad_group(ag, L, Hb, f.dz, f.hct, dH, o.dH_bf16, dW != nullptr, g0, grows, d, V,
                    (accumulate_dW || g0 > 0) ? 1 : 0, sms,
                    s);
    if (st != KD_OK) return st;
  }
  return KD_OK;
}

int kd_fused_kl_bwd(const void* H, const void* W, const int32_t* ids, const float* logp, const float* lse,
                    int64_t T, int64_t d, int64_t V, int32_t K, int64_t chunk, float grad_scale,
                    const float* grad_scale_dev, float* dH, float* dW, int32_t accumulate_dW, void* ws,
                    size_t ws_bytes, void* stream) {
  return kd_fused_kl_bwd_ex(H, W, ids, logp, lse, T, d, V, K, chunk, grad_scale, grad_scale_dev, dH, dW,
                            accumulate_dW, nullptr, ws, ws_bytes, stream);
}

int kd_fused_kl_fwdbwd_ex(const void* H, const void* W, const int32_t* ids, const float* logp, int64_t T, int64_t d,
                          int64_t V, int32_t K, int64_t chunk, float grad_scale, const float* grad_scale_dev,
                          float* loss, float* lse, float* loss_rows, void* dH, float* dW, int32_t accumulate_dW,
                          const kd_kl_options* opt, void* ws, size_t ws_bytes, void* stream) {
  CallRange call_range("kd_fused_kl_fwdbwd");
  LossOpts o;
  int st = parse_opts(opt, &o);
  if (st != KD_OK) return st;
  st = check_fused_args(H, W, ids, logp, T, d, V, K, chunk, o.group, ws, ws_bytes);
  if (st != KD_OK) return st;
  if (!loss || !lse || (!dH && !dW)) return KD_ERR_INVALID_ARG;
  if ((dH && !aligned(dH, 16)) || (dW && !aligned(dW, 16))) return KD_ERR_UNSUPPORTED;
  const int sms = num_sms_current();
  if (sms <= 0) return KD_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Layout L = fused_layout(d, V, K, chunk, o.group);
  const FusedWs f = fused_ws(ws, L);
  const __nv_bfloat16* Hb = static_cast<const __nv_bfloat16*>(H);
  cudaError_t e = cudaMemsetAsync(f.done, 0, sizeof(unsigned), s);
  if (e != cudaSuccess) return cuda_status(e);
  {
    ProfScope ps(K_GRAD_SCALE, s);
    e = launch_grad_scale(grad_scale, grad_scale_dev, o.inv_tau, o.mask, T, o.mean_over_mask, f.scale, s);
  }
  if (e != cudaSuccess) return cuda_status(e);

  GemmArgs a, ag;
  if ((st = logits_setup(a, 1, o.inv_tau, W, d, V)) != KD_OK) return st;
  if ((st = grad_setup(ag, W, dW, d, V, f.status, f.counter)) != KD_OK) return st;

  // One group of G chunks at a time: the group's logits are computed once,
  // and kept only as e = exp((z - m_tile) / tau) (bf16, in the dz buffer)
  // until the group's lse is known.
  const int64_t gchunk = L.G * chunk;
  for (int64_t g0 = 0; g0 < T; g0 += gchunk) {
    const int grows = (int)((T - g0) < gchunk ? (T - g0) : gchunk);
    e = prep_group(ids, logp, g0, grows, K, V, L, o.inv_tau, f, s);
    if (e != cudaSuccess) return cuda_status(e);
    if ((st = logits_group(a, L, f, Hb, g0, grows, d, V, true)) != KD_OK) return st;
    {
      ProfScope ps(K_LOGITS_FWD_STORE, s);
      e = launch_logits_fwd_store(a, sms, s);
    }
    if (e != cudaSuccess) return cuda_status(e);
    {
      ProfScope ps(K_MERGE, s);
      e = launch_merge(f.part_m, f.part_s, (int)L.S, grows, f.ent, f.p_sorted, f.zK, f.cnt, L.Kp, mask_at(o, g0),
                       lse + g0, loss_rows ? loss_rows + g0 : nullptr, f.bsum, f.done, f.acc, g0 == 0, s);
    }
    if (e != cudaSuccess) return cuda_status(e);
    {
      ProfScope ps(K_DZ_FROM_EXP, s);
      e = launch_dz_from_exp(f.dz, L.ldz, (int)V, (int)L.S, grows, f.part_m, lse + g0, f.ids_sorted, f.p_sorted,
                             f.zK, f.cnt, L.Kp, 1.f, f.scale, mask_at(o, g0), s);
    }
    if (e != cudaSuccess) return cuda_status(e);
    st = grad_group(ag, L, Hb, f.dz, f.hct, dH, o.dH_bf16, dW != nullptr, g0, grows, d, V,
                    (accumulate_dW || g0 > 0) ? 1 : 0, sms,
                    s);
    if (st != KD_OK) return st;
  }
  ProfScope ps(K_FINALIZE, s);
  return cuda_status(launch_finalize(f.acc, T, o.mask, o.mean_over_mask, loss, s));
}

int kd_fused_kl_fwdbwd(const void* H, const void* W, const int32_t* ids, const float* logp, int64_t T, int64_t d,
                       int64_t V, int32_t K, int64_t chunk, float grad_scale, const float* grad_scale_dev,
                       float* loss, float* lse, float* loss_rows, float* dH, float* dW, int32_t accumulate_dW,
                       void* ws, size_t ws_bytes, void* stream) {
  return kd_fused_kl_fwdbwd_ex(H, W, ids, logp, T, d, V, K, chunk, grad_scale, grad_scale_dev, loss, lse, loss_rows,
                               dH, dW, accumulate_dW, nullptr, ws, ws_bytes, stream);
}

size_t kd_teacher_topk_workspace_size(int64_t d, int64_t V, int32_t K, int64_t chunk) {
  if (d <= 0 || V <= 0 || K <= 0 || chunk <= 0) return 0;
  if (K > V || K > 65536 || V >= (int64_t(1) << 31) || d > (int64_t(1) << 24) || chunk > (int64_t(1) << 24))
    return 0;
  return teacher_layout(V, chunk).total;
}

int kd_teacher_topk_cache(const void* H, const void* W, int64_t T, int64_t d, int64_t V, int32_t K, int64_t chunk,
                          int32_t* ids, float* logp, void* ws, size_t ws_bytes, void* stream) {
  CallRange call_range("kd_teacher_topk_cache");
  if (!H || !W || !ids || !logp || T <= 0 || d <= 0 || V <= 0 || K <= 0 || chunk <= 0 || K > V)
    return KD_ERR_INVALID_ARG;
  if (V >= (int64_t(1) << 31) || K > 65536 || d % 8 != 0 || d > (int64_t(1) << 24) || chunk > (int64_t(1) << 24))
    return KD_ERR_UNSUPPORTED;
  if (!aligned(H, 16) || !aligned(W, 16)) return KD_ERR_UNSUPPORTED;
  if (tile_topk_smem_bytes(K) > 200 * 1024) return KD_ERR_UNSUPPORTED;
  const TeacherLayout L = teacher_layout(V, chunk);
  if (!ws || !aligned(ws, 256) || ws_bytes < L.total) return KD_ERR_WORKSPACE;
  const int sms = num_sms_current();
  if (sms <= 0) return KD_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  int* words = reinterpret_cast<int*>(w);
  float* Z = reinterpret_cast<float*>(w + L.z);
  float* part_m = reinterpret_cast<float*>(w + L.part_m);
  float* part_s = reinterpret_cast<float*>(w + L.part_s);
  const __nv_bfloat16* Hb = static_cast<const __nv_bfloat16*>(H);
  const int force = topk_force_exact();

  GemmArgs a;
  std::memset(&a, 0, sizeof(a));
  a.cta2 = gemm_cta2();
  a.wide = gemm_wide(1);
  a.zscale = 1.f;
  const int TR = gemm_tile_rows(a.cta2), BR = gemm_b_box_rows(a.cta2);
  if (encode_map_2d(&a.tmB[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, (uint64_t)d, (uint64_t)V, (uint64_t)d * 2, kBK,
                    BR) != cudaSuccess)
    return KD_ERR_UNSUPPORTED;
  for (int64_t c0 = 0; c0 < T; c0 += chunk) {
    const int rows = (int)((T - c0) < chunk ? (T - c0) : chunk);
    if (encode_map_2d(&a.tmA[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Hb + c0 * d, (uint64_t)d, (uint64_t)rows,
                      (uint64_t)d * 2, kBK, kBM) != cudaSuccess ||
        encode_map_2d(&a.tmC[0], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, Z, (uint64_t)V, (uint64_t)rows, (uint64_t)L.ldz * 4,
                      32, 32) != cudaSuccess)
      return KD_ERR_UNSUPPORTED;
    Problem& P = a.pr[0];
    P.m_blocks = (int)ceil_div(rows, TR);
    P.n_blocks = (int)ceil_div(V, gemm_tile_cols(a.cta2, a.wide));
    P.k_blocks = (int)ceil_div(d, kBK);
    P.a_mn = 0; P.b_mn = 0; P.M = rows; P.N = (int)V;
    P.tile_begin = 0; P.n_fastest = 0; P.reduce_add = 0; P.c_trans = 0;
    a.nprob = 1;
    a.total_tiles = P.m_blocks * P.n_blocks;
    a.rows = rows; a.S = (int)L.S; a.V = (int)V;
    a.part_m = part_m; a.part_s = part_s;
    a.status = words;
    a.tile_counter = reinterpret_cast<int*>(w + kCounterOffset);
    cudaError_t e;
    {
      ProfScope ps(K_TEACHER_GEMM, s);
      e = launch_logits_teacher(a, sms, s);
    }
    if (e != cudaSuccess) return cuda_status(e);
    {
      ProfScope ps(K_TILE_TOPK, s);
      e = launch_tile_topk(Z, L.ldz, rows, (int)V, (int)L.S, part_m, part_s, K, ids + c0 * K, logp + c0 * K, words,
                           force, s);
    }
    if (e != cudaSuccess) return cuda_status(e);
  }
  return KD_OK;
}

int kd_read_device_status(void* ws, void* stream) {
  if (!ws) return KD_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Read, then clear, in the order of `stream` (after the work that may have
  // set the word), and wait for that stream alone.
  int v = 0;
  if (cudaMemcpyAsync(&v, ws, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return KD_ERR_CUDA;
  if (cudaMemsetAsync(ws, 0, sizeof(int), s) != cudaSuccess) return KD_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return KD_ERR_CUDA;
  return v;
}

int kd_test_set_gemm_tiles(int32_t cta2, int32_t wide) {
  if (cta2 < -1 || cta2 > 1 || wide < -1 || wide > 1) return KD_ERR_INVALID_ARG;
  g_test_cta2.store(cta2, std::memory_order_relaxed);
  g_test_wide.store(wide, std::memory_order_relaxed);
  return KD_OK;
}

int kd_test_get_gemm_tiles(int32_t* cta2, int32_t* wide) {
  if (!cta2 || !wide) return KD_ERR_INVALID_ARG;
  *cta2 = g_test_cta2.load(std::memory_order_relaxed);
  *wide = g_test_wide.load(std::memory_order_relaxed);
  return KD_OK;
}

int kd_test_set_topk_force_exact(int32_t on) {
  if (on != 0 && on != 1) return KD_ERR_INVALID_ARG;
  g_test_force_exact.store(on, std::memory_order_relaxed);
  return KD_OK;
}

int kd_test_wait_timeout(int64_t limit_ns, void* ws, void* stream) {
  if (!ws || limit_ns <= 0 || limit_ns > 10000000000ll) return KD_ERR_INVALID_ARG;
  return cuda_status(launch_wait_timeout((uint64_t)limit_ns, static_cast<int*>(ws), static_cast<cudaStream_t>(stream)));
}

int kd_test_gemm(const void* A, const void* B, float* C, int64_t M, int64_t N, int64_t K, int32_t a_mn,
                 int32_t b_mn, int32_t flags, void* ws, void* stream) {
  if (!A || !B || !C || !ws || M <= 0 || N <= 0 || K <= 0) return KD_ERR_INVALID_ARG;
  const int reduce_add = flags & 1, c_trans = (flags >> 1) & 1, cta2 = (flags >> 2) & 1, wide = (flags >> 3) & 1;
  const int n240 = (flags >> 4) & 1;  // 480-wide pair tiles (two N = 240 MMAs)
  const int64_t ldc = c_trans ? M : N;  // C is [M, N], or [N, M] when stored transposed
  if (K % 8 || (a_mn && M % 8) || (b_mn && N % 8) || ldc % 4) return KD_ERR_UNSUPPORTED;
  if (cta2 && b_mn) return KD_ERR_UNSUPPORTED;  // the pair tiles read a K-major B only
  if (n240 && (!cta2 || !wide || c_trans)) return KD_ERR_UNSUPPORTED;  // wide pair tiles, plain C only
  if (M >= (1 << 30) || N >= (1 << 30) || K >= (1 << 30)) return KD_ERR_UNSUPPORTED;
  const int sms = num_sms_current();
  if (sms <= 0) return KD_ERR_CUDA;
  GemmArgs a;
  std::memset(&a, 0, sizeof(a));
  cudaError_t e1 = a_mn ? encode_map_2d(&a.tmA[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A, M, K, M * 2, 64, 64)
                        : encode_map_2d(&a.tmA[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A, K, M, K * 2, kBK, kBM);
  cudaError_t e2 = b_mn ? encode_map_2d(&a.tmB[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, B, N, K, N * 2, 64, 64)
                        : encode_map_2d(&a.tmB[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, B, K, N, K * 2, kBK,
                                        n240 ? 120 : gemm_b_box_rows(cta2));
  cudaError_t e3 = c_trans ? encode_map_2d(&a.tmC[0], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, C, M, N, M * 4, 32, 32)
                           : encode_map_2d(&a.tmC[0], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, C, N, M, N * 4, 32, 32);
  if (e1 != cudaSuccess || e2 != cudaSuccess || e3 != cudaSuccess) return KD_ERR_UNSUPPORTED;
  if (n240 && encode_map_2d_plain(&a.tmCt[0], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, C, N, M, N * 4, 16, 32) != cudaSuccess)
    return KD_ERR_UNSUPPORTED;
  a.cta2 = cta2;
  a.wide = wide;
  a.zscale = 1.f;
  Problem& P = a.pr[0];
  P.m_blocks = (int)ceil_div(M, gemm_tile_rows(cta2));
  P.n_blocks = (int)ceil_div(N, n240 ? 480 : gemm_tile_cols(cta2, wide));
  P.k_blocks = (int)ceil_div(K, kBK);
  P.bnh = n240 ? 240 : 256;
  P.a_mn = a_mn ? 1 : 0; P.b_mn = b_mn ? 1 : 0;
  P.M = (int)M; P.N = (int)N;
  P.tile_begin = 0; P.n_fastest = 0; P.reduce_add = reduce_add; P.c_trans = c_trans;
  a.nprob = 1;
  a.total_tiles = P.m_blocks * P.n_blocks;
  a.status = static_cast<int*>(ws);
  a.tile_counter = reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + kCounterOffset);
  ProfScope ps(K_TEST, static_cast<cudaStream_t>(stream));
  return cuda_status(launch_grad(a, sms, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

extern "C" {

int kd_profile_begin(void) {
  std::lock_guard<std::mutex> g(g_prof_mu);
  for (auto& r : g_prof_recs) {
    g_prof_pool.push_back(r.a);
    g_prof_pool.push_back(r.b);
  }
  g_prof_recs.clear();
  g_prof_on = true;
  return KD_OK;
}

int kd_profile_end(kd_prof_entry* out, int32_t max_entries, int32_t* n_out) {
  std::lock_guard<std::mutex> g(g_prof_mu);
  g_prof_on = false;
  int launches[K_COUNT] = {0};
  double ms[K_COUNT] = {0.0};
  int rc = KD_OK;
  for (auto& r : g_prof_recs) {
    float t = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) {
      rc = KD_ERR_CUDA;
    } else {
      launches[r.kid] += 1;
      ms[r.kid] += t;
    }
    g_prof_pool.push_back(r.a);
    g_prof_pool.push_back(r.b);
  }
  g_prof_recs.clear();
  int n = 0;
  for (int k = 0; k < K_COUNT; ++k) {
    if (!launches[k]) continue;
    if (out && n < max_entries) {
      std::memset(out[n].name, 0, sizeof(out[n].name));
      std::strncpy(out[n].name, kKernelNames[k], sizeof(out[n].name) - 1);
      out[n].launches = launches[k];
      out[n].total_ms = ms[k];
      ++n;
    }
  }
  if (n_out) *n_out = n;
  return rc;
}

}  // extern "C"
