/*
 * kd.h - C ABI of libkd: offline top-K knowledge distillation on one B300.
 *
 * Two operations, both from the method "Efficient Knowledge Distillation for
 * LLMs: Offline Top-K Logits and a Fused Chunked KL Loss" as described on
 * the pages:
 *   [KD-TH] "ทำให้ Knowledge Distillation มีประสิทธิภาพ คุ้มค่า และใช้งานได้จริงใน
 *           ระดับ Scale ใหญ่" (ai-thai.com)
 *   [KD-RU] "Multiverse Computing сократила видеопамять для дистилляции
 *           нейросетей до 15,6 раза" (iitog.ru)
 *   [KD-TA] "பெரிய மொழி மாதிரிகளைச் சுருக்குதல்: ஒற்றை GPU-க்குள் நினைவகத்தைக்
 *           கொண்டு வரும் புதிய முறை" (scitechpulse.com)
 *
 *  1. kd_topk_cache: the offline teacher cache. Teacher logits become the K
 *     most probable token ids per position plus their full-vocabulary
 *     log-softmax values ([KD-TH] section "การทำ Distillation แบบ Offline";
 *     [KD-RU] fourth paragraph).
 *  2. kd_fused_kl_fwd / kd_fused_kl_bwd: the fused chunked KL loss. The
 *     student's final projection z = H W^T is folded into the loss and
 *     computed chunk by chunk of positions, so the T x V logit matrix never
 *     exists. The backward pass recomputes each chunk instead of storing it
 *     ([KD-TH] section "กลไก Fused Chunked KL Loss", variant "Fused chunked KL";
 *     [KD-TA] fifth paragraph). kd_fused_kl_fwdbwd does both in one call
 *     without the recompute.
 *
 * What is computed (the oracle's definition). Per position t:
 *   lse_t  = log sum_j exp z_tj over the full vocabulary, z_t = W h_t
 *   p_tk   = exp(l_tk - log sum_k' exp l_tk')   (teacher renormalised over K)
 *   L_t    = sum_k p_tk log p_tk - sum_k p_tk z_{t,id_tk} + lse_t
 *   loss   = (1/T) sum_t L_t
 *   dz_tj  = s * (exp(z_tj - lse_t) - sum_k p_tk [id_tk == j])
 *   dH     = dz W,   dW (+)= dz^T H
 * with s = grad_scale (times *grad_scale_dev when given). For the mean loss,
 * s = dLoss_total/dloss * (1/T).
 *
 * Conventions for every entry point:
 *  - Pointers are device pointers into memory that the caller owns. The
 *    library never allocates or frees device memory. The workspace `ws` is
 *    caller-allocated scratch of at least the size its *_workspace_size query
 *    returns, aligned to 256 bytes.
 *  - All matrices are row-major and contiguous unless an `ld` (row stride in
 *    elements) is given. bf16 is IEEE bfloat16 (1-8-7) stored as uint16.
 *  - `stream` is a cudaStream_t cast to void*. NULL means the legacy default
 *    stream. Calls enqueue their work and return without synchronising.
 *    Calls that share one workspace must not overlap on the GPU. Calls on
 *    distinct workspaces may run concurrently: on different streams, and
 *    from different host threads (except kd_topk_cache_noalloc, whose
 *    scratch is shared).
 *  - Argument errors come back synchronously, before anything is launched,
 *    as KD_ERR_INVALID_ARG / KD_ERR_UNSUPPORTED / KD_ERR_WORKSPACE. A failed
 *    launch returns KD_ERR_CUDA. Errors found on the device are recorded in a
 *    status word inside `ws`: a cache id outside [0, V), or a pipeline wait
 *    that gave up after its time limit. The first error wins, and the word
 *    keeps it until kd_read_device_status reads and clears it.
 */
#ifndef KD_H_
#define KD_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KD_API __attribute__((visibility("default")))
#else
#define KD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kd_status {
  KD_OK = 0,
  KD_ERR_INVALID_ARG = 1,   /* null pointer, non-positive size, K > V, bad dtype */
  KD_ERR_UNSUPPORTED = 2,   /* a size the kernels do not handle (see each call) */
  KD_ERR_WORKSPACE = 3,     /* ws is NULL, misaligned or smaller than required */
  KD_ERR_CUDA = 4,          /* a CUDA launch or runtime call failed */
  KD_ERR_DEVICE_TIMEOUT = 5,/* a device-side wait exceeded its time limit */
  KD_ERR_BAD_ID = 6,        /* a cached id outside [0, V) (that entry was ignored) */
  KD_ERR_IO = 7,            /* a cache file could not be opened, read or written */
  KD_ERR_FORMAT = 8         /* not a cache file, an unfinished one, or a truncated one */
} kd_status;

typedef enum kd_dtype { KD_BF16 = 0, KD_F32 = 1 } kd_dtype;

/* Human-readable name of a status code. Never NULL. */
KD_API const char* kd_status_string(int status);

/* Library ABI version (major * 100 + minor). */
KD_API int kd_version(void);

/* ---------------------------------------------------------------- top-K cache
 *
 * kd_topk_cache: teacher logits -> offline top-K cache.
 *   logits  [T, ld] of `dtype` (KD_BF16 or KD_F32), device. Row t holds V
 *           logits in its first V entries. ld >= V.
 *   ids     [T, K] int32, device, written: per row the K ids with the largest
 *           logits, ordered by value descending and then id ascending. Ties at
 *           the K-th place therefore go to the lowest ids, and -0.0 ties +0.0.
 *   logp    [T, K] float32, device, written: x[t, id] - log sum_j exp x[t, j]
 *           (the full-vocabulary log-softmax at those ids), computed in fp32.
 *   Requires 1 <= K <= V, V < 2^31, and finite logits. The logits pointer
 *   needs only element alignment, and any ld is accepted (each row is read
 *   with 16-byte loads from its first 16-byte boundary). For K <= 1024 a row
 *   is streamed once for its log-sum-exp and a lower bound of its K-th value,
 *   and the elements at or above that bound (collected into a buffer of 2048)
 *   are sorted. A row whose buffer overflows (heavy ties at the K-th value)
 *   or K > 1024 is redone by an exact radix selection. Both paths give the
 *   same result.
 *   Workspace: kd_topk_workspace_size(T, V, K, dtype) bytes: the status word,
 *   then (second int32) a running count of rows that took the radix path.
 */
KD_API size_t kd_topk_workspace_size(int64_t T, int64_t V, int32_t K, int32_t dtype);
KD_API int kd_topk_cache(const void* logits, int32_t dtype, int64_t T, int64_t V, int64_t ld,
                  int32_t K, int32_t* ids, float* logp, void* ws, size_t ws_bytes,
                  void* stream);

/* kd_teacher_topk_cache: the same cache straight from the teacher's final
 * hidden states and LM head, without the [T, V] logits ever existing:
 *   H  [T, d] bf16, device: teacher final hidden states.
 *   W  [V, d] bf16, device: teacher LM-head weights (fold any logit scale or
 *      temperature into W).
 * The logits x = H W^T are computed in fp32 (bf16 products, fp32
 * accumulation on the tensor cores), one chunk of positions at a time, into
 * the workspace. The GEMM epilogue also produces, per position and
 * 256-column vocabulary tile, the maximum and the sum of exp for the
 * log-sum-exp. The selection then reads only the tiles whose maximum
 * reaches the K-th largest tile maximum: every top-K element lies in such a
 * tile. Output contract: that of kd_topk_cache applied to the fp32 logits
 * x (ids by value descending, then id ascending; logp = x - lse in fp32).
 * Requires d % 8 == 0, 16-byte aligned H and W, 1 <= K <= min(V, 65536).
 * Workspace: kd_teacher_topk_workspace_size(d, V, K, chunk) bytes
 * (4 * chunk * round_up(V, 64) for the logits of one chunk, plus 8 bytes per
 * position and vocabulary tile; independent of T; 0 for sizes the call
 * refuses). Its first two int32
 * words are the status word and the running count of rows that took the
 * exact radix path (see kd_topk_cache). This is the teacher-side fusion
 * that the offline step needs ([KD-TH] section "การทำ Distillation แบบ
 * Offline"). */
KD_API size_t kd_teacher_topk_workspace_size(int64_t d, int64_t V, int32_t K, int64_t chunk);
KD_API int kd_teacher_topk_cache(const void* H, const void* W, int64_t T, int64_t d, int64_t V, int32_t K,
                                 int64_t chunk, int32_t* ids, float* logp, void* ws, size_t ws_bytes,
                                 void* stream);

/* kd_topk_cache_noalloc: the same extraction, for callers that cannot
 * allocate device memory and so cannot pass a workspace. Examples: a step
 * running inside a host application that owns every device allocation
 * through its own pool, or a loop that cannot accept cudaMalloc's implicit
 * synchronisation. The paper has no counterpart; this is a library
 * convenience. Arguments are those of kd_topk_cache without ws/ws_bytes.
 * Scratch comes from a fixed 4096-byte array in device memory owned by
 * libkd. Every GPU that loads the library holds it until the process exits.
 * The call allocates nothing.
 *  - Arguments are checked, as kd_topk_cache checks them, before anything is
 *    enqueued; a refused call leaves the stream untouched.
 *  - The first call on a device looks up that array's device address
 *    (cudaGetSymbolAddress, a host call) and keeps it. The lookup is
 *    repeated when the device's context has changed since (after
 *    cudaDeviceReset, for example).
 *  - Each call clears the array on `stream`. Calls that overlap on the GPU
 *    (unordered streams) share the array and race on it.
 *  - If the workspace that kd_topk_cache would need exceeds the array, the call
 *    returns KD_ERR_WORKSPACE (it never does for the current kernel, which
 *    needs 256 bytes).
 *  - A device-side status cannot be read back afterwards; use kd_topk_cache
 *    with your own workspace when you need it. */
KD_API int kd_topk_cache_noalloc(const void* logits, int32_t dtype, int64_t T, int64_t V,
                                 int64_t ld, int32_t K, int32_t* ids, float* logp, void* stream);

/* ------------------------------------------------------------ fused KL loss
 *
 * Shared arguments:
 *   H     [T, d] bf16, device: student final hidden states.
 *   W     [V, d] bf16, device: student LM-head (final projection) weights.
 *   ids   [T, K] int32 and logp [T, K] float32, device: the teacher cache
 *         (any order within a row; logp need not be normalised). Ids should
 *         be distinct within a row. Duplicates are summed, as the scatter-add
 *         gradient does. An id outside [0, V) is ignored and sets
 *         KD_ERR_BAD_ID in the status word.
 *   chunk positions per chunk, 1 <= chunk. The chunk size changes results
 *         only by fp32 rounding order. Each GEMM launch covers a group of
 *         G chunks (G * chunk positions): G = kd_kl_options.group when that
 *         is set, else clamp(4096 / chunk, 1, 4) (integer division). Grouping
 *         makes the dW tiles' contraction longer, so their fp32
 *         read-modify-write of dW is paid once per group. The workspace holds
 *         one group's bf16 dz: about 2 * G * chunk * V bytes. A caller who
 *         sizes `chunk` to bound memory passes group = 1 (through the _ex
 *         calls) and gets about 2 * chunk * V.
 *   Requires d % 8 == 0 (16-byte rows for TMA), 16-byte aligned H and W,
 *   1 <= K <= 4096, 1 <= V < 2^31.
 *   Workspace: kd_fused_kl_workspace_size(d, V, K, chunk) bytes for the
 *   default group, kd_fused_kl_workspace_size_ex(d, V, K, chunk, group) for
 *   an explicit one (group = 0 is the default). It does not depend on T; one
 *   workspace serves all three calls made with the same group. Both return 0
 *   for a non-positive size, a negative group, or any size the calls refuse
 *   (K > 4096 or K > V, V >= 2^31, d, chunk or group * chunk above 2^24).
 */
KD_API size_t kd_fused_kl_workspace_size(int64_t d, int64_t V, int32_t K, int64_t chunk);
KD_API size_t kd_fused_kl_workspace_size_ex(int64_t d, int64_t V, int32_t K, int64_t chunk, int32_t group);

/* Forward. Writes:
 *   loss       device float32 scalar: (1/T) sum_t L_t.
 *   lse        [T] float32 device: log-sum-exp of the student logits per
 *              position. Saved for the backward pass (4 bytes per position).
 *   loss_rows  [T] float32 device, optional (NULL to skip): L_t per position.
 */
KD_API int kd_fused_kl_fwd(const void* H, const void* W, const int32_t* ids, const float* logp,
                    int64_t T, int64_t d, int64_t V, int32_t K, int64_t chunk,
                    float* loss, float* lse, float* loss_rows,
                    void* ws, size_t ws_bytes, void* stream);

/* Backward. Recomputes each chunk's logits, forms dz (bf16, in ws), then
 *   dH [T, d] float32 device, overwritten: dz W.
 *   dW [V, d] float32 device: dz^T H. It is added to the existing contents
 *      when accumulate_dW != 0, and overwritten otherwise.
 *   Either of dH and dW may be NULL (not both): that gradient is then not
 *   computed, and its GEMM (a quarter of the step's tensor work) is not
 *   run. For a frozen LM head pass dW = NULL; for a frozen body, dH = NULL.
 *   lse        [T] float32 from kd_fused_kl_fwd on the same inputs.
 *   grad_scale host float s, and grad_scale_dev an optional device float32
 *              (NULL = 1) that multiplies s. The autograd binding passes
 *              1/T here and the upstream gradient through grad_scale_dev, so
 *              it never synchronises.
 */
KD_API int kd_fused_kl_bwd(const void* H, const void* W, const int32_t* ids, const float* logp,
                    const float* lse, int64_t T, int64_t d, int64_t V, int32_t K,
                    int64_t chunk, float grad_scale, const float* grad_scale_dev,
                    float* dH, float* dW, int32_t accumulate_dW,
                    void* ws, size_t ws_bytes, void* stream);

/* Forward and backward in one call, for a loss that ends the graph (its
 * gradient scale is known before the forward runs). The pages point out
 * that recomputing each chunk in the backward pass doubles the projection
 * work ([KD-TA] fifth paragraph). This call computes each chunk's logits
 * once. It keeps them, until the chunk's lse is known, as
 * e = exp(z - m_tile) in bf16 inside the O(chunk * V) workspace
 * (m_tile = the row's maximum over one 256-column vocabulary tile). The
 * projection costs 6 T d V flops instead of 8, with the same workspace as
 * kd_fused_kl_fwd/bwd and nothing that grows with T. The teacher side and
 * the loss are those of [KD-TH] section "กลไก Fused Chunked KL Loss".
 * Outputs and arguments are those of kd_fused_kl_fwd followed by
 * kd_fused_kl_bwd (loss, lse and the optional loss_rows; dH overwritten,
 * dW overwritten or accumulated; either of dH and dW may be NULL, not
 * both, to skip it). The difference is that s = grad_scale
 * (times *grad_scale_dev) must be known at call time. Results match the
 * two calls within rounding. dz off the teacher ids is rounded to bf16
 * twice (e, then dz), so it carries up to about 2^-8 relative error instead
 * of 2^-9. At the teacher ids, dz is formed from the fp32 logit as in
 * kd_fused_kl_bwd.
 * Workspace: kd_fused_kl_workspace_size(d, V, K, chunk), the same as for the
 * two separate calls. */
KD_API int kd_fused_kl_fwdbwd(const void* H, const void* W, const int32_t* ids, const float* logp,
                       int64_t T, int64_t d, int64_t V, int32_t K, int64_t chunk,
                       float grad_scale, const float* grad_scale_dev,
                       float* loss, float* lse, float* loss_rows, float* dH, float* dW,
                       int32_t accumulate_dW, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------- loss variants (_ex)
 *
 * kd_fused_kl_fwd_ex / kd_fused_kl_bwd_ex / kd_fused_kl_fwdbwd_ex take the
 * arguments of the plain calls plus `opt`, just before `ws`. opt == NULL
 * gives exactly the plain calls. The pages leave these variants open; they
 * follow the usual distillation conventions.
 *   temperature     tau > 0 (1 = none). The student distribution is
 *                   softmax(z / tau) and the teacher's is its cached
 *                   log-probs divided by tau, renormalised over K. lse is
 *                   that of z / tau, and dL/dz gains a factor 1/tau. No
 *                   tau^2 factor is applied; to use Hinton's scaling,
 *                   multiply the loss and grad_scale by tau^2.
 *   mask            [T] uint8, device, or NULL. A position with mask[t] == 0
 *                   adds nothing to the loss (its loss_rows entry is 0),
 *                   gets a zero dH row and contributes nothing to dW.
 *   mean_over_mask  0: loss = sum_t L_t / T, and grad_scale carries the
 *                   reduction as in the plain calls (1/T for the mean).
 *                   1: loss = sum_t L_t / N with N = the included positions
 *                   (loss 0 if N = 0); the backward then applies 1/N itself,
 *                   so grad_scale is d objective / d loss (1 for the loss
 *                   alone). N is counted on the device; nothing synchronises.
 *   dH_bf16         1: dH is written as bf16 [T, d] (dH points to bf16).
 *   group           chunks per GEMM launch (see `chunk` above); 0 = the
 *                   default rule. The workspace must then be at least
 *                   kd_fused_kl_workspace_size_ex(d, V, K, chunk, group).
 *                   group * chunk must not exceed 2^24 (KD_ERR_UNSUPPORTED).
 * An invalid option (tau <= 0 or not finite, flags outside {0, 1}, a
 * negative group) returns KD_ERR_INVALID_ARG.
 */
typedef struct kd_kl_options {
  float temperature;
  const uint8_t* mask;
  int32_t mean_over_mask;
  int32_t dH_bf16;
  int32_t group;
} kd_kl_options;

KD_API int kd_fused_kl_fwd_ex(const void* H, const void* W, const int32_t* ids, const float* logp,
                              int64_t T, int64_t d, int64_t V, int32_t K, int64_t chunk,
                              float* loss, float* lse, float* loss_rows, const kd_kl_options* opt,
                              void* ws, size_t ws_bytes, void* stream);
KD_API int kd_fused_kl_bwd_ex(const void* H, const void* W, const int32_t* ids, const float* logp,
                              const float* lse, int64_t T, int64_t d, int64_t V, int32_t K,
                              int64_t chunk, float grad_scale, const float* grad_scale_dev,
                              void* dH, float* dW, int32_t accumulate_dW, const kd_kl_options* opt,
                              void* ws, size_t ws_bytes, void* stream);
KD_API int kd_fused_kl_fwdbwd_ex(const void* H, const void* W, const int32_t* ids, const float* logp,
                                 int64_t T, int64_t d, int64_t V, int32_t K, int64_t chunk,
                                 float grad_scale, const float* grad_scale_dev,
                                 float* loss, float* lse, float* loss_rows, void* dH, float* dW,
                                 int32_t accumulate_dW, const kd_kl_options* opt,
                                 void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------- cache files on disk
 *
 * The offline cache is computed once and reused by every training run
 * ([KD-TH] section "การทำ Distillation แบบ Offline"). These calls store it in
 * a file and read any range of positions back. All pointers are HOST memory;
 * none of these calls touches the GPU. Format (little-endian): a 64-byte
 * header (magic "KDTOPK01", uint32 version 1, uint32 header size 64, int64 T,
 * int64 V, int32 K, uint32 flags 0, 24 zero bytes), then T fixed-size
 * records of 8*K bytes: the position's K int32 ids, then its K float32 logp.
 * A record is what kd_topk_cache writes for one row.
 *
 * Writing: kd_cache_create truncates or creates `path` and returns a writer.
 * kd_cache_append adds `rows` records from ids/logp ([rows, K] each,
 * row-major). It returns KD_ERR_BAD_ID and writes nothing if an id lies
 * outside [0, V). kd_cache_close syncs the data and only then records T in
 * the header. A file whose writer never closed it keeps T = -1, and
 * kd_cache_open rejects it with KD_ERR_FORMAT.
 * Reading: kd_cache_open validates the header and the file size
 * (KD_ERR_FORMAT if they disagree) and reports T, V and K (each optional).
 * kd_cache_read copies records [row0, row0 + rows) into ids/logp. It may run
 * concurrently from several threads on one reader. rows = 0 is a no-op for
 * append and read (ids/logp may then be NULL). kd_cache_close releases
 * a handle of either kind.
 */
typedef struct kd_cache_file kd_cache_file;
KD_API int kd_cache_create(const char* path, int64_t V, int32_t K, kd_cache_file** out);
KD_API int kd_cache_append(kd_cache_file* f, const int32_t* ids, const float* logp, int64_t rows);
KD_API int kd_cache_open(const char* path, kd_cache_file** out, int64_t* T, int64_t* V, int32_t* K);
KD_API int kd_cache_read(kd_cache_file* f, int64_t row0, int64_t rows, int32_t* ids, float* logp);
KD_API int kd_cache_close(kd_cache_file* f);

/* Synchronises `stream`, returns the status word kept in `ws` (KD_OK when no
 * device-side error was recorded) and clears it. Returns KD_ERR_CUDA if the
 * stream itself failed. */
KD_API int kd_read_device_status(void* ws, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KD_H_ */
