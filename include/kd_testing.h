/*
 * kd_testing.h - test hooks of libkd. These are not part of the method's
 * interface; the tests use them to check building blocks in isolation.
 */
#ifndef KD_TESTING_H_
#define KD_TESTING_H_

#include <stdint.h>

#include "kd.h"

#ifdef __cplusplus
extern "C" {
#endif

/* C = A * B^T (fp32, row-major, device) on the tcgen05 GEMM that the
 * backward pass uses for dH and dW (dynamic tile scheduling, TMA loads, TMEM
 * accumulators, TMA store / reduce-add). The tile shape follows `flags`:
 * one CTA per 128 x 256 tile by default.
 *   A: a_mn == 0 -> [M, K] row-major; a_mn == 1 -> [K, M] row-major (bf16).
 *   B: b_mn == 0 -> [N, K] row-major; b_mn == 1 -> [K, N] row-major (bf16).
 *   flags bit 0: add into C instead of overwriting it.
 *   flags bit 1: store C transposed, i.e. C is [N, M] row-major.
 *   flags bit 2: CTA-pair tiles (256 x 256 per cluster of two CTAs, tcgen05
 *                cta_group::2); needs b_mn == 0 (else KD_ERR_UNSUPPORTED).
 *   flags bit 3: with bit 2, wide pair tiles (256 x 512, one 512-column
 *                accumulator, eight epilogue warps).
 *   flags bit 4: with bits 2 and 3, 256 x 480 tiles (two N = 240 MMAs; the
 *                backward's dW uses them when d is a multiple of 480 but not
 *                of 512); C not transposed (else KD_ERR_UNSUPPORTED).
 * Requires K, and M or N for MN-major operands, to be multiples of 8, and
 * C's row length a multiple of 4. `ws` (>= 256 bytes, device) holds the
 * status word and the tile counter. Returns a kd_status value. */
KD_API int kd_test_gemm(const void* A, const void* B, float* C, int64_t M, int64_t N, int64_t K, int32_t a_mn,
                        int32_t b_mn, int32_t flags, void* ws, void* stream);

/* Launches a one-warp kernel that waits on an mbarrier nothing arrives at,
 * with the bounded wait all libkd pipelines use, here limited to limit_ns
 * (0 < limit_ns <= 1e10). When the limit passes, the kernel writes
 * KD_ERR_DEVICE_TIMEOUT into the status word at ws and returns normally, so
 * the context stays usable. Read the word with kd_read_device_status. */
KD_API int kd_test_wait_timeout(int64_t limit_ns, void* ws, void* stream);

/* Process-wide switches of the kernels a call runs, for tests and
 * measurements. Production callers leave them at their defaults; nothing in
 * the environment changes them.
 * kd_test_set_gemm_tiles: cta2 = -1 (default: CTA-pair tiles), 0 (one CTA
 *   per 128 x 256 tile) or 1 (CTA pairs); wide = -1 (default: each GEMM's
 *   own width), 0 (every pair GEMM 256 x 256) or 1 (every pair GEMM
 *   256 x 512). Calls already enqueued keep the shape they were set up with;
 *   calls made afterwards, from any thread, use the new one. Values outside
 *   {-1, 0, 1} return KD_ERR_INVALID_ARG and change nothing.
 * kd_test_get_gemm_tiles: the current switch values (-1 = default).
 * kd_test_set_topk_force_exact: on = 1 sends every row of kd_topk_cache and
 *   kd_teacher_topk_cache through the exact radix selection (the path that
 *   otherwise handles overflowing rows); 0 restores the default. */
KD_API int kd_test_set_gemm_tiles(int32_t cta2, int32_t wide);
KD_API int kd_test_get_gemm_tiles(int32_t* cta2, int32_t* wide);
KD_API int kd_test_set_topk_force_exact(int32_t on);

#ifdef __cplusplus
}
#endif

#endif /* KD_TESTING_H_ */
