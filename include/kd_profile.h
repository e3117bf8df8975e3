/*
 * kd_profile.h - per-kernel timing hook of libkd.
 *
 * Between kd_profile_begin() and kd_profile_end(), every kernel that libkd
 * launches is bracketed by two CUDA events recorded on the launch stream.
 * kd_profile_end() waits for the recorded events and returns, per kernel
 * name, the number of launches and their summed device time. The events are
 * created on the host; no device memory is allocated. When profiling is off
 * (the default), launches record nothing.
 *
 * Independently of these calls, every compute call of the C ABI runs inside
 * an NVTX range named after it ("kd_fused_kl_fwd", "kd_topk_cache", ...), and
 * each of its kernel launches inside a nested range named as in the entries
 * below (e.g. "grad_dH_dW"). A tool such as ncu can select launches by these
 * ranges (--nvtx --nvtx-include "kd_fused_kl_bwd/grad_dH_dW/"). With no tool
 * attached the ranges cost a pointer check each.
 */
#ifndef KD_PROFILE_H_
#define KD_PROFILE_H_

#include <stdint.h>

#include "kd.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct kd_prof_entry {
  char name[32];     /* kernel name, e.g. "grad_dH_dW" */
  int32_t launches;  /* launches recorded */
  double total_ms;   /* summed event-to-event time of those launches */
} kd_prof_entry;

/* Start recording (clears earlier records). Returns KD_OK. */
KD_API int kd_profile_begin(void);

/* Stop recording, synchronise the recorded events and write up to
 * max_entries aggregated entries to `out`, with the number written in
 * *n_out. Returns KD_OK, or KD_ERR_CUDA if an event failed. */
KD_API int kd_profile_end(kd_prof_entry* out, int32_t max_entries, int32_t* n_out);

#ifdef __cplusplus
}
#endif

#endif /* KD_PROFILE_H_ */
