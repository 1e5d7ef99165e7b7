/*
 * ttt_profile.h - launch accounting of the library's kernels.
 *
 * The pages have no counterpart for these calls: they expose, for tests and
 * benchmarks, how many kernels the library launched and (while a profile is
 * recording) the device time of each launch, measured with CUDA events on the
 * launching stream, with the algorithmic work of that launch (FLOPs of the
 * matrix products it computes, bytes a bandwidth kernel must move).
 * Host-only bookkeeping; the library's numerics do not change.
 */
#ifndef TTT_GB300_TTT_PROFILE_H
#define TTT_GB300_TTT_PROFILE_H

#include "ttt.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  char name[32];   /* launch kind, e.g. "gemm.proj", "norm" */
  char kernel[32]; /* CUDA kernel it ran */
  int launches;
  double ms;       /* summed device time of those launches */
  double flops;    /* summed algorithmic FLOPs (matrix products) */
  double bytes;    /* summed algorithmic DRAM bytes (bandwidth kernels) */
  double sm_ms;    /* summed device time x the fraction of the SMs each launch's
                      grid holds (at most 1): the GPU time the launches occupy */
} ttt_profile_entry;

/* Total kernel launches the library has made in this process. */
unsigned long long ttt_launch_count(void);

/* Starts recording launch events (clears the previous record). */
void ttt_profile_start(void);

/* Stops recording, synchronises the recorded events and writes at most
 * max_entries per-kind totals to `entries` (host memory).  Returns the number
 * of kinds written, or TTT_ERR_CUDA. */
int ttt_profile_stop(ttt_profile_entry* entries, int max_entries);

#ifdef __cplusplus
}
#endif

#endif /* TTT_GB300_TTT_PROFILE_H */
