/*
 * dsa_probe.h -- a measurement probe of libdsa_gb300.so, outside the layer.
 *
 * The sparse attention kernels gather whole pools of K/V rows from a table
 * that stays in the L2 cache, and the backward adds fp32 dK/dV rows back
 * into a table of the same kind.  Their bound is the rate at which the SMs
 * can move that traffic through L2, not HBM bandwidth and not the tensor
 * cores.  This probe replays exactly that traffic with no arithmetic, so a
 * kernel's achieved rate can be put against a ceiling measured on the same
 * GPU in the same run.  The pages have no counterpart: it is a measuring
 * instrument, not part of the method.
 *
 * Same conventions as dsa.h: device pointers owned by the caller, work
 * enqueued on `stream`, validation before any launch, no allocation.
 */
#ifndef DSA_GB300_PROBE_H
#define DSA_GB300_PROBE_H

#include <stdint.h>

#include "dsa.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Replay the memory traffic of `steps` 16-key attention steps.
 *   d      head dim, 64 or 128
 *   L      rows of k, v (and of dk, dv); a multiple of 4, >= 4
 *   k, v   [L, d] bf16 (read)
 *   dk, dv [L, d] fp32, or both NULL.  When given, they are ADDED to (the
 *          probe adds tiny values; their contents are meaningless afterwards)
 *   steps  >= 1
 *   seed   selects the pseudo-random pools
 * One step picks 4 pools uniformly at random (a counter-based hash of seed,
 * step and slot) and gathers their 16 K rows and 16 V rows with the same
 * 16-byte cp.async copies the attention kernels use (16 * 2 * d * 2 bytes).
 * With dk/dv it then adds 4 * d fp32 values per pool into each of dk and dv
 * with one bulk (TMA-engine) reduction per pool and tensor, as the backward
 * does (16 * 2 * d * 4 bytes).  Returns DSA_OK, DSA_ERR_INVALID_ARG (NULL or
 * misaligned pointer, only one of dk/dv, bad L or steps), DSA_ERR_UNSUPPORTED
 * (d) or DSA_ERR_CUDA. */
dsa_status dsa_probe_traffic(int32_t d, int64_t L, const void *k, const void *v, float *dk, float *dv,
                             int64_t steps, uint64_t seed, dsa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_GB300_PROBE_H */
