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

/* Replay the memory traffic of the sparse attention kernels for a given
 * selection, with no arithmetic.
 *   dims   the layer (bf16; d, Hq, k and L as for dsa_sparse_attn_fwd)
 *   k, v   [L, d] bf16 (read)
 *   idx    [L, k] int32, the selection the attention kernels would use
 *   dk, dv [L, d] fp32, or both NULL.  When given, they are ADDED to (the
 *          probe adds tiny values; their contents are meaningless afterwards)
 * For every (query, 16-head group) one warp walks the same 16-key steps as
 * the attention kernels (the pools of idx[t] in order, then the query's own
 * partial pool), gathering each step's K and V rows with the same 16-byte
 * cp.async copies, with the forward's warps per CTA, gather stages and CTAs
 * per SM.  With dk/dv it also adds each pool slot's visible rows into dk and
 * dv with one bulk (TMA-engine) fp32 reduction per slot and tensor, as the
 * backward does, with the backward's occupancy.  The bytes moved are the
 * kernels' logical bytes: 2*d*2 per attended key gathered, plus 2*d*4 per
 * attended key reduced.  idx entries outside 0..elig(t)-1 are skipped.
 * Returns DSA_OK, DSA_ERR_INVALID_ARG (NULL or misaligned pointer, only one
 * of dk/dv), DSA_ERR_UNSUPPORTED (a shape the bf16 attention kernels do not
 * take) or DSA_ERR_CUDA. */
dsa_status dsa_probe_traffic(const dsa_dims *dims, const void *k, const void *v, const int32_t *idx, float *dk,
                             float *dv, dsa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_GB300_PROBE_H */
