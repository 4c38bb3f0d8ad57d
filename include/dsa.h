/*
 * dsa.h -- C ABI of the GB300 (sm_103a) DeepSeek Sparse Attention layer library
 * (libdsa_gb300.so).
 *
 * One DSA layer: a lightning indexer scores every causal 4-token key pool for
 * every query, a per-query top-k keeps the best pools, and attention runs
 * only over the tokens of those pools (plus the query's own partial pool).
 *
 * Source passages (page "SkyRL extends GLM-5.3-Flash training context to 1
 * million tokens"):
 *   section "Model and bottleneck": the indexer scores one pool per 4 tokens
 *     for every query; attention then reads about 2048 keys per query;
 *   section "1. DSA truly sparse": no positional encoding (NoPE); 2051 keys
 *     rather than 2048; the indexer is scored in query chunks; selected pool
 *     indices are int32; a kernel that silently rejects a shape and falls back
 *     to dense attention is the failure to avoid.
 * The pages print no formula; the definitions below are the plainest reading
 * of those passages:
 *   elig(t)      = floor((t+1)/4)   pools whose 4 tokens are all <= t
 *   kpool[p]     = k_I[4p] + k_I[4p+1] + k_I[4p+2] + k_I[4p+3]
 *                  (fp32 adds in that order, rounded once to the layer dtype)
 *   s[t,p]       = sum_h w[t,h] * max(0, q_I[t,h,:] . kpool[p,:]),  p < elig(t)
 *   idx[t,:]     = the min(k, elig(t)) best pools by (score desc, pool asc),
 *                  listed in ascending pool order, padded with -1
 *   keys(t)      = tokens of idx[t,:], plus 4*floor(t/4) .. t when t%4 != 3
 *   O[t,h]       = softmax_j(scale * Q[t,h] . K[j]) V[j] over j in keys(t)
 *   LSE[t,h]     = log sum_j exp(scale * Q[t,h] . K[j])  (natural log)
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers, row-major and contiguous, owned
 *     by the caller.  The library never allocates, frees or synchronises
 *     device memory or streams, except dsa_check_device_error (which
 *     synchronises the given stream).
 *   - Work is enqueued on `stream` and runs asynchronously; a DSA_OK return
 *     means the launches were accepted, not that they finished.
 *   - Arguments are validated before anything is launched.  A shape the
 *     kernels do not support returns DSA_ERR_UNSUPPORTED: there is no
 *     fallback to another algorithm, dense or otherwise.
 *   - Every pointer must be 16-byte aligned.
 *   - Layer-dtype tensors (Q, K, V, q_I, k_I, kpool, O, dO) are fp32 or bf16
 *     per dims->dtype; w, scores, LSE, dQ, dK, dV are fp32; idx is int32.
 *   - Kernels never trap.  A bad index inside idx (a pool the query may not
 *     see) is skipped and recorded in a device error word, read back by
 *     dsa_check_device_error.
 *   - Results of the forward steps (pool keys, scores, top-k, attention
 *     forward) are bitwise reproducible run to run.  The backward adds dK/dV
 *     contributions with fp32 atomics, so its summation order varies.
 */
#ifndef DSA_GB300_H
#define DSA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *dsa_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
    DSA_OK = 0,
    DSA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad range, L % 4 != 0, k < 1, ... */
    DSA_ERR_UNSUPPORTED = 2,  /* a shape or dtype the kernels do not implement */
    DSA_ERR_WORKSPACE = 3,    /* workspace pointer missing or smaller than required */
    DSA_ERR_CUDA = 4,         /* a CUDA runtime/driver call or launch failed */
    DSA_ERR_TIMEOUT = 5,      /* a bounded device-side wait gave up (see dsa_check_device_error) */
    DSA_ERR_BAD_INDEX = 6     /* idx named a pool outside 0..elig(t)-1 (entry skipped) */
} dsa_status;

typedef enum { DSA_FP32 = 0, DSA_BF16 = 1 } dsa_dtype;

/* Layer shape, passed by pointer to every entry point.
 *   L       tokens; a multiple of 4 (pool size), >= 4
 *   Hq      query heads sharing the single K/V head
 *   d       attention head dim
 *   Hi      indexer heads
 *   di      indexer head dim
 *   pool    tokens per pool; must be 4
 *   k       pools kept per query, >= 1
 *   q_chunk queries scored per indexer chunk inside dsa_layer_fwd (bounds the
 *           score workspace to q_chunk * (L/4) fp32 values); >= 1
 *   scale   softmax scale (1/sqrt(d) for the usual layer)
 *   dtype   dsa_dtype of the layer-dtype tensors
 * Supported shapes (anything else -> DSA_ERR_UNSUPPORTED):
 *   bf16: d in {64,128}, Hq in {16,32}, di in {64,128}, Hi in {4,8}, k <= 1024
 *   fp32: d in {64,128}, 1 <= Hq <= 32, di in {64,128}, 1 <= Hi <= 8, k <= 1024
 *         (backward is bf16 only)
 */
typedef struct dsa_dims {
    int64_t L;
    int32_t Hq;
    int32_t d;
    int32_t Hi;
    int32_t di;
    int32_t pool;
    int32_t k;
    int32_t q_chunk;
    float scale;
    int32_t dtype;
} dsa_dims;

/* Short English name of a status code (static storage). */
const char *dsa_status_string(dsa_status status);

/* Detail of the last non-OK status returned on the calling host thread
 * (static thread-local storage; empty string if none). */
const char *dsa_last_error_message(void);

/* Validate `dims` for the given pass (0 = forward, 1 = forward+backward)
 * without touching the GPU.  Returns DSA_OK, DSA_ERR_INVALID_ARG or
 * DSA_ERR_UNSUPPORTED. */
dsa_status dsa_validate_dims(const dsa_dims *dims, int32_t with_backward);

/* Bytes of device workspace dsa_layer_fwd needs: that of dsa_indexer_topk
 * for one query chunk, dsa_indexer_topk_workspace_bytes(dims,
 * min(q_chunk, L)).  Returns 0 if dims are invalid. */
size_t dsa_workspace_bytes(const dsa_dims *dims);

/* Bytes of device workspace dsa_indexer_topk needs for q_count queries.
 * fp32 layers: the fp32 score block, q_count * (L/4) * 4 bytes.  bf16 layers:
 * the score rows of the fallback (q_count * (L/4) * 4 bytes), a sampled score
 * block (1/32 of that), the candidate lists (q_count * S * 8 bytes, with
 * S = max(4096, 64 * ceil(L/8192))), their lengths (q_count * ceil(L/8192) *
 * 16 bytes) and a few per-row words, each part rounded up to 256.  Returns 0
 * if dims are invalid or q_count is outside 1 .. L. */
size_t dsa_indexer_topk_workspace_bytes(const dsa_dims *dims, int64_t q_count);

/* Bytes of device workspace dsa_sparse_attn_bwd / dsa_layer_bwd need when
 * they are called without o_acc: one fp32 value per (query, head),
 * L * Hq * 4 bytes, rounded up to 256 (it holds D[t,h] = dO[t,h] . O[t,h]
 * between the backward's two kernels).  Returns 0 if dims are invalid for a
 * backward. */
size_t dsa_bwd_workspace_bytes(const dsa_dims *dims);

/* Pool keys.  Page "SkyRL extends GLM-5.3-Flash ...", section "Model and
 * bottleneck" (one pool per 4 tokens).
 *   k_idx  [L, di]     layer dtype, the indexer's per-token keys k_I
 *   kpool  [L/4, di]   layer dtype, output: kpool[p] as defined above
 * Bitwise equal to the definition (fp32 sum in token order, one rounding). */
dsa_status dsa_pool_keys(const dsa_dims *dims, const void *k_idx, void *kpool, dsa_stream_t stream);

/* Gated pool keys: each token's key weighted by a per-token gate before the
 * pool's sum.  Same page, section "3. Context parallelism (CP)", names k-pool
 * gate scores that must stay aligned with the keys and defines nothing more;
 * the reading implemented is
 *   kpool[p] = sum_{j<4} gate[4p+j] * k_idx[4p+j]
 * accumulated in fp32 in token order with one fused multiply-add per token
 * (from 0), then rounded once to the layer dtype.  With every gate 1 it is
 * dsa_pool_keys bit for bit.  Any normalisation of the gates (a softmax over
 * the pool, say) is the caller's; the result feeds dsa_indexer_score or
 * dsa_indexer_topk exactly as dsa_pool_keys' does.
 *   k_idx  [L, di]   layer dtype
 *   gate   [L]       fp32, 16-byte aligned
 *   kpool  [L/4, di] layer dtype, output
 * Bitwise equal to that definition.  Returns DSA_ERR_INVALID_ARG for a NULL
 * or misaligned pointer, before any launch. */
dsa_status dsa_pool_keys_gated(const dsa_dims *dims, const void *k_idx, const float *gate, void *kpool,
                               dsa_stream_t stream);

/* Indexer scores for queries q_begin .. q_begin+q_count-1.  Same page,
 * sections "Model and bottleneck" and "1. DSA truly sparse" (chunked by
 * query).  bf16 runs on the tcgen05 tensor cores (fp32 accumulation in
 * tensor memory, ReLU and the weighted head sum fused into the epilogue).
 *   q_idx   [L, Hi, di] layer dtype, indexer queries q_I
 *   kpool   [L/4, di]   layer dtype, from dsa_pool_keys
 *   w       [L, Hi]     fp32 head weights
 *   scores  [q_count, L/4] fp32, output; row r is query q_begin+r.  The
 *           entries p < elig(q_begin+r) hold the scores.  Entries past that
 *           prefix are unspecified: those inside the last 128-pool tile a
 *           32-query block visits may be overwritten, later ones are not
 *           touched.
 * Requires 0 <= q_begin, q_count >= 1, q_begin+q_count <= L. */
dsa_status dsa_indexer_score(const dsa_dims *dims, const void *q_idx, const void *kpool, const float *w,
                             int64_t q_begin, int64_t q_count, float *scores, dsa_stream_t stream);

/* Per-query top-k pool selection.  Same page, "Model and bottleneck" (about
 * 2048 keys = 512 pools per query) and "1. DSA truly sparse" (int32 pool
 * indices).  Radix select over the fp32 score bits; -0 and +0 tie; ties go
 * to the lower pool index; only p < elig(t) is considered (causality).
 *   scores  [q_count, L/4] fp32 as written by dsa_indexer_score for the same
 *           q_begin/q_count
 *   idx     [L, k] int32; rows q_begin .. q_begin+q_count-1 are written:
 *           selected pools in ascending order, then -1 padding. */
dsa_status dsa_topk(const dsa_dims *dims, const float *scores, int64_t q_begin, int64_t q_count,
                    int32_t *idx, dsa_stream_t stream);

/* Indexer scores and top-k selection of queries q_begin .. q_begin+q_count-1
 * in one call: the same idx rows as dsa_indexer_score followed by dsa_topk,
 * bit for bit.  Same page, "Model and bottleneck" (the quadratic scoring of
 * every causal pool) and "1. DSA truly sparse" (scored per query chunk; only
 * int32 pool indices leave the indexer).  Two routes for bf16 layers
 * (dsa_set_indexer_topk_route); by default the score block is written to
 * the workspace and selected from.  The other route does not materialise the
 * fp32 score block: a tensor-core pass over every 32nd pool gives each row a
 * threshold below its k-th score (with high probability), the full
 * tensor-core pass keeps only the scores at or above it as candidates, and
 * the exact selection (ties to the lower pool index) runs on those.  A row
 * whose candidates number fewer than k, or overflow their fixed share of the
 * candidate lists, is recomputed through the score block in the workspace and
 * the row-wise top-k, so the result never depends on the threshold; only the
 * time does.  fp32 layers run the unfused pair with the score block in ws.
 *   idx  [L, k] int32; rows q_begin .. q_begin+q_count-1 are written
 *   ws   >= dsa_indexer_topk_workspace_bytes(dims, q_count) bytes of device
 *        memory (scratch; nothing in it needs to start at zero)
 * Requires 0 <= q_begin, q_count >= 1, q_begin+q_count <= L. */
dsa_status dsa_indexer_topk(const dsa_dims *dims, const void *q_idx, const void *kpool, const float *w,
                            int64_t q_begin, int64_t q_count, int32_t *idx, void *ws, size_t ws_bytes,
                            dsa_stream_t stream);

/* Sparse attention forward over keys(t).  Same page, "1. DSA truly sparse"
 * (sparse kernel, NoPE, 2051 keys).  One K/V head shared by all Hq heads.
 *   q     [L, Hq, d]  layer dtype        k, v [L, d] layer dtype
 *   idx   [L, k]      int32 (from dsa_topk or the caller; entries < 0 skipped)
 *   o     [L, Hq, d]  layer dtype, output
 *   lse   [L, Hq]     fp32, output (natural log)
 *   o_acc [L, Hq, d]  fp32, optional output (NULL: not written), 16-byte
 *                     aligned.  O before the cast to the layer dtype, with the
 *                     softmax probabilities entering P.V as bf16 hi + lo parts
 *                     (about 2^-17 relative instead of bf16's 2^-9).  Handing
 *                     it to the backward replaces the backward's D
 *                     recomputation pass; keeping it costs L*Hq*d*4 bytes. */
dsa_status dsa_sparse_attn_fwd(const dsa_dims *dims, const void *q, const void *k, const void *v,
                               const int32_t *idx, void *o, float *lse, float *o_acc, dsa_stream_t stream);

/* Sparse attention backward (bf16 only).  Given dO, writes
 *   dq [L, Hq, d] fp32 (overwritten), dk, dv [L, d] fp32 (zeroed on the
 *   stream, then accumulated with fp32 atomics).
 * o, lse and o_acc must be the forward's outputs for the same q, k, v, idx.
 * The bf16 rounding of o would enter every gradient through D = dO . O, so o
 * is validated but not read.  With o_acc (non-NULL, 16-byte aligned) D is
 * dO . o_acc, formed inside the gradient kernel, and ws is not used (may be
 * NULL).  Without it a first kernel forms D = sum_j P_j dP_j from the
 * recomputed P and dP into ws.  The selection is piecewise constant: no
 * gradient reaches the indexer inputs.
 *   ws   >= dsa_bwd_workspace_bytes(dims) bytes of device memory (scratch),
 *        required when o_acc is NULL */
dsa_status dsa_sparse_attn_bwd(const dsa_dims *dims, const void *q, const void *k, const void *v,
                               const int32_t *idx, const void *o, const float *lse, const float *o_acc,
                               const void *dout, float *dq, float *dk, float *dv, void *ws, size_t ws_bytes,
                               dsa_stream_t stream);

/* Bytes of device workspace dsa_sparse_attn_bwd_det needs: D (L*Hq*4), the
 * inverted selection (per-(pool, 1024-query block) offsets and the L*k query
 * lists, int32) and one band's partial dK/dV sums.  Returns 0 if dims are
 * invalid for a backward or L*(k+1) >= 2^31. */
size_t dsa_bwd_det_workspace_bytes(const dsa_dims *dims);

/* Deterministic sparse attention backward (bf16): the gradients of
 * dsa_sparse_attn_bwd, with dK and dV summed in a fixed order, so repeated
 * calls on the same inputs give the same bits.  Same page, section "Real
 * data" (the trainer's log-probs are checked against the inference
 * engine's, which wants gradients that do not change run to run).
 * dQ is formed query-major as in dsa_sparse_attn_bwd.  For dK/dV the
 * selection is inverted into per-pool query lists in ascending query order
 * (no atomics decide the order), and per band of 4096 queries each pool's
 * contributions are accumulated key-major in registers and added to dK/dV
 * in a fixed (band, chunk, query) order.  Arguments as dsa_sparse_attn_bwd,
 * except the workspace, which is always required:
 *   ws   >= dsa_bwd_det_workspace_bytes(dims) bytes of device memory
 *        (scratch; nothing in it needs to start at zero)
 * idx entries outside 0..elig(t)-1 are skipped.  Returns
 * DSA_ERR_UNSUPPORTED when L*(k+1) >= 2^31. */
dsa_status dsa_sparse_attn_bwd_det(const dsa_dims *dims, const void *q, const void *k, const void *v,
                                   const int32_t *idx, const void *o, const float *lse, const float *o_acc,
                                   const void *dout, float *dq, float *dk, float *dv, void *ws, size_t ws_bytes,
                                   dsa_stream_t stream);

/* Whole forward: dsa_pool_keys once, then per chunk of q_chunk queries
 * dsa_indexer_topk (the fused indexer + top-k) in the workspace, then
 * dsa_sparse_attn_fwd.
 *   outputs: o [L,Hq,d], lse [L,Hq], idx [L,k], kpool [L/4,di];
 *            o_acc [L,Hq,d] fp32 when non-NULL (as in dsa_sparse_attn_fwd)
 *   ws      >= dsa_workspace_bytes(dims) bytes of device memory */
dsa_status dsa_layer_fwd(const dsa_dims *dims, const void *q, const void *k, const void *v,
                         const void *q_idx, const void *k_idx, const float *w,
                         void *o, float *lse, float *o_acc, int32_t *idx, void *kpool,
                         void *ws, size_t ws_bytes, dsa_stream_t stream);

/* Whole backward: dsa_sparse_attn_bwd with the idx, lse and (optionally)
 * o_acc the forward saved (the indexer is not recomputed and gets no gradient).
 *   ws   >= dsa_bwd_workspace_bytes(dims) bytes of device memory when o_acc
 *        is NULL; unused otherwise */
dsa_status dsa_layer_bwd(const dsa_dims *dims, const void *q, const void *k, const void *v,
                         const int32_t *idx, const void *o, const float *lse, const float *o_acc,
                         const void *dout, float *dq, float *dk, float *dv, void *ws, size_t ws_bytes,
                         dsa_stream_t stream);

/* Synchronise `stream`, then read and clear the device error word that the
 * kernels set instead of trapping.  Returns DSA_OK, DSA_ERR_TIMEOUT (a
 * bounded wait gave up; the kernel freed its resources and returned),
 * DSA_ERR_BAD_INDEX, or DSA_ERR_CUDA if the synchronisation itself failed. */
dsa_status dsa_check_device_error(dsa_stream_t stream);

/* Test and measurement hook: the route dsa_indexer_topk (and so
 * dsa_layer_fwd) takes for bf16 layers.  Both give the same idx bit for bit.
 *   1 (default): the indexer writes the chunk's fp32 score block into the
 *      workspace and the row-wise top-k selects from it (dsa_indexer_score
 *      then dsa_topk).
 *   0: no score block; the candidate lists described at dsa_indexer_topk.
 * Applies to calls made afterwards from any host thread.  Returns
 * DSA_ERR_INVALID_ARG for any other value. */
dsa_status dsa_set_indexer_topk_route(int32_t route);

/* Test and measurement hook: the kernel dsa_sparse_attn_fwd (and so
 * dsa_layer_fwd) runs for bf16 layers.
 *   0 (default): the warp-level kernel (one warp per query and 16-head
 *      group, m16n8k16 MMAs, 16-key cp.async gathers).
 *   1: for d = 128, the tcgen05 kernel: keys on the MMA's M side (128-key
 *      tiles gathered by producer warps), all Hq heads on N, S^T and O^T in
 *      tensor memory; other shapes take route 0.  About 3x slower at
 *      L = 131072: with N = Hq = 16 each MMA does little work.
 * Both meet the same tolerances; they differ in summation order.  Applies to
 * calls made afterwards from any host thread.  Returns DSA_ERR_INVALID_ARG
 * for any other value. */
dsa_status dsa_set_attn_fwd_route(int32_t route);

/* Test hook: the number of spin iterations after which a bounded device-side
 * wait gives up (default 1<<20).  Independently of this, every device wait
 * gives up after 2 s of wall time.  Lowering it lets a test make a wait run
 * out.  Takes effect for launches enqueued after the call. */
void dsa_set_wait_limit(uint32_t spins);

/* Size of the fixed device scratch array behind dsa_layer_fwd_noalloc. */
#define DSA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

/* dsa_layer_fwd without a workspace, for callers that cannot allocate device
 * memory for the library: for example a plugin inside a host framework whose
 * own caching allocator owns the device memory and whose operator interface
 * has no workspace argument, or a code path where a cudaMalloc (which may
 * synchronise the device) is not allowed.  The paper has no counterpart; it
 * is an interface convenience.
 *   Same arguments and outputs as dsa_layer_fwd, minus ws/ws_bytes and
 *   o_acc (this entry point does not write one).  The
 *   indexer's score block lives in one fixed device array of
 *   DSA_NOALLOC_SCRATCH_BYTES (64 MiB), which every GPU that loads the
 *   library holds until the process exits; the query chunk is shrunk to
 *   min(q_chunk, 64 MiB / (4 * L/4)) queries, which does not change any
 *   result.  A layer whose single score row (L/4 fp32 values) exceeds the
 *   array returns DSA_ERR_UNSUPPORTED.
 *   Calls no cudaMalloc, cudaFree or other allocating routine.  Its first
 *   call on a device looks up the array's device address (once per device,
 *   with that device current), so make that first call before any stream
 *   capture.  Every call on a device shares the one array: calls whose work
 *   overlaps on the GPU (different streams without ordering) race on it.
 *   Nothing in the array needs to start at zero. */
dsa_status dsa_layer_fwd_noalloc(const dsa_dims *dims, const void *q, const void *k, const void *v,
                                 const void *q_idx, const void *k_idx, const float *w,
                                 void *o, float *lse, int32_t *idx, void *kpool, dsa_stream_t stream);

/* Test hook for the failure-detection path: enqueue a one-CTA kernel that
 * waits on an mbarrier nothing arrives on.  The bounded wait gives up after
 * `spins` polls (1 .. 2^24) and records a timeout; the kernel then returns
 * normally and the stream stays usable.  dsa_check_device_error(stream)
 * afterwards returns DSA_ERR_TIMEOUT. */
dsa_status dsa_selftest_bounded_wait(uint32_t spins, dsa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_GB300_H */
