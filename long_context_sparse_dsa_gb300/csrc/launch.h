// launch.h -- host-side launchers of the DSA kernels (internal to the library).
// Each returns cudaSuccess or the launch error; argument validation happens in
// the C ABI layer (api.cu) before any of these is called.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace dsa {

// Pool keys: kpool[p] = sum of k_I rows 4p..4p+3 (fp32 adds in order, one rounding).
// gate: [L] fp32 per-token gates, or nullptr for the plain sum
cudaError_t launch_pool_keys(bool bf16, int64_t L, int di, const void* k_idx, const float* gate, void* kpool,
                             cudaStream_t s);

// Indexer scores, fp32 layer: plain FFMA kernel.
cudaError_t launch_indexer_simt_f32(int64_t L, int Hi, int di, const float* q_idx, const float* kpool,
                                    const float* w, int64_t q_begin, int64_t q_count, float* scores,
                                    cudaStream_t s);

// Indexer scores, bf16 layer: tcgen05 tensor-core kernel fed by TMA.
cudaError_t launch_indexer_tc_bf16(int64_t L, int Hi, int di, const void* q_idx, const void* kpool,
                                   const float* w, int64_t q_begin, int64_t q_count, float* scores,
                                   cudaStream_t s);

// What one launch computes.  Score mode writes the fp32 score block of the
// query range (column j = pool j*col_stride: col_stride 1 is the full block,
// a larger stride the sampled block of the fused top-k).  Emit mode (the EMIT
// template flag) writes no scores: every eligible score >= tau[row] goes to
// the row's candidate list.  With a block list only the listed 32-query
// blocks are computed.
// Candidate lists of the fused indexer + top-k.  Row r of a chunk owns
// cand_stride(P) entries: for each 2048-pool segment s < nseg(t) of its
// eligible prefix and each TMEM lane quarter q (the epilogue warp that scores
// pools 2048 s + 128 i + 32 q .. +31 of every tile i), a sub-list of
// cand_stride / (4 nseg(t)) entries, filled by that warp alone.
constexpr int kSegPools = 2048;     // pools per indexer work unit (16 tiles of 128)
__host__ __device__ constexpr int64_t fused_nseg_max(int64_t P) { return (P + kSegPools - 1) / kSegPools; }
__host__ __device__ constexpr int64_t fused_cand_stride(int64_t P) {
  return 64 * fused_nseg_max(P) > 4096 ? 64 * fused_nseg_max(P) : 4096;
}

struct IdxArgs {
  const float* w;
  float* scores;              // score mode: [q_count, P_cols] fp32
  int64_t P_cols;             // score mode: row pitch of `scores` (columns)
  int64_t q_begin, q_count;
  int col_stride;             // column j of the block is pool j * col_stride
  int tma_store;              // score mode: tiles leave through TMA stores
  const float* tau;           // emit mode: per-row threshold [q_count]
  uint2* cand;                // emit mode: [q_count, cand_stride] (score bits, pool) sub-lists
  uint32_t* cntq;             // emit mode: [q_count, nseg_max, 4] sub-list lengths (may exceed capacity)
  int64_t cand_stride;        // emit mode: entries per row of cand
  int64_t nseg_max;           // emit mode: segments per row of cntq
  const int32_t* blist;       // optional: 32-query blocks (relative to q_begin) to compute
  const uint32_t* blist_n;    // its length
};

// The tensor-core indexer in any of the modes above (emit: candidate lists
// instead of scores).
cudaError_t launch_indexer_tc_bf16_ex(int64_t L, int Hi, int di, const void* q_idx, const void* kpool,
                                      const IdxArgs& a, bool emit, cudaStream_t s);

// Indexer scores and top-k selection of one query chunk without the score
// block (bf16; tensor-core indexer).  ws holds fused_indexer_topk_ws_bytes(L,
// q_count) bytes of scratch: the fallback score rows, the sampled scores and
// the candidate lists.
// Two routes: 0 = the candidate lists (no score block), 1 = the score block
// and the row-wise top-k (the unfused pair).
size_t fused_indexer_topk_ws_bytes(int64_t L, int64_t rows);
cudaError_t launch_indexer_topk_bf16(int64_t L, int Hi, int di, int k, const void* q_idx, const void* kpool,
                                     const float* w, int64_t q_begin, int64_t q_count, int32_t* idx, void* ws,
                                     int route, cudaStream_t s);

// Top-k over the score rows listed in rlist[0 .. *rlist_n) (at most max_rows).
cudaError_t launch_topk_list(int64_t L, int k, const float* scores, int64_t q_begin, int64_t max_rows,
                             const int32_t* rlist, const uint32_t* rlist_n, int32_t* idx, cudaStream_t s);

// Top-k pool selection for rows q_begin..q_begin+q_count-1.
cudaError_t launch_topk(int64_t L, int k, const float* scores, int64_t q_begin, int64_t q_count, int32_t* idx,
                        cudaStream_t s);

// Sparse attention forward; o_acc (optional, fp32) gets O with P carried beyond bf16.
cudaError_t launch_attn_fwd_bf16(int64_t L, int Hq, int d, int k, float scale, const void* q, const void* kk,
                                 const void* v, const int32_t* idx, void* o, float* lse, float* o_acc,
                                 cudaStream_t s);
// tcgen05 forward (attn_fwd_tc.cu): d = 128, Hq in {16, 32}
bool attn_fwd_tc_supported(int Hq, int d);
cudaError_t launch_attn_fwd_tc_bf16(int64_t L, int Hq, int d, int k, float scale, const void* q, const void* kk,
                                    const void* v, const int32_t* idx, void* o, float* lse, float* o_acc,
                                    cudaStream_t s);
cudaError_t launch_attn_fwd_f32(int64_t L, int Hq, int d, int k, float scale, const float* q, const float* kk,
                                const float* v, const int32_t* idx, float* o, float* lse, cudaStream_t s);

// Sparse attention backward (bf16): dq overwritten; dk, dv must be zeroed by the
// caller.  With oacc (the forward's fp32 output) D = dO . oacc is formed in the
// gradient kernel; without it dbuf, an [L, Hq] fp32 workspace, carries D from
// a first kernel.
cudaError_t launch_attn_bwd_bf16(int64_t L, int Hq, int d, int k, float scale, const void* q, const void* kk,
                                 const void* v, const int32_t* idx, const float* lse, const void* dout,
                                 const float* oacc, float* dbuf, float* dq, float* dk, float* dv, cudaStream_t s);

// The query-major half of the deterministic backward: dQ, and D into dbuf
// (formed from oacc when given, else by a first D pass).
cudaError_t launch_attn_bwd_dq_bf16(int64_t L, int Hq, int d, int k, float scale, const void* q, const void* kk,
                                    const void* v, const int32_t* idx, const float* lse, const void* dout,
                                    const float* oacc, float* dbuf, float* dq, cudaStream_t s);

// The deterministic (key-major) backward: dq, dk, dv overwritten; ws holds
// det_bwd_ws_bytes(L, Hq, d, k) bytes of scratch.
size_t det_bwd_ws_bytes(int64_t L, int Hq, int d, int k);
cudaError_t launch_attn_bwd_det_bf16(int64_t L, int Hq, int d, int k, float scale, const void* q, const void* kk,
                                     const void* v, const int32_t* idx, const float* lse, const void* dout,
                                     const float* oacc, float* dq, float* dk, float* dv, void* ws, cudaStream_t s);

int device_sm_count();

}  // namespace dsa
