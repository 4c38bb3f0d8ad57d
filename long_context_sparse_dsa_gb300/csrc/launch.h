// launch.h -- host-side launchers of the DSA kernels (internal to the library).
// Each returns cudaSuccess or the launch error; argument validation happens in
// the C ABI layer (api.cu) before any of these is called.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace dsa {

// Pool keys: kpool[p] = sum of k_I rows 4p..4p+3 (fp32 adds in order, one rounding).
cudaError_t launch_pool_keys(bool bf16, int64_t L, int di, const void* k_idx, void* kpool, cudaStream_t s);

// Indexer scores, fp32 layer: plain FFMA kernel.
cudaError_t launch_indexer_simt_f32(int64_t L, int Hi, int di, const float* q_idx, const float* kpool,
                                    const float* w, int64_t q_begin, int64_t q_count, float* scores,
                                    cudaStream_t s);

// Indexer scores, bf16 layer: tcgen05 tensor-core kernel fed by TMA.
cudaError_t launch_indexer_tc_bf16(int64_t L, int Hi, int di, const void* q_idx, const void* kpool,
                                   const float* w, int64_t q_begin, int64_t q_count, float* scores,
                                   cudaStream_t s);

// Top-k pool selection for rows q_begin..q_begin+q_count-1.
cudaError_t launch_topk(int64_t L, int k, const float* scores, int64_t q_begin, int64_t q_count, int32_t* idx,
                        cudaStream_t s);

// Sparse attention forward; o_acc (optional, fp32) gets O with P carried beyond bf16.
cudaError_t launch_attn_fwd_bf16(int64_t L, int Hq, int d, int k, float scale, const void* q, const void* kk,
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

int device_sm_count();

}  // namespace dsa
