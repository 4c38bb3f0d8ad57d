// indexer_simt.cu -- indexer scores for fp32 layers (plain FFMA).
//
// Page "SkyRL extends GLM-5.3-Flash training context to 1 million tokens",
// section "Model and bottleneck" (every query scores every 4-token pool) and
// section "1. DSA truly sparse" (scored in query chunks):
//   s[t,p] = sum_h w[t,h] * max(0, q_I[t,h,:] . kpool[p,:])  for p < elig(t).
// fp32 layers are the small configuration; bf16 layers use the tcgen05
// kernel in indexer_tc.cu.  One thread owns one pool column and loops over a
// block of QB queries whose q_I rows sit in shared memory.
#include "common.cuh"
#include "launch.h"

namespace dsa {

constexpr int kSimtQB = 8;
constexpr int kSimtPB = 128;

__global__ void __launch_bounds__(kSimtPB) indexer_simt_f32_kernel(const float* __restrict__ q_idx,
                                                                   const float* __restrict__ kpool,
                                                                   const float* __restrict__ w, int64_t P, int Hi,
                                                                   int di, int64_t q_begin, int64_t q_count,
                                                                   float* __restrict__ scores) {
  extern __shared__ float qs[];  // [kSimtQB][Hi][di]
  const int64_t r0 = (int64_t)blockIdx.y * kSimtQB;
  const int64_t q_end = q_begin + q_count;
  const int row_len = Hi * di;
  for (int i = threadIdx.x; i < kSimtQB * row_len; i += blockDim.x) {
    const int64_t t = q_begin + r0 + i / row_len;
    qs[i] = (t < q_end) ? q_idx[t * row_len + (i % row_len)] : 0.f;
  }
  __syncthreads();
  const int64_t p = (int64_t)blockIdx.x * kSimtPB + threadIdx.x;
  if (p >= P) return;
  const float* kp = kpool + p * di;
  for (int j = 0; j < kSimtQB; ++j) {
    const int64_t t = q_begin + r0 + j;
    if (t >= q_end || p >= elig(t)) continue;
    float s = 0.f;
    for (int h = 0; h < Hi; ++h) {
      const float* q = qs + (j * Hi + h) * di;
      float dot = 0.f;
      for (int i = 0; i < di; i += 4) {
        const float4 k4 = __ldg(reinterpret_cast<const float4*>(kp + i));
        dot = fmaf(q[i], k4.x, dot);
        dot = fmaf(q[i + 1], k4.y, dot);
        dot = fmaf(q[i + 2], k4.z, dot);
        dot = fmaf(q[i + 3], k4.w, dot);
      }
      s = fmaf(fmaxf(dot, 0.f), __ldg(w + t * Hi + h), s);
    }
    scores[(t - q_begin) * P + p] = s;
  }
}

cudaError_t launch_indexer_simt_f32(int64_t L, int Hi, int di, const float* q_idx, const float* kpool,
                                    const float* w, int64_t q_begin, int64_t q_count, float* scores,
                                    cudaStream_t s) {
  const int64_t P = L / 4;
  const int64_t max_pools = (q_begin + q_count) / 4;  // elig(last query)
  if (max_pools == 0) return cudaSuccess;
  dim3 grid((unsigned)((max_pools + kSimtPB - 1) / kSimtPB), (unsigned)((q_count + kSimtQB - 1) / kSimtQB));
  const size_t smem = (size_t)kSimtQB * Hi * di * sizeof(float);
  indexer_simt_f32_kernel<<<grid, kSimtPB, smem, s>>>(q_idx, kpool, w, P, Hi, di, q_begin, q_count, scores);
  return cudaGetLastError();
}

}  // namespace dsa
