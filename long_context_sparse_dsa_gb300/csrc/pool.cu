// pool.cu -- pool keys (page "SkyRL extends GLM-5.3-Flash training context to
// 1 million tokens", section "Model and bottleneck": the indexer works on one
// pool per 4 tokens).  kpool[p,:] = k_I[4p] + k_I[4p+1] + k_I[4p+2] + k_I[4p+3],
// added in that order in fp32 and rounded once to the layer dtype.
//
// HBM-bound and tiny: each thread moves 16 bytes of one pool row (8 bf16 or 4
// fp32 values) from each of the pool's 4 token rows, so every load and store
// is a coalesced 16-byte access.
//
// Gated variant (same page, section "3. Context parallelism (CP)", which names
// k-pool gate scores aligned with the keys and defines nothing more): each
// token's key is weighted by a per-token fp32 gate before the sum,
// kpool[p,:] = sum_j gate[4p+j] * k_I[4p+j,:], as one fused multiply-add per
// token from zero in token order, rounded once.  All-one gates give the plain
// pool bit for bit.
#include "common.cuh"
#include "launch.h"

namespace dsa {

template <typename T>
struct Vec16;
template <>
struct Vec16<float> {
  static constexpr int N = 4;
};
template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
};

template <typename T>
__device__ __forceinline__ void unpack16(const uint4& u, float* f);
template <>
__device__ __forceinline__ void unpack16<float>(const uint4& u, float* f) {
  f[0] = __uint_as_float(u.x);
  f[1] = __uint_as_float(u.y);
  f[2] = __uint_as_float(u.z);
  f[3] = __uint_as_float(u.w);
}
template <>
__device__ __forceinline__ void unpack16<__nv_bfloat16>(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
template <typename T>
__device__ __forceinline__ uint4 pack16(const float* f);
template <>
__device__ __forceinline__ uint4 pack16<float>(const float* f) {
  return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
}
template <>
__device__ __forceinline__ uint4 pack16<__nv_bfloat16>(const float* f) {
  return make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]), pack_bf16(f[6], f[7]));
}

template <typename T, bool GATED>
__global__ void pool_keys_kernel(const uint4* __restrict__ k_idx, const float* __restrict__ gate,
                                 uint4* __restrict__ kpool, int64_t P, int vec_per_row) {
  constexpr int N = Vec16<T>::N;
  const int64_t total = P * vec_per_row;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t p = i / vec_per_row;
    const int c = (int)(i - p * vec_per_row);
    const uint4* src = k_idx + (4 * p) * vec_per_row + c;
    float acc[N], x[N];
    if constexpr (GATED) {
      const float4 g = __ldg(reinterpret_cast<const float4*>(gate) + p);   // the pool's 4 gates
      const float gj[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
      for (int e = 0; e < N; ++e) acc[e] = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        unpack16<T>(__ldg(src + j * vec_per_row), x);
#pragma unroll
        for (int e = 0; e < N; ++e) acc[e] = __fmaf_rn(gj[j], x[e], acc[e]);
      }
    } else {
      unpack16<T>(__ldg(src), acc);
#pragma unroll
      for (int j = 1; j < 4; ++j) {
        unpack16<T>(__ldg(src + j * vec_per_row), x);
#pragma unroll
        for (int e = 0; e < N; ++e) acc[e] = __fadd_rn(acc[e], x[e]);
      }
    }
    kpool[i] = pack16<T>(acc);
  }
}

cudaError_t launch_pool_keys(bool bf16, int64_t L, int di, const void* k_idx, const float* gate, void* kpool,
                             cudaStream_t s) {
  const int64_t P = L / 4;
  const int vec = bf16 ? di / 8 : di / 4;
  const int64_t total = P * vec;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = (int64_t)device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  auto src = static_cast<const uint4*>(k_idx);
  auto dst = static_cast<uint4*>(kpool);
  if (bf16) {
    if (gate)
      pool_keys_kernel<__nv_bfloat16, true><<<(unsigned)blocks, threads, 0, s>>>(src, gate, dst, P, vec);
    else
      pool_keys_kernel<__nv_bfloat16, false><<<(unsigned)blocks, threads, 0, s>>>(src, nullptr, dst, P, vec);
  } else {
    if (gate)
      pool_keys_kernel<float, true><<<(unsigned)blocks, threads, 0, s>>>(src, gate, dst, P, vec);
    else
      pool_keys_kernel<float, false><<<(unsigned)blocks, threads, 0, s>>>(src, nullptr, dst, P, vec);
  }
  return cudaGetLastError();
}

}  // namespace dsa
