// probe.cu -- traffic replay of the attention kernels (dsa_probe_traffic).
//
// The attention kernels are bound by L2 traffic: the 16-byte pool gathers of
// K and V (a 64 MiB table at L=131072 that stays in L2) and, in the backward,
// the fp32 bulk reductions of dK and dV rows.  This kernel moves the same
// traffic with the same instructions -- gather_step16 for the copies, one
// cp.reduce.async.bulk per pool and tensor -- and no arithmetic, so its rate
// is the ceiling the attention kernels are measured against.  Pools are drawn
// uniformly at random by a counter-based hash (splitmix64's finaliser).
#include "../../include/dsa_probe.h"
#include "common.cuh"
#include "gather.cuh"
#include "launch.h"

namespace dsa {
void set_last_error_message(const char* msg);  // api.cu
}

namespace {

using namespace dsa;

constexpr int kProbeWarps = 4;
constexpr int kProbeStages = 2;
constexpr int kProbeRedInFlight = 4;   // bulk groups a lane may still be reading before it issues more

__device__ __forceinline__ uint64_t mix64(uint64_t x) {
  x += 0x9E3779B97F4A7C15ull;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
  return x ^ (x >> 31);
}

__device__ __forceinline__ void probe_red_add_f32(float* gdst, uint32_t ssrc, uint32_t bytes, bool pred) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %3, 0;\n"
      "@p cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;\n"
      "@p cp.async.bulk.commit_group;\n}\n" ::"l"(gdst),
      "r"(ssrc), "r"(bytes), "r"((uint32_t)pred)
      : "memory");
}
__device__ __forceinline__ void probe_wait_read(bool pred) {
  asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %0, 0;\n@p cp.async.bulk.wait_group.read %1;\n}\n" ::"r"(
                   (uint32_t)pred),
               "n"(kProbeRedInFlight)
               : "memory");
}

template <int D, bool RED>
struct ProbeCfg {
  static constexpr int RED_POOL = 4 * D * 4;   // one pool's fp32 rows
  static constexpr int WARP_BYTES = kProbeStages * GatherCfg<D>::STAGE_BYTES + (RED ? 4 * RED_POOL : 0);
  static constexpr int SMEM = kProbeWarps * WARP_BYTES;
  static constexpr int CTAS_PER_SM = RED ? 2 : 3;
};

template <int D, bool RED>
__global__ void __launch_bounds__(32 * kProbeWarps) probe_traffic_kernel(const __nv_bfloat16* __restrict__ K,
                                                                        const __nv_bfloat16* __restrict__ V,
                                                                        float* __restrict__ dK,
                                                                        float* __restrict__ dV, int64_t P,
                                                                        int64_t steps, uint64_t seed) {
  using C = ProbeCfg<D, RED>;
  extern __shared__ __align__(128) unsigned char probe_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t wbase = smem_u32(probe_smem) + warp * C::WARP_BYTES;
  const uint32_t rbase = wbase + kProbeStages * GatherCfg<D>::STAGE_BYTES;
  if (RED) {
    float* r = reinterpret_cast<float*>(probe_smem + warp * C::WARP_BYTES + kProbeStages * GatherCfg<D>::STAGE_BYTES);
    for (int i = lane; i < 4 * 4 * D; i += 32) r[i] = 1e-30f;
    fence_proxy_async_shared();
    __syncwarp();
  }
  const GatherLane<D> gl = gather_lane<D>(lane);
  const int64_t nw = (int64_t)gridDim.x * kProbeWarps;
  int stage = 0;
  for (int64_t s = (int64_t)blockIdx.x * kProbeWarps + warp; s < steps; s += nw) {
    const uint64_t h = mix64(seed ^ (uint64_t)(s * 4 + (lane & 3)));
    const uint32_t mine = ((uint32_t)(h % (uint64_t)P) << 3) | 4u;   // a whole pool, 4 visible rows
    uint32_t slots[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) slots[i] = __shfl_sync(0xffffffffu, mine, i);
    gather_step16<D>(wbase + stage * GatherCfg<D>::STAGE_BYTES, K, V, slots, gl);
    cp_async_commit();
    cp_async_wait<kProbeStages - 1>();
    __syncwarp();
    if (RED) {
      const bool on = lane < 4;
      probe_wait_read(on);
      const int64_t row = 4 * (int64_t)slot_pool(mine);
      probe_red_add_f32(dV + row * D, rbase + (lane & 3) * C::RED_POOL, C::RED_POOL, on);
      probe_red_add_f32(dK + row * D, rbase + (lane & 3) * C::RED_POOL, C::RED_POOL, on);
    }
    stage ^= 1;
  }
  cp_async_wait<0>();
  if (RED) bulk_wait<0>();
}

template <int D, bool RED>
cudaError_t launch_probe(int64_t L, const void* k, const void* v, float* dk, float* dv, int64_t steps,
                         uint64_t seed, cudaStream_t s) {
  using C = ProbeCfg<D, RED>;
  auto kern = probe_traffic_kernel<D, RED>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  int64_t grid = (int64_t)device_sm_count() * C::CTAS_PER_SM;
  const int64_t need = (steps + kProbeWarps - 1) / kProbeWarps;
  if (grid > need) grid = need;
  kern<<<(unsigned)grid, 32 * kProbeWarps, C::SMEM, s>>>(static_cast<const __nv_bfloat16*>(k),
                                                          static_cast<const __nv_bfloat16*>(v), dk, dv, L / 4,
                                                          steps, seed);
  return cudaGetLastError();
}

dsa_status probe_fail(dsa_status st, const char* msg) {
  set_last_error_message(msg);
  return st;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" dsa_status dsa_probe_traffic(int32_t d, int64_t L, const void* k, const void* v, float* dk, float* dv,
                                        int64_t steps, uint64_t seed, dsa_stream_t stream) {
  dsa::set_last_error_message("");
  if (d != 64 && d != 128) return probe_fail(DSA_ERR_UNSUPPORTED, "dsa_probe_traffic: d must be 64 or 128");
  if (L < 4 || L % 4 != 0 || L > ((int64_t)1 << 31))
    return probe_fail(DSA_ERR_INVALID_ARG, "dsa_probe_traffic: L must be a multiple of 4 in [4, 2^31]");
  if (steps < 1) return probe_fail(DSA_ERR_INVALID_ARG, "dsa_probe_traffic: steps must be >= 1");
  if (!aligned16(k) || !aligned16(v))
    return probe_fail(DSA_ERR_INVALID_ARG, "dsa_probe_traffic: k and v must be 16-byte aligned device pointers");
  if ((dk == nullptr) != (dv == nullptr))
    return probe_fail(DSA_ERR_INVALID_ARG, "dsa_probe_traffic: give both dk and dv, or neither");
  const bool red = dk != nullptr;
  if (red && (!aligned16(dk) || !aligned16(dv)))
    return probe_fail(DSA_ERR_INVALID_ARG, "dsa_probe_traffic: dk and dv must be 16-byte aligned");
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e;
  if (d == 128)
    e = red ? launch_probe<128, true>(L, k, v, dk, dv, steps, seed, s)
            : launch_probe<128, false>(L, k, v, dk, dv, steps, seed, s);
  else
    e = red ? launch_probe<64, true>(L, k, v, dk, dv, steps, seed, s)
            : launch_probe<64, false>(L, k, v, dk, dv, steps, seed, s);
  if (e != cudaSuccess) {
    dsa::set_last_error_message(cudaGetErrorString(e));
    return DSA_ERR_CUDA;
  }
  return DSA_OK;
}
