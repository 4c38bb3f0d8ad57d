// probe.cu -- traffic replay of the attention kernels (dsa_probe_traffic).
//
// The attention kernels are bound by L2 traffic: the 16-byte pool gathers of
// K and V (a table of L*d*2*2 bytes that stays in L2 at L = 131072) and, in
// the backward, the fp32 bulk reductions of dK and dV rows.  This kernel walks
// the same steps over the same selection with the same instructions
// (step_pools and gather_step16 for the copies, one cp.reduce.async.bulk per
// pool slot and tensor) and the same occupancy, and does no arithmetic, so
// its time is the floor for the kernels' data movement and its rate the
// ceiling they are measured against.
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
};

template <int D, bool RED>
__global__ void __launch_bounds__(32 * kProbeWarps) probe_traffic_kernel(const __nv_bfloat16* __restrict__ K,
                                                                        const __nv_bfloat16* __restrict__ V,
                                                                        const int32_t* __restrict__ idx,
                                                                        float* __restrict__ dK,
                                                                        float* __restrict__ dV, int64_t L, int Hq,
                                                                        int k) {
  using C = ProbeCfg<D, RED>;
  extern __shared__ __align__(128) unsigned char probe_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int HG = Hq / 16;
  const int64_t items = L * HG;
  const int64_t item = items - 1 - ((int64_t)blockIdx.x * kProbeWarps + warp);   // late queries first
  if (item < 0) return;
  const int64_t t = item / HG;
  const uint32_t wbase = smem_u32(probe_smem) + warp * C::WARP_BYTES;
  const uint32_t rbase = wbase + kProbeStages * GatherCfg<D>::STAGE_BYTES;
  if (RED) {
    float* r = reinterpret_cast<float*>(probe_smem + warp * C::WARP_BYTES + kProbeStages * GatherCfg<D>::STAGE_BYTES);
    for (int i = lane; i < 4 * 4 * D; i += 32) r[i] = 1e-30f;
    fence_proxy_async_shared();
    __syncwarp();
  }
  const int32_t* irow = idx + t * k;
  const int nsteps = (k + 1 + 3) / 4;   // k selected slots + the partial-pool slot
  const GatherLane<D> gl = gather_lane<D>(lane);
  bool bad = false;
  uint32_t pc[4];
  step_pools(irow, k, 0, t, pc, bad);
  gather_step16<D>(wbase, K, V, pc, gl);
  cp_async_commit();
  int stage = 0;
  for (int step = 0; step < nsteps; ++step) {
    uint32_t pf[4] = {0u, 0u, 0u, 0u};
    if (step + 1 < nsteps) {
      step_pools(irow, k, step + 1, t, pf, bad);
      gather_step16<D>(wbase + (stage ^ 1) * GatherCfg<D>::STAGE_BYTES, K, V, pf, gl);
    }
    cp_async_commit();
    cp_async_wait<kProbeStages - 1>();
    __syncwarp();
    if (RED) {
      const uint32_t mine = (lane & 3) == 0 ? pc[0] : (lane & 3) == 1 ? pc[1] : (lane & 3) == 2 ? pc[2] : pc[3];
      const bool on = lane < 4 && slot_nrows(mine) > 0;
      probe_wait_read(lane < 4);
      const int64_t row = 4 * (int64_t)slot_pool(mine);
      const uint32_t bytes = (uint32_t)(slot_nrows(mine) * D * 4);
      probe_red_add_f32(dV + row * D, rbase + (lane & 3) * C::RED_POOL, bytes, on);
      probe_red_add_f32(dK + row * D, rbase + (lane & 3) * C::RED_POOL, bytes, on);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) pc[i] = pf[i];
    stage ^= 1;
  }
  cp_async_wait<0>();
  if (RED) bulk_wait<0>();
}

template <int D, bool RED>
cudaError_t launch_probe(const dsa_dims* d, const void* k, const void* v, const int32_t* idx, float* dk, float* dv,
                         cudaStream_t s) {
  using C = ProbeCfg<D, RED>;
  auto kern = probe_traffic_kernel<D, RED>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const int64_t items = d->L * (d->Hq / 16);
  const int64_t blocks = (items + kProbeWarps - 1) / kProbeWarps;
  kern<<<(unsigned)blocks, 32 * kProbeWarps, C::SMEM, s>>>(static_cast<const __nv_bfloat16*>(k),
                                                            static_cast<const __nv_bfloat16*>(v), idx, dk, dv, d->L,
                                                            d->Hq, d->k);
  return cudaGetLastError();
}

dsa_status probe_fail(dsa_status st, const char* msg) {
  set_last_error_message(msg);
  return st;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" dsa_status dsa_probe_traffic(const dsa_dims* dims, const void* k, const void* v, const int32_t* idx,
                                        float* dk, float* dv, dsa_stream_t stream) {
  dsa::set_last_error_message("");
  dsa_status st = dsa_validate_dims(dims, 0);
  if (st != DSA_OK) return st;
  if (dims->dtype != DSA_BF16) return probe_fail(DSA_ERR_UNSUPPORTED, "dsa_probe_traffic: bf16 layers only");
  if (!aligned16(k) || !aligned16(v) || !aligned16(idx))
    return probe_fail(DSA_ERR_INVALID_ARG, "dsa_probe_traffic: k, v and idx must be 16-byte aligned device pointers");
  if ((dk == nullptr) != (dv == nullptr))
    return probe_fail(DSA_ERR_INVALID_ARG, "dsa_probe_traffic: give both dk and dv, or neither");
  const bool red = dk != nullptr;
  if (red && (!aligned16(dk) || !aligned16(dv)))
    return probe_fail(DSA_ERR_INVALID_ARG, "dsa_probe_traffic: dk and dv must be 16-byte aligned");
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e;
  if (dims->d == 128)
    e = red ? launch_probe<128, true>(dims, k, v, idx, dk, dv, s) : launch_probe<128, false>(dims, k, v, idx, dk, dv, s);
  else
    e = red ? launch_probe<64, true>(dims, k, v, idx, dk, dv, s) : launch_probe<64, false>(dims, k, v, idx, dk, dv, s);
  if (e != cudaSuccess) {
    dsa::set_last_error_message(cudaGetErrorString(e));
    return DSA_ERR_CUDA;
  }
  return DSA_OK;
}
