// attn_fwd.cu -- sparse attention forward over the selected pools.
//
// Page "SkyRL extends GLM-5.3-Flash training context to 1 million tokens",
// section "Model and bottleneck" (about 2048 keys read per query, so the
// attention itself is close to linear in L) and section "1. DSA truly sparse"
// (a truly sparse kernel; no positional encoding; 2051 = 4*512+3 keys).
//
// Keys of query t: the tokens of the pools in idx[t,:] (entries < 0 skipped),
// then the query's own partial pool 4*floor(t/4) .. t when t%4 != 3.
// O[t,h] = softmax(scale * Q[t,h] . K[keys]) V[keys]; LSE in natural log.
//
// bf16 kernel: one warp per (query, 16-head group).  A pool's 4 K rows (and
// 4 V rows) are one contiguous 1 KB block, so the warp gathers 4 pools = 16
// keys per step with 16-byte cp.async copies into an XOR-swizzled shared
// tile (2-stage ring per warp, no CTA-wide barriers).  The 16 heads of one
// query share every gathered key, which makes heads the M=16 side of
// m16n8k16 bf16 MMAs: S = Q K^T and O += P V, fp32 accumulation, online
// softmax in registers with a lazily moved base.  The kernel is bound by the
// L2->SM gather and by issue (about 16 flop per gathered byte), not by the MMAs.
//
// With an o_acc buffer (the ACC variant) the probabilities enter P V as two
// bf16 terms, P = hi + lo with hi = bf16(P) and lo = bf16(P - hi), so the fp32
// output carries P to about 2^-17 relative instead of bf16's 2^-9; o_acc then
// gives the backward D = dO . O without a recomputation pass.
#include "common.cuh"
#include "gather.cuh"
#include "launch.h"

namespace dsa {

template <int D, int NST_ = 3>
struct FwdCfg {
  static constexpr int NST = NST_;                               // gather stages per warp (2 or 3)
  static constexpr int WARPS = 4;
  static constexpr int ROW_BYTES = GatherCfg<D>::ROW_BYTES;
  static constexpr int TILE_BYTES = GatherCfg<D>::TILE_BYTES;
  static constexpr int STAGE_BYTES = GatherCfg<D>::STAGE_BYTES;
  static constexpr int SMEM = WARPS * NST * STAGE_BYTES;
};

// x = hi + lo for two fp32 values: hi their bf16 rounding, lo the bf16
// rounding of the (exact) fp32 remainder.
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16(x0, x1);
  lo = pack_bf16(x0 - __uint_as_float(hi << 16), x1 - __uint_as_float(hi & 0xFFFF0000u));
}

constexpr float kLazyLog2 = 8.f;   // the softmax base lags the running max by at most this (log2 units)

template <int D, int NST, int MINB, bool ACC>
__global__ void __launch_bounds__(128, MINB) attn_fwd_bf16_kernel(const __nv_bfloat16* __restrict__ Q,
                                                            const __nv_bfloat16* __restrict__ K,
                                                            const __nv_bfloat16* __restrict__ V,
                                                            const int32_t* __restrict__ idx,
                                                            __nv_bfloat16* __restrict__ O, float* __restrict__ LSE,
                                                            float* __restrict__ Oacc, int64_t L, int Hq, int k,
                                                            float scale_log2) {
  using C = FwdCfg<D, NST>;
  static_assert(NST == 2 || NST == 3, "the pool ring below is written for two or three stages");
  extern __shared__ __align__(128) unsigned char fwd_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int HG = Hq / 16;
  const int64_t items = L * HG;
  const int64_t item = items - 1 - ((int64_t)blockIdx.x * C::WARPS + warp);  // late queries first
  if (item < 0) return;
  const int64_t t = item / HG;
  const int hg = (int)(item % HG);
  const uint32_t wbase = smem_u32(fwd_smem) + warp * C::NST * C::STAGE_BYTES;
  const int32_t* irow = idx + t * k;
  const int ngroups = (k + 1 + 3) / 4;   // k selected slots + the partial-pool slot
  const int g = lane >> 2, qi = lane & 3;
  const GatherLane<D> gl = gather_lane<D>(lane);

  // Q fragments (A operand, rows = heads hg*16 .. +15).
  uint32_t qa[D / 16][4];
  {
    const uint32_t* q32 = reinterpret_cast<const uint32_t*>(Q + (t * Hq + hg * 16) * D);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const int c0 = (g * D + ks * 16 + 2 * qi) / 2, c1 = ((g + 8) * D + ks * 16 + 2 * qi) / 2;
      qa[ks][0] = __ldg(q32 + c0);
      qa[ks][1] = __ldg(q32 + c1);
      qa[ks][2] = __ldg(q32 + c0 + 4);
      qa[ks][3] = __ldg(q32 + c1 + 4);
    }
  }

  float o[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  // pools of the current step (pc) and, with three stages, of the next (pn)
  uint32_t pc[4], pn[4] = {0u, 0u, 0u, 0u};   // packed pool slots (gather.cuh)
  bool bad_idx = false;   // an idx entry outside the causal range (skipped, reported once)
  step_pools(irow, k, 0, t, pc, bad_idx);
  gather_step16<D>(wbase, K, V, pc, gl);
  cp_async_commit();
  if constexpr (NST == 3) {
    if (ngroups > 1) {
      step_pools(irow, k, 1, t, pn, bad_idx);
      gather_step16<D>(wbase + C::STAGE_BYTES, K, V, pn, gl);
    }
    cp_async_commit();
  }

  int raw_next = slot_raw(irow, k, NST - 1);   // idx entry of the first prefetch in the loop
  int stage = 0;
  for (int grp = 0; grp < ngroups; ++grp) {
    uint32_t pf[4] = {0u, 0u, 0u, 0u};
    {
      const int nx = grp + NST - 1;
      if (nx < ngroups) {
        step_pools_from(raw_next, k, nx, t, pf, bad_idx);
        const int st = stage + NST - 1 >= NST ? stage - 1 : stage + NST - 1;
        gather_step16<D>(wbase + st * C::STAGE_BYTES, K, V, pf, gl);
      }
      raw_next = slot_raw(irow, k, nx + 1);   // the next prefetch's idx entry, a step early
      cp_async_commit();
    }
    // visibility of this lane's S columns: keys nt*8 + 2*qi + {0,1}
    bool kv[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      // slot nt*2 + (qi >> 1), without dynamic register indexing
      const int nrows = slot_nrows((qi >> 1) ? pc[nt * 2 + 1] : pc[nt * 2]);
#pragma unroll
      for (int e = 0; e < 2; ++e) kv[nt][e] = 2 * (qi & 1) + e < nrows;
    }
    cp_async_wait<C::NST - 1>();
    __syncwarp();
    const uint32_t ks_base = wbase + stage * C::STAGE_BYTES;
    const uint32_t vs_base = ks_base + C::TILE_BYTES;

    // S = Q K^T as four independent accumulation chains (two per key octet,
    // even and odd k-steps) so consecutive MMAs do not wait on each other
    float s[2][4], s2[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[nt][e] = s2[nt][e] = 0.f;
    {
      const int mtx = lane >> 3, r = lane & 7;
      const int key = (mtx >> 1) * 8 + r;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int ch = 2 * ks + (mtx & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(ks_base + key * C::ROW_BYTES + ((ch ^ (key & 7)) << 4), b0, b1, b2, b3);
        if (ks & 1) {
          mma_bf16_16816(s2[0], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
          mma_bf16_16816(s2[1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
        } else {
          mma_bf16_16816(s[0], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
          mma_bf16_16816(s[1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
        }
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[nt][e] += s2[nt][e];
    }
    // online softmax (log2 domain); c0,c1 -> head g, c2,c3 -> head g+8.  The
    // scores stay unscaled (invisible keys masked to -inf) and the scale
    // enters with the exponent: p = 2^(s * scale_log2 - base), one FMA; the
    // step max is scaled once (scale > 0 keeps the order).
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      s[nt][0] = kv[nt][0] ? s[nt][0] : -INFINITY;
      s[nt][1] = kv[nt][1] ? s[nt][1] : -INFINITY;
      s[nt][2] = kv[nt][0] ? s[nt][2] : -INFINITY;
      s[nt][3] = kv[nt][1] ? s[nt][3] : -INFINITY;
      mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
      mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    mx0 *= scale_log2;
    mx1 *= scale_log2;
    // Lazy rescaling: the exponent base m moves only when the step's max
    // exceeds it by more than kLazyLog2 (so P <= 2^kLazyLog2 in fp32, and
    // O and l are rescaled rarely); LSE = m + log2(l) holds for any base.
    const bool up0 = mx0 > m0 + kLazyLog2, up1 = mx1 > m1 + kLazyLog2;
    const float mn0 = up0 ? mx0 : m0, mn1 = up1 ? mx1 : m1;
    const float base0 = mn0 == -INFINITY ? 0.f : mn0, base1 = mn1 == -INFINITY ? 0.f : mn1;
    const float a0 = up0 ? ex2_approx(m0 - base0) : 1.f, a1 = up1 ? ex2_approx(m1 - base1) : 1.f;
    m0 = mn0;
    m1 = mn1;
    float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      s[nt][0] = ex2_approx(fmaf(s[nt][0], scale_log2, -base0));
      s[nt][1] = ex2_approx(fmaf(s[nt][1], scale_log2, -base0));
      s[nt][2] = ex2_approx(fmaf(s[nt][2], scale_log2, -base1));
      s[nt][3] = ex2_approx(fmaf(s[nt][3], scale_log2, -base1));
      rs0 += s[nt][0] + s[nt][1];
      rs1 += s[nt][2] + s[nt][3];
    }
    l0 = l0 * a0 + rs0;
    l1 = l1 * a1 + rs1;
    // rescale O only when some row's running max moved (a == 1 otherwise, and
    // multiplying by 1 is exact, so skipping changes nothing)
    if (__any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        o[n][0] *= a0;
        o[n][1] *= a0;
        o[n][2] *= a1;
        o[n][3] *= a1;
      }
    }
    uint32_t pa0, pa1, pa2, pa3, pl0 = 0, pl1 = 0, pl2 = 0, pl3 = 0;
    if constexpr (ACC) {
      split_bf16x2(s[0][0], s[0][1], pa0, pl0);
      split_bf16x2(s[0][2], s[0][3], pa1, pl1);
      split_bf16x2(s[1][0], s[1][1], pa2, pl2);
      split_bf16x2(s[1][2], s[1][3], pa3, pl3);
    } else {
      pa0 = pack_bf16(s[0][0], s[0][1]);
      pa1 = pack_bf16(s[0][2], s[0][3]);
      pa2 = pack_bf16(s[1][0], s[1][1]);
      pa3 = pack_bf16(s[1][2], s[1][3]);
    }
    {
      const int mtx = lane >> 3, r = lane & 7;
      const int key = (mtx & 1) * 8 + r;
      // V fragments two 16-column blocks at a time: the four hi MMAs go before
      // the four lo MMAs, so MMAs into the same accumulator are four apart
#pragma unroll
      for (int j = 0; j < D / 16; j += 2) {
        const int ch = 2 * j + (mtx >> 1);
        uint32_t b0, b1, b2, b3, c0, c1, c2, c3;
        ldsm_x4_t(vs_base + key * C::ROW_BYTES + ((ch ^ (key & 7)) << 4), b0, b1, b2, b3);
        ldsm_x4_t(vs_base + key * C::ROW_BYTES + (((ch + 2) ^ (key & 7)) << 4), c0, c1, c2, c3);
        mma_bf16_16816(o[2 * j], pa0, pa1, pa2, pa3, b0, b1);
        mma_bf16_16816(o[2 * j + 1], pa0, pa1, pa2, pa3, b2, b3);
        mma_bf16_16816(o[2 * j + 2], pa0, pa1, pa2, pa3, c0, c1);
        mma_bf16_16816(o[2 * j + 3], pa0, pa1, pa2, pa3, c2, c3);
        if constexpr (ACC) {
          mma_bf16_16816(o[2 * j], pl0, pl1, pl2, pl3, b0, b1);
          mma_bf16_16816(o[2 * j + 1], pl0, pl1, pl2, pl3, b2, b3);
          mma_bf16_16816(o[2 * j + 2], pl0, pl1, pl2, pl3, c0, c1);
          mma_bf16_16816(o[2 * j + 3], pl0, pl1, pl2, pl3, c2, c3);
        }
      }
    }
    __syncwarp();
#pragma unroll
    for (int s4 = 0; s4 < 4; ++s4) {
      if constexpr (NST == 3) {
        pc[s4] = pn[s4];
        pn[s4] = pf[s4];
      } else {
        pc[s4] = pf[s4];
      }
    }
    stage = stage == NST - 1 ? 0 : stage + 1;
  }
  cp_async_wait<0>();
  if (bad_idx && lane == 0) record_error(DSA_DEV_ERR_BAD_INDEX);

  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const float inv0 = 1.f / l0, inv1 = 1.f / l1;
  __nv_bfloat16* orow0 = O + (t * Hq + hg * 16 + g) * D;
  __nv_bfloat16* orow1 = orow0 + 8 * D;
#pragma unroll
  for (int n = 0; n < D / 8; ++n) {
    *reinterpret_cast<uint32_t*>(orow0 + n * 8 + 2 * qi) = pack_bf16(o[n][0] * inv0, o[n][1] * inv0);
    *reinterpret_cast<uint32_t*>(orow1 + n * 8 + 2 * qi) = pack_bf16(o[n][2] * inv1, o[n][3] * inv1);
  }
  if constexpr (ACC) {
    float* arow0 = Oacc + (t * Hq + hg * 16 + g) * D + 2 * qi;
    float* arow1 = arow0 + 8 * D;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      __stcs(reinterpret_cast<float2*>(arow0 + n * 8), make_float2(o[n][0] * inv0, o[n][1] * inv0));
      __stcs(reinterpret_cast<float2*>(arow1 + n * 8), make_float2(o[n][2] * inv1, o[n][3] * inv1));
    }
  }
  if (qi == 0) {
    constexpr float kLn2 = 0.6931471805599453f;
    LSE[t * Hq + hg * 16 + g] = (m0 + log2f(l0)) * kLn2;
    LSE[t * Hq + hg * 16 + g + 8] = (m1 + log2f(l1)) * kLn2;
  }
}

// ------------------------------------------------------------ fp32 (SIMT)
// One CTA of 128 threads per query; keys in tiles of 32 staged in shared
// memory; S, online-softmax state and O for all Hq heads kept in SMEM.
constexpr int kF32Tile = 32;

__global__ void __launch_bounds__(128) attn_fwd_f32_kernel(const float* __restrict__ Q,
                                                           const float* __restrict__ K,
                                                           const float* __restrict__ V,
                                                           const int32_t* __restrict__ idx, float* __restrict__ O,
                                                           float* __restrict__ LSE, int64_t L, int Hq, int d,
                                                           int k, float scale) {
  extern __shared__ float f32_smem[];
  float* qs = f32_smem;                    // [Hq][d]
  float* ks = qs + Hq * d;                 // [32][d]
  float* vs = ks + kF32Tile * d;           // [32][d]
  float* os = vs + kF32Tile * d;           // [Hq][d]
  float* ss = os + Hq * d;                 // [Hq][32]
  float* ms = ss + Hq * kF32Tile;          // [Hq] running max
  float* ls = ms + Hq;                     // [Hq] running sum
  float* as = ls + Hq;                     // [Hq] rescale
  int64_t* keys = reinterpret_cast<int64_t*>(as + Hq + (Hq & 1));  // [32]
  const int64_t t = L - 1 - blockIdx.x;
  const int tid = threadIdx.x;
  for (int i = tid; i < Hq * d; i += blockDim.x) {
    qs[i] = Q[t * Hq * d + i];
    os[i] = 0.f;
  }
  for (int h = tid; h < Hq; h += blockDim.x) {
    ms[h] = -INFINITY;
    ls[h] = 0.f;
  }
  const int32_t* irow = idx + t * k;
  const int nkeys_max = 4 * (k + 1);
  for (int kb = 0; kb < nkeys_max; kb += kF32Tile) {
    __syncthreads();
    if (tid < kF32Tile) {
      const int kk = kb + tid;
      const int slot = kk >> 2, row = kk & 3;
      int64_t p = -1;
      if (slot < k) {
        p = irow[slot];
        if (p >= elig(t)) {
          record_error(DSA_DEV_ERR_BAD_INDEX);
          p = -1;
        }
        if (p < 0) p = -1;
      } else if (slot == k && (t & 3) != 3) {
        p = t >> 2;
      }
      const int64_t tok = 4 * p + row;
      keys[tid] = (p >= 0 && (slot != k || tok <= t)) ? tok : -1;
    }
    __syncthreads();
    for (int i = tid; i < kF32Tile * d; i += blockDim.x) {
      const int j = i / d, c = i % d;
      const int64_t key = keys[j];
      ks[i] = key >= 0 ? K[key * d + c] : 0.f;
      vs[i] = key >= 0 ? V[key * d + c] : 0.f;
    }
    __syncthreads();
    for (int i = tid; i < Hq * kF32Tile; i += blockDim.x) {
      const int h = i / kF32Tile, j = i % kF32Tile;
      float acc = 0.f;
      for (int c = 0; c < d; ++c) acc = fmaf(qs[h * d + c], ks[j * d + c], acc);
      ss[i] = keys[j] >= 0 ? acc * scale : -INFINITY;
    }
    __syncthreads();
    for (int h = tid; h < Hq; h += blockDim.x) {
      float mx = ms[h];
      for (int j = 0; j < kF32Tile; ++j) mx = fmaxf(mx, ss[h * kF32Tile + j]);
      const float base = mx == -INFINITY ? 0.f : mx;
      const float a = expf(ms[h] - base);
      float sum = ls[h] * a;
      for (int j = 0; j < kF32Tile; ++j) {
        const float pj = expf(ss[h * kF32Tile + j] - base);
        ss[h * kF32Tile + j] = pj;
        sum += pj;
      }
      ms[h] = mx;
      ls[h] = sum;
      as[h] = a;
    }
    __syncthreads();
    for (int i = tid; i < Hq * d; i += blockDim.x) {
      const int h = i / d, c = i % d;
      float acc = os[i] * as[h];
      for (int j = 0; j < kF32Tile; ++j) acc = fmaf(ss[h * kF32Tile + j], vs[j * d + c], acc);
      os[i] = acc;
    }
  }
  __syncthreads();
  for (int i = tid; i < Hq * d; i += blockDim.x) O[t * Hq * d + i] = os[i] / ls[i / d];
  for (int h = tid; h < Hq; h += blockDim.x) LSE[t * Hq + h] = ms[h] + logf(ls[h]);
}

// Gather stages per warp and CTAs per SM the kernel is compiled for.  Two
// stages (16 KB per warp) with registers capped for three 4-warp CTAs per SM
// measured 11.0 ms at L=131072, against 12.4 ms for three stages at two CTAs
// per SM: more warps hide more of the MMA and softmax latency.
constexpr int kFwdStages = 2;
constexpr int kFwdMinBlocks = 3;

template <int D, bool ACC>
static cudaError_t launch_fwd(int64_t blocks, const __nv_bfloat16* q, const __nv_bfloat16* k,
                              const __nv_bfloat16* v, const int32_t* idx, __nv_bfloat16* o, float* lse,
                              float* o_acc, int64_t L, int Hq, int kk, float scale_log2, cudaStream_t s) {
  constexpr int smem = FwdCfg<D, kFwdStages>::SMEM;
  auto kern = attn_fwd_bf16_kernel<D, kFwdStages, kFwdMinBlocks, ACC>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)blocks, 128, smem, s>>>(q, k, v, idx, o, lse, o_acc, L, Hq, kk, scale_log2);
  return cudaGetLastError();
}

cudaError_t launch_attn_fwd_bf16(int64_t L, int Hq, int d, int k, float scale, const void* q, const void* kk,
                                 const void* v, const int32_t* idx, void* o, float* lse, float* o_acc,
                                 cudaStream_t s) {
  const float scale_log2 = scale * 1.4426950408889634f;
  const int64_t items = L * (Hq / 16);
  const int64_t blocks = (items + 3) / 4;
  auto qp = static_cast<const __nv_bfloat16*>(q);
  auto kp = static_cast<const __nv_bfloat16*>(kk);
  auto vp = static_cast<const __nv_bfloat16*>(v);
  auto op = static_cast<__nv_bfloat16*>(o);
  if (d == 128)
    return o_acc ? launch_fwd<128, true>(blocks, qp, kp, vp, idx, op, lse, o_acc, L, Hq, k, scale_log2, s)
                 : launch_fwd<128, false>(blocks, qp, kp, vp, idx, op, lse, o_acc, L, Hq, k, scale_log2, s);
  if (d == 64)
    return o_acc ? launch_fwd<64, true>(blocks, qp, kp, vp, idx, op, lse, o_acc, L, Hq, k, scale_log2, s)
                 : launch_fwd<64, false>(blocks, qp, kp, vp, idx, op, lse, o_acc, L, Hq, k, scale_log2, s);
  return cudaErrorNotSupported;
}

cudaError_t launch_attn_fwd_f32(int64_t L, int Hq, int d, int k, float scale, const float* q, const float* kk,
                                const float* v, const int32_t* idx, float* o, float* lse, cudaStream_t s) {
  const size_t smem = sizeof(float) * ((size_t)Hq * d * 2 + 2 * kF32Tile * d + Hq * kF32Tile + 3 * Hq + 1) +
                      sizeof(int64_t) * kF32Tile + 16;
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  attn_fwd_f32_kernel<<<(unsigned)L, 128, smem, s>>>(q, kk, v, idx, o, lse, L, Hq, d, k, scale);
  return cudaGetLastError();
}

}  // namespace dsa
