// attn_bwd.cu -- sparse attention backward (bf16 inputs, fp32 gradients).
//
// Page "SkyRL extends GLM-5.3-Flash training context to 1 million tokens",
// section "1. DSA truly sparse" (the sparse kernel runs forward and backward)
// and section "2. Activation recomputation and offload" (the layer is
// recomputed from saved inputs, which is why only idx and LSE are kept).
//
// For query t, head h, key j in keys(t) (as in the forward):
//   P = exp(scale*Q.K[j] - LSE),  D = dO . O,  dP = dO . V[j],
//   dS = P (dP - D),  dQ = scale sum_j dS K[j],
//   dK[j] += scale sum_h dS Q[t,h],  dV[j] += sum_h P dO[t,h].
// The selection is piecewise constant, so q_I, k_I and w get no gradient.
//
// Two kernels, one warp per (query, 16-head group) each, with the same 16-key
// gather pipeline as the forward.  The first forms D[t,h] = sum_j P_j dP_j
// into a [L, Hq] fp32 workspace; the second does everything else, so the
// atomic traffic of the second is not interleaved with a pass that has none.
// When the forward kept its output in fp32 with P carried beyond bf16 (o_acc),
// the second kernel forms D = dO . o_acc itself and the first is not launched.
// dQ stays in registers for the whole query.  Per 16-key step
// the warp computes the 16x16 S and dP tiles with m16n8k16 MMAs (heads on M),
// then the 16-key x d tiles of dK and dV with the keys on M: the transposed
// P and dS operands are built in registers with movmatrix, and Q / dO come
// from a per-warp swizzled shared copy.  Those sums collect contributions
// from every query that selected a key, so P and scale*dS enter the dK/dV
// products as two bf16 terms each, x = hi + lo with hi = bf16(x) and
// lo = bf16(x - hi) (about 2^-17 relative instead of bf16's 2^-9), against
// the exact bf16 Q and dO.  Every operand keeps the fp32 exponent range, so
// loss-scaled gradients (dO ~ 1e-6) and inputs beyond fp16's 65504 are
// carried without overflow or underflow.
// The tile is gathered pool-interleaved (row m = token m >> 2 of slot m & 3),
// so each finished 16-key dK/dV tile can be staged in shared memory as four
// pool blocks (padded so the fragment writes do not conflict) and each pool's
// visible rows are added to global memory by one bulk fp32 reduction of the
// TMA engine (cp.reduce.async.bulk, up to 4*D contiguous floats).
// Row-contiguous reductions are absorbed by the L2 about 1.6x faster than
// fragment-shaped ones; the summation order across queries is not fixed.
#include "common.cuh"
#include "gather.cuh"
#include "launch.h"

namespace dsa {

// PASS 1 forms D[t,h] = sum_j P_j dP_j into a [L, Hq] fp32 buffer; PASS 2
// forms dS and the gradients.  PASS 2 also keeps swizzled copies of Q and dO.
// PASS 3 (the deterministic backward's query-major half) forms dQ only, and
// when it takes D from o_acc it also stores D in the [L, Hq] buffer for the
// key-major half.
// Gather stages per warp and warps per CTA (two CTAs per SM either way:
// shared memory allows 2 x 4 warps x 2 stages or 2 x 3 warps x 3 stages).
// Measured at L=131072: 45.8 ms for two stages at four warps, 46.6 ms for
// three stages at three warps -- the extra tile in flight does not make up
// for a quarter fewer warps.
constexpr int kBwdStages = 2;
constexpr int kBwdWarps = 4;

template <int D, int PASS>
struct BwdCfg {
  static constexpr int ROW_BYTES = GatherCfg<D>::ROW_BYTES;
  static constexpr int CHUNKS = GatherCfg<D>::CHUNKS;
  static constexpr int TILE_BYTES = GatherCfg<D>::TILE_BYTES;
  static constexpr int STAGE_BYTES = GatherCfg<D>::STAGE_BYTES;
  // A consumed stage also holds a 16-key fp32 dK or dV tile as four pool
  // blocks POOL_PITCH bytes apart, each the pool's four rows back to back (one
  // contiguous bulk reduction per pool); the 32 bytes between blocks keep the
  // fragment writes free of bank conflicts.  Each stage is padded to fit it.
  static constexpr int RED_ROW = D * 4;
  static constexpr int POOL_PITCH = 4 * RED_ROW + 32;
  static constexpr int STAGE_PITCH = 4 * POOL_PITCH > STAGE_BYTES ? 4 * POOL_PITCH : STAGE_BYTES;
  static constexpr int NST = kBwdStages;      // gather stages per warp (2 or 3)
  static constexpr int WARPS = kBwdWarps;     // warps (queries) per CTA
  static constexpr int WARP_BYTES = NST * STAGE_PITCH + (PASS == 2 ? 2 * TILE_BYTES : 0);
  static constexpr int SMEM = WARPS * WARP_BYTES;
  static_assert(STAGE_PITCH % 16 == 0 && WARP_BYTES % 16 == 0 && POOL_PITCH % 16 == 0, "16-byte alignment");
};

// Advance the pool-slot ring by one step: current <- next (<- fetched).
template <int NST>
__device__ __forceinline__ void rotate_slots(uint32_t (&pc)[4], uint32_t (&pn)[4], const uint32_t (&pf)[4]) {
#pragma unroll
  for (int s4 = 0; s4 < 4; ++s4) {
    if constexpr (NST == 3) {
      pc[s4] = pn[s4];
      pn[s4] = pf[s4];
    } else {
      pc[s4] = pf[s4];
    }
  }
}

// Bulk (TMA-engine) fp32 add of `bytes` contiguous shared-memory bytes into
// global memory, then a commit of this thread's bulk group; both only where
// `pred` holds.
__device__ __forceinline__ void bulk_red_add_f32_if(float* gdst, uint32_t ssrc, uint32_t bytes, bool pred) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %3, 0;\n"
      "@p cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;\n"
      "@p cp.async.bulk.commit_group;\n}\n" ::"l"(gdst),
      "r"(ssrc), "r"(bytes), "r"((uint32_t)pred)
      : "memory");
}
// Wait (where `pred` holds) until this thread's bulk groups no longer read shared memory.
__device__ __forceinline__ void bulk_wait_read0_if(bool pred) {
  asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %0, 0;\n@p cp.async.bulk.wait_group.read 0;\n}\n" ::"r"(
                   (uint32_t)pred)
               : "memory");
}

// x = hi + lo for two fp32 values: hi their bf16 rounding, lo the bf16
// rounding of the (exact) fp32 remainder.
__device__ __forceinline__ void split_bf16x2_bwd(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16(x0, x1);
  lo = pack_bf16(x0 - __uint_as_float(hi << 16), x1 - __uint_as_float(hi & 0xFFFF0000u));
}

template <int D, int PASS>
__global__ void __launch_bounds__(32 * kBwdWarps) attn_bwd_bf16_kernel(
    const __nv_bfloat16* __restrict__ Q, const __nv_bfloat16* __restrict__ K, const __nv_bfloat16* __restrict__ V,
    const int32_t* __restrict__ idx, const float* __restrict__ LSE, const __nv_bfloat16* __restrict__ dO,
    const float* __restrict__ Oacc, float* __restrict__ Dbuf, float* __restrict__ dQ, float* __restrict__ dK,
    float* __restrict__ dV, int64_t L, int Hq, int k, float scale, float scale_log2) {
  using C = BwdCfg<D, PASS>;
  extern __shared__ __align__(128) unsigned char bwd_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int HG = Hq / 16;
  const int64_t items = L * HG;
  const int64_t item = items - 1 - ((int64_t)blockIdx.x * C::WARPS + warp);
  if (item < 0) return;
  const int64_t t = item / HG;
  const int hg = (int)(item % HG);
  const uint32_t wbase = smem_u32(bwd_smem) + warp * C::WARP_BYTES;
  const uint32_t qs = wbase + C::NST * C::STAGE_PITCH;
  const uint32_t dos = qs + C::TILE_BYTES;
  const int32_t* irow = idx + t * k;
  const int nslots = k + 1;
  const int ngroups = (nslots + 3) / 4;
  const int g = lane >> 2, qi = lane & 3;
  const int64_t row0 = t * Hq + hg * 16;  // first (t, head) row of this warp

  // Per-warp swizzled bf16 copies of Q and dO (16 heads x D), 16-byte chunks;
  // the B operands of the dK and dV products.
  if (PASS == 2) {
    const uint4* q4 = reinterpret_cast<const uint4*>(Q + row0 * D);
    const uint4* d4 = reinterpret_cast<const uint4*>(dO + row0 * D);
    unsigned char* qsp = bwd_smem + (qs - smem_u32(bwd_smem));
    unsigned char* dsp = bwd_smem + (dos - smem_u32(bwd_smem));
    for (int c = lane; c < 16 * C::CHUNKS; c += 32) {
      const int r = c / C::CHUNKS, ch = c % C::CHUNKS;
      const int off = r * C::ROW_BYTES + ((ch ^ (r & 7)) << 4);
      *reinterpret_cast<uint4*>(qsp + off) = __ldg(q4 + c);
      *reinterpret_cast<uint4*>(dsp + off) = __ldg(d4 + c);
    }
  }
  constexpr float kLog2e = 1.4426950408889634f;
  const float lse_g = __ldg(LSE + row0 + g) * kLog2e;
  const float lse_g8 = __ldg(LSE + row0 + g + 8) * kLog2e;
  __syncwarp();

  // A fragments of Q and dO (rows = heads), bf16, straight from global memory.
  uint32_t qa[D / 16][4], da[D / 16][4];
  {
    const uint32_t* q32 = reinterpret_cast<const uint32_t*>(Q + row0 * D);
    const uint32_t* d32 = reinterpret_cast<const uint32_t*>(dO + row0 * D);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const int c0 = (g * D + ks * 16 + 2 * qi) / 2, c1 = ((g + 8) * D + ks * 16 + 2 * qi) / 2;
      qa[ks][0] = __ldg(q32 + c0);
      qa[ks][1] = __ldg(q32 + c1);
      qa[ks][2] = __ldg(q32 + c0 + 4);
      qa[ks][3] = __ldg(q32 + c1 + 4);
      da[ks][0] = __ldg(d32 + c0);
      da[ks][1] = __ldg(d32 + c1);
      da[ks][2] = __ldg(d32 + c0 + 4);
      da[ks][3] = __ldg(d32 + c1 + 4);
    }
  }

  float dq[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n) dq[n][0] = dq[n][1] = dq[n][2] = dq[n][3] = 0.f;

  // One pass over the key groups.  PASS 1 accumulates D[h] = sum_j P_j dP_j
  // (equal to dO . O, but from the exact P and dP rather than the
  // bf16-rounded O); PASS 2 reads it back and forms dS and the gradients.
  static_assert(C::NST == 2 || C::NST == 3, "the pool ring below is written for two or three stages");
  const GatherLane<D> gl = gather_lane<D>(lane);
  const int nsteps = ngroups;
  // packed pool slots (gather.cuh) of the current step and, with three stages, the next
  uint32_t pc[4], pn[4] = {0u, 0u, 0u, 0u};
  bool bad_idx = false;   // an idx entry outside the causal range (skipped, reported once)
  step_pools(irow, k, 0, t, pc, bad_idx);
  gather_step16_il<D>(wbase, K, V, pc, gl);
  cp_async_commit();
  if constexpr (C::NST == 3) {
    if (nsteps > 1) {
      step_pools(irow, k, 1, t, pn, bad_idx);
      gather_step16_il<D>(wbase + C::STAGE_PITCH, K, V, pn, gl);
    }
    cp_async_commit();
  }
  float Dg = 0.f, Dg8 = 0.f;
  if (PASS >= 2) {
    if (Oacc != nullptr) {
      // D = dO . O over this lane's dO fragment columns (ks*16 + 2qi + {0,1}
      // and ks*16 + 8 + 2qi + {0,1}), then summed over the quad
      const float* a0 = Oacc + (row0 + g) * D + 2 * qi;
      const float* a8 = a0 + 8 * D;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const float2 x0 = __ldg(reinterpret_cast<const float2*>(a0 + ks * 16));
        const float2 x1 = __ldg(reinterpret_cast<const float2*>(a0 + ks * 16 + 8));
        const float2 y0 = __ldg(reinterpret_cast<const float2*>(a8 + ks * 16));
        const float2 y1 = __ldg(reinterpret_cast<const float2*>(a8 + ks * 16 + 8));
        Dg = fmaf(__uint_as_float(da[ks][0] << 16), x0.x, Dg);
        Dg = fmaf(__uint_as_float(da[ks][0] & 0xFFFF0000u), x0.y, Dg);
        Dg = fmaf(__uint_as_float(da[ks][2] << 16), x1.x, Dg);
        Dg = fmaf(__uint_as_float(da[ks][2] & 0xFFFF0000u), x1.y, Dg);
        Dg8 = fmaf(__uint_as_float(da[ks][1] << 16), y0.x, Dg8);
        Dg8 = fmaf(__uint_as_float(da[ks][1] & 0xFFFF0000u), y0.y, Dg8);
        Dg8 = fmaf(__uint_as_float(da[ks][3] << 16), y1.x, Dg8);
        Dg8 = fmaf(__uint_as_float(da[ks][3] & 0xFFFF0000u), y1.y, Dg8);
      }
      Dg += __shfl_xor_sync(0xffffffffu, Dg, 1);
      Dg += __shfl_xor_sync(0xffffffffu, Dg, 2);
      Dg8 += __shfl_xor_sync(0xffffffffu, Dg8, 1);
      Dg8 += __shfl_xor_sync(0xffffffffu, Dg8, 2);
    } else {
      Dg = __ldg(Dbuf + row0 + g);
      Dg8 = __ldg(Dbuf + row0 + g + 8);
    }
  }

  int raw_next = slot_raw(irow, k, C::NST - 1);   // idx entry of the first prefetch in the loop
  int stage = 0;
  for (int step = 0; step < nsteps; ++step) {
    constexpr bool pass1 = PASS == 1;
    uint32_t pf[4] = {0u, 0u, 0u, 0u};
    {
      const int nx = step + C::NST - 1;
      if (nx < nsteps) {
        // the stage being refilled is the one the previous step consumed and
        // staged its dK tile in: those bulk reductions must have read it
        if (PASS == 2) {
          bulk_wait_read0_if(lane < 4);
          __syncwarp();
        }
        const int st = stage == 0 ? C::NST - 1 : stage - 1;
        step_pools_from(raw_next, k, nx, t, pf, bad_idx);
        gather_step16_il<D>(wbase + st * C::STAGE_PITCH, K, V, pf, gl);
      }
      raw_next = slot_raw(irow, k, nx + 1);   // the next prefetch's idx entry, a step early
      cp_async_commit();
    }
    // visibility of this lane's S/dP columns (keys nt*8 + 2qi + e)
    bool kv[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      // the tile is pool-interleaved: column n = nt*8 + 2qi + e is token n >> 2
      // of slot n & 3 = 2(qi & 1) + e
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const uint32_t sl = (qi & 1) ? (e ? pc[3] : pc[2]) : (e ? pc[1] : pc[0]);
        kv[nt][e] = 2 * nt + (qi >> 1) < slot_nrows(sl);
      }
    }
    cp_async_wait<C::NST - 1>();
    __syncwarp();
    const uint32_t ks_base = wbase + stage * C::STAGE_PITCH;
    const uint32_t vs_base = ks_base + C::TILE_BYTES;

    // S = Q K^T and dP = dO V^T (heads x 16 keys), each as two independent
    // accumulation chains (even / odd k-steps)
    float s[2][4], dp[2][4], s2[2][4], dp2[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[nt][e] = dp[nt][e] = s2[nt][e] = dp2[nt][e] = 0.f;
    {
      const int mtx = lane >> 3, r = lane & 7;
      const int key = (mtx >> 1) * 8 + r;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int ch = 2 * ks + (mtx & 1);
        const uint32_t off = key * C::ROW_BYTES + ((ch ^ (key & 7)) << 4);
        uint32_t b0, b1, b2, b3, c0, c1, c2, c3;
        ldsm_x4(ks_base + off, b0, b1, b2, b3);
        ldsm_x4(vs_base + off, c0, c1, c2, c3);
        if (ks & 1) {
          mma_bf16_16816(s2[0], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
          mma_bf16_16816(s2[1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
          mma_bf16_16816(dp2[0], da[ks][0], da[ks][1], da[ks][2], da[ks][3], c0, c1);
          mma_bf16_16816(dp2[1], da[ks][0], da[ks][1], da[ks][2], da[ks][3], c2, c3);
        } else {
          mma_bf16_16816(s[0], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
          mma_bf16_16816(s[1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
          mma_bf16_16816(dp[0], da[ks][0], da[ks][1], da[ks][2], da[ks][3], c0, c1);
          mma_bf16_16816(dp[1], da[ks][0], da[ks][1], da[ks][2], da[ks][3], c2, c3);
        }
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          s[nt][e] += s2[nt][e];
          dp[nt][e] += dp2[nt][e];
        }
    }
    if (pass1) {
      // D partial sums over this lane's columns: rows g and g+8
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        // an invisible key gets P = +0 (its zero-filled V row gives dP = 0)
        Dg = fmaf(ex2_approx(kv[nt][0] ? s[nt][0] * scale_log2 - lse_g : -INFINITY), dp[nt][0], Dg);
        Dg8 = fmaf(ex2_approx(kv[nt][0] ? s[nt][2] * scale_log2 - lse_g8 : -INFINITY), dp[nt][2], Dg8);
        Dg = fmaf(ex2_approx(kv[nt][1] ? s[nt][1] * scale_log2 - lse_g : -INFINITY), dp[nt][1], Dg);
        Dg8 = fmaf(ex2_approx(kv[nt][1] ? s[nt][3] * scale_log2 - lse_g8 : -INFINITY), dp[nt][3], Dg8);
      }
      __syncwarp();
      rotate_slots<C::NST>(pc, pn, pf);
      stage = stage == C::NST - 1 ? 0 : stage + 1;
      continue;
    }
    // P and scale*dS as bf16 hi + lo (rows g: elements 0,1; rows g+8: 2,3)
    uint32_t pp[2][2], pl[2][2], dd[2][2], dl[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      // an invisible key gets 2^-inf = +0 exactly (no branch around the ex2)
      const float p0 = ex2_approx(kv[nt][0] ? s[nt][0] * scale_log2 - lse_g : -INFINITY);
      const float p1 = ex2_approx(kv[nt][1] ? s[nt][1] * scale_log2 - lse_g : -INFINITY);
      const float p2 = ex2_approx(kv[nt][0] ? s[nt][2] * scale_log2 - lse_g8 : -INFINITY);
      const float p3 = ex2_approx(kv[nt][1] ? s[nt][3] * scale_log2 - lse_g8 : -INFINITY);
      const float s0 = scale * p0 * (dp[nt][0] - Dg), s1 = scale * p1 * (dp[nt][1] - Dg);
      const float s2 = scale * p2 * (dp[nt][2] - Dg8), s3 = scale * p3 * (dp[nt][3] - Dg8);
      split_bf16x2_bwd(p0, p1, pp[nt][0], pl[nt][0]);
      split_bf16x2_bwd(p2, p3, pp[nt][1], pl[nt][1]);
      split_bf16x2_bwd(s0, s1, dd[nt][0], dl[nt][0]);
      split_bf16x2_bwd(s2, s3, dd[nt][1], dl[nt][1]);
    }
    // dQ += scale*dS K   (A = dS rows=heads, hi and lo parts; B = K^T via
    // transposed loads).  A needle query's dQ sums large dS K terms, so the
    // bf16 rounding of dS alone (2^-9) is not enough there.
    {
      const int mtx = lane >> 3, r = lane & 7;
      const int key = (mtx & 1) * 8 + r;
#pragma unroll
      for (int j = 0; j < D / 16; ++j) {
        const int ch = 2 * j + (mtx >> 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(ks_base + key * C::ROW_BYTES + ((ch ^ (key & 7)) << 4), b0, b1, b2, b3);
        mma_bf16_16816(dq[2 * j], dd[0][0], dd[0][1], dd[1][0], dd[1][1], b0, b1);
        mma_bf16_16816(dq[2 * j + 1], dd[0][0], dd[0][1], dd[1][0], dd[1][1], b2, b3);
        mma_bf16_16816(dq[2 * j], dl[0][0], dl[0][1], dl[1][0], dl[1][1], b0, b1);
        mma_bf16_16816(dq[2 * j + 1], dl[0][0], dl[0][1], dl[1][0], dl[1][1], b2, b3);
      }
    }
    if constexpr (PASS == 2) {
    // dV[keys] += P^T dO and dK[keys] += (scale*dS)^T Q   (rows = keys)
    // transposed A operands (rows = keys): [0] the hi parts, [1] the lo parts
    uint32_t pt[2][4], dt[2][4];
#pragma unroll
    for (int part = 0; part < 2; ++part) {
      const uint32_t (&ps)[2][2] = part ? pl : pp;
      const uint32_t (&ds)[2][2] = part ? dl : dd;
      pt[part][0] = movmatrix_t(ps[0][0]);
      pt[part][1] = movmatrix_t(ps[1][0]);
      pt[part][2] = movmatrix_t(ps[0][1]);
      pt[part][3] = movmatrix_t(ps[1][1]);
      dt[part][0] = movmatrix_t(ds[0][0]);
      dt[part][1] = movmatrix_t(ds[1][0]);
      dt[part][2] = movmatrix_t(ds[0][1]);
      dt[part][3] = movmatrix_t(ds[1][1]);
    }
    // The step's K/V stage is free now (S, dP and dQ are done).  Each 16-key
    // fp32 tile (dV, then dK) is written into it in fragment order: tile row m
    // (token m >> 2 of slot m & 3) at (m & 3) * POOL_PITCH + (m >> 2) * RED_ROW,
    // so the 8 rows of one fragment write fall in 4 pool blocks whose 32-byte
    // offsets put them in distinct bank groups, and each pool's rows are one
    // contiguous run.  Lanes 0..3 then hand one pool each (its visible rows)
    // to the TMA engine as one bulk fp32 reduction into global memory.
    __syncwarp();
    {
      const int mtx = lane >> 3, r = lane & 7;
      const int hrow = (mtx & 1) * 8 + r;
      const uint32_t tile = ks_base;
      // this lane's fragment rows g and g+8 (tile rows m = g, g+8), columns 2qi..
      const uint32_t frag = tile + (g & 3) * C::POOL_PITCH + (g >> 2) * C::RED_ROW + 8 * qi;
      // the pool this lane reduces (lanes 0..3): slot `lane`
      const uint32_t rslot = (lane & 3) == 0 ? pc[0] : (lane & 3) == 1 ? pc[1] : (lane & 3) == 2 ? pc[2] : pc[3];
      const bool rok = lane < 4 && slot_nrows(rslot) > 0;
      const int64_t rrow_g = 4 * (int64_t)slot_pool(rslot);
      const uint32_t rbytes = (uint32_t)(slot_nrows(rslot) * C::RED_ROW);
      const uint32_t rsrc = tile + (lane & 3) * C::POOL_PITCH;
#pragma unroll
      for (int which = 0; which < 2; ++which) {   // 0: dV = P^T dO, 1: dK = (scale dS)^T Q
        const uint32_t bsrc = which ? qs : dos;
        const uint32_t (&ah)[4] = which ? dt[0] : pt[0];
        const uint32_t (&alo)[4] = which ? dt[1] : pt[1];
        if (which == 1) {
          // the dV tile's reductions must have read it before dK overwrites it
          bulk_wait_read0_if(lane < 4);
          __syncwarp();
        }
        // two 16-column blocks per iteration: four independent accumulators
        // (each takes the hi and then the lo part) before their results are stored
#pragma unroll
        for (int j = 0; j < D / 16; j += 2) {
          uint32_t b[2][4];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int ch = 2 * (j + u) + (mtx >> 1);
            ldsm_x4_t(bsrc + hrow * C::ROW_BYTES + ((ch ^ (hrow & 7)) << 4), b[u][0], b[u][1], b[u][2], b[u][3]);
          }
          float c2[2][2][4];
#pragma unroll
          for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
              for (int e = 0; e < 4; ++e) c2[u][h][e] = 0.f;
              mma_bf16_16816(c2[u][h], ah[0], ah[1], ah[2], ah[3], b[u][2 * h], b[u][2 * h + 1]);
            }
#pragma unroll
          for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int h = 0; h < 2; ++h)
              mma_bf16_16816(c2[u][h], alo[0], alo[1], alo[2], alo[3], b[u][2 * h], b[u][2 * h + 1]);
#pragma unroll
          for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint32_t off = (uint32_t)((2 * (j + u) + h) * 32);   // columns (2(j+u)+h)*8 + 2qi, +1
              st_shared_v2(frag + off, c2[u][h][0], c2[u][h][1]);
              st_shared_v2(frag + 2 * C::RED_ROW + off, c2[u][h][2], c2[u][h][3]);   // row g+8: token +2
            }
        }
        fence_proxy_async_shared();   // the tile's generic-proxy writes before the bulk reads
        __syncwarp();
        float* gdst = which ? dK : dV;
        bulk_red_add_f32_if(gdst + rrow_g * D, rsrc, rbytes, rok);
      }
    }
    }
    __syncwarp();
    rotate_slots<C::NST>(pc, pn, pf);
    stage = stage == C::NST - 1 ? 0 : stage + 1;
  }
  cp_async_wait<0>();
  if (PASS == 2) {
    bulk_wait<0>();   // every bulk reduction of this thread has completed before the CTA exits
  }
  if (bad_idx && lane == 0) record_error(DSA_DEV_ERR_BAD_INDEX);
  if (PASS == 3 && Oacc != nullptr && qi == 0) {
    Dbuf[row0 + g] = Dg;
    Dbuf[row0 + g + 8] = Dg8;
  }
  if (PASS == 1) {
    Dg += __shfl_xor_sync(0xffffffffu, Dg, 1);
    Dg += __shfl_xor_sync(0xffffffffu, Dg, 2);
    Dg8 += __shfl_xor_sync(0xffffffffu, Dg8, 1);
    Dg8 += __shfl_xor_sync(0xffffffffu, Dg8, 2);
    if (qi == 0) {
      Dbuf[row0 + g] = Dg;
      Dbuf[row0 + g + 8] = Dg8;
    }
    return;
  }

  float* q0 = dQ + (row0 + g) * D + 2 * qi;
  float* q8 = q0 + 8 * D;
#pragma unroll
  for (int n = 0; n < D / 8; ++n) {
    *reinterpret_cast<float2*>(q0 + n * 8) = make_float2(dq[n][0], dq[n][1]);
    *reinterpret_cast<float2*>(q8 + n * 8) = make_float2(dq[n][2], dq[n][3]);
  }
}

template <int D, int PASS>
static cudaError_t launch_pass(int64_t L, int Hq, int k, float scale, const __nv_bfloat16* q, const __nv_bfloat16* kk,
                               const __nv_bfloat16* v, const int32_t* idx, const float* lse,
                               const __nv_bfloat16* dout, const float* oacc, float* dbuf, float* dq, float* dk,
                               float* dv, cudaStream_t s) {
  using C = BwdCfg<D, PASS>;
  const float scale_log2 = scale * 1.4426950408889634f;
  const int64_t items = L * (Hq / 16);
  const int64_t blocks = (items + C::WARPS - 1) / C::WARPS;
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_bf16_kernel<D, PASS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM);
  if (e != cudaSuccess) return e;
  attn_bwd_bf16_kernel<D, PASS><<<(unsigned)blocks, 32 * C::WARPS, C::SMEM, s>>>(
      q, kk, v, idx, lse, dout, oacc, dbuf, dq, dk, dv, L, Hq, k, scale, scale_log2);
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd_dq_bf16(int64_t L, int Hq, int d, int k, float scale, const void* q, const void* kk,
                                    const void* v, const int32_t* idx, const float* lse, const void* dout,
                                    const float* oacc, float* dbuf, float* dq, cudaStream_t s) {
  auto qp = static_cast<const __nv_bfloat16*>(q);
  auto kp = static_cast<const __nv_bfloat16*>(kk);
  auto vp = static_cast<const __nv_bfloat16*>(v);
  auto gp = static_cast<const __nv_bfloat16*>(dout);
  cudaError_t e = cudaSuccess;
  if (d == 128) {
    if (oacc == nullptr) e = launch_pass<128, 1>(L, Hq, k, scale, qp, kp, vp, idx, lse, gp, nullptr, dbuf, dq, nullptr, nullptr, s);
    if (e == cudaSuccess) e = launch_pass<128, 3>(L, Hq, k, scale, qp, kp, vp, idx, lse, gp, oacc, dbuf, dq, nullptr, nullptr, s);
    return e;
  }
  if (d == 64) {
    if (oacc == nullptr) e = launch_pass<64, 1>(L, Hq, k, scale, qp, kp, vp, idx, lse, gp, nullptr, dbuf, dq, nullptr, nullptr, s);
    if (e == cudaSuccess) e = launch_pass<64, 3>(L, Hq, k, scale, qp, kp, vp, idx, lse, gp, oacc, dbuf, dq, nullptr, nullptr, s);
    return e;
  }
  return cudaErrorNotSupported;
}

template <int D>
static cudaError_t launch_passes(int64_t L, int Hq, int k, float scale, const __nv_bfloat16* q,
                                 const __nv_bfloat16* kk, const __nv_bfloat16* v, const int32_t* idx,
                                 const float* lse, const __nv_bfloat16* dout, const float* oacc, float* dbuf,
                                 float* dq, float* dk, float* dv, cudaStream_t s) {
  cudaError_t e = cudaSuccess;
  if (oacc == nullptr) e = launch_pass<D, 1>(L, Hq, k, scale, q, kk, v, idx, lse, dout, nullptr, dbuf, dq, dk, dv, s);
  if (e == cudaSuccess) e = launch_pass<D, 2>(L, Hq, k, scale, q, kk, v, idx, lse, dout, oacc, dbuf, dq, dk, dv, s);
  return e;
}

cudaError_t launch_attn_bwd_bf16(int64_t L, int Hq, int d, int k, float scale, const void* q, const void* kk,
                                 const void* v, const int32_t* idx, const float* lse, const void* dout,
                                 const float* oacc, float* dbuf, float* dq, float* dk, float* dv, cudaStream_t s) {
  auto qp = static_cast<const __nv_bfloat16*>(q);
  auto kp = static_cast<const __nv_bfloat16*>(kk);
  auto vp = static_cast<const __nv_bfloat16*>(v);
  auto gp = static_cast<const __nv_bfloat16*>(dout);
  if (d == 128) return launch_passes<128>(L, Hq, k, scale, qp, kp, vp, idx, lse, gp, oacc, dbuf, dq, dk, dv, s);
  if (d == 64) return launch_passes<64>(L, Hq, k, scale, qp, kp, vp, idx, lse, gp, oacc, dbuf, dq, dk, dv, s);
  return cudaErrorNotSupported;
}

}  // namespace dsa
