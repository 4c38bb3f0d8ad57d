// indexer_tc.cu -- lightning-indexer scores on the tcgen05 tensor cores (bf16).
//
// Page "SkyRL extends GLM-5.3-Flash training context to 1 million tokens",
// section "Model and bottleneck" (every query scores one pool per 4 tokens;
// this scoring is the layer's quadratic part) and section "1. DSA truly
// sparse" (scored in query chunks, so the L x L/4 score matrix is never
// materialised at once):
//   s[t,p] = sum_h w[t,h] * max(0, q_I[t,h,:] . kpool[p,:]),   p < elig(t).
//
// Design (one persistent CTA per SM, warp-specialised):
//   * MMA shape M=128 pools x N=32*Hi x K=16.  A 3D TMA box loads the q_I
//     rows of a 32-query block ([L, Hi, di] row-major) head-major into shared
//     memory (row h*32 + t), so one MMA computes D[p, h*32+t] = kpool[p,:] .
//     q_I[t,h,:] for all heads at once (N = 256 at Hi = 8), with fp32
//     accumulators in tensor memory.  An epilogue thread owns one pool (TMEM
//     lane) and holds every head of its queries in its own registers, so
//     ReLU, the head weight and the head sum need no cross-thread exchange;
//     head-major columns put consecutive queries of one head side by side, so
//     the weighted sums of two queries advance in one packed fp32x2 FMA (each
//     query's FMA chain over the heads is unchanged: the same bits).
//   * Two accumulators (2 x Hi x 32 columns) let the MMAs of tile i+1 run
//     while the epilogue drains tile i.
//   * Warp 0 issues TMA loads (128-byte swizzle): the q_I block of a work unit
//     (one box of 32*Hi rows per 64-wide K chunk, double-buffered) and a ring
//     of kpool tiles.  Warp 1 allocates
//     TMEM and issues the MMAs from one thread; warps 2..17 run the epilogue
//     (four warps per TMEM lane quarter, each taking 8 of the 32 queries).
//   * Work unit = (32-query block, up to kSeg pool tiles).  Pool tiles wholly
//     in the future of every query of the block are never visited.  Each
//     epilogue warp stages its 16 queries x 32 pools of a tile in shared
//     memory and writes them with one TMA store (entries past a query's
//     causal prefix inside the diagonal tile are written too; nothing reads
//     them).  Units are handed out round-robin
//     to the persistent CTAs, later (longer) query blocks first.
//   * Every mbarrier wait is bounded; on expiry the CTA records a timeout,
//     unwinds, and still frees its TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "launch.h"

namespace dsa {

template <int HI, int DI>
struct IdxCfg {
  static constexpr int BM = 128;                      // pools per tile (MMA M = TMEM lanes)
  static constexpr int BN = 32;                       // queries per block (MMA N)
  static constexpr int KC = DI / 64;                  // 128-byte K chunks
  static constexpr int A_CHUNK = BM * 128;            // bytes of one K chunk of a kpool tile
  static constexpr int NCOL = BN * HI;                 // MMA N: 32 queries x Hi heads
  static constexpr int B_CHUNK = NCOL * 128;          // bytes of one K chunk of a q_I block
  static constexpr int A_BYTES = KC * A_CHUNK;
  static constexpr int B_BYTES = KC * B_CHUNK;
  static constexpr int NSA = DI == 64 ? 4 : 2;        // kpool tile stages
  static_assert(NSA <= 4, "the barrier slots below hold at most four kpool stages");
  static constexpr int ACC_COLS = HI * BN;            // TMEM columns per accumulator
  static constexpr int TMEM_COLS = 2 * ACC_COLS;      // 256 or 512 (power of two)
  static constexpr int SEG = 16;                      // pool tiles per work unit
  static constexpr int EW = 4;                        // epilogue warps per TMEM lane quarter
  static constexpr int QPW = BN / EW;                  // queries per epilogue warp
  static constexpr int NEPI = 4 * EW;                  // epilogue warps
  static constexpr int THREADS = 64 + 32 * NEPI;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + NSA * A_BYTES;
  static constexpr int OFF_W = OFF_B + 2 * B_BYTES;
  static constexpr int OFF_EMIT = OFF_W + NEPI * QPW * HI * 4;  // private w slice per epilogue warp
  static constexpr int OFF_STG = OFF_EMIT + NEPI * QPW * 32;    // emit mode: per query {tau, cap, list base, length}
  static constexpr int NSTG = DI == 64 ? 2 : 1;            // score staging buffers per epilogue warp
  static constexpr int STG_BYTES = QPW * 32 * 4;           // QPW queries x 32 pools fp32
  static constexpr int OFF_BAR = OFF_STG + NEPI * NSTG * STG_BYTES;
  static constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;  // + alignment slack
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
};

// A 3D TMA tile load signalling `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, uint32_t bar, int32_t x, int32_t y,
                                            int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
      "[%2];\n" ::"r"(dst),
      "l"(tmap), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}
// Eight consecutive TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// One-lane operations of the epilogue as predicated instructions (no branch
// and no reconvergence around them): the lane with `pred` set performs them.
__device__ __forceinline__ void mbar_arrive_if(uint32_t bar, bool pred) {
  asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %1, 0;\n@p mbarrier.arrive.shared::cta.b64 _, [%0];\n}\n" ::"r"(bar),
               "r"((uint32_t)pred)
               : "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait_read_if(bool pred) {
  asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %1, 0;\n@p cp.async.bulk.wait_group.read %0;\n}\n" ::"n"(N),
               "r"((uint32_t)pred)
               : "memory");
}
// TMA tile store of `src` at (x, y), then commit of the bulk group.
__device__ __forceinline__ void tma_store_2d_commit_if(const void* tmap, uint32_t src, int32_t x, int32_t y,
                                                       bool pred) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "@p cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];\n"
      "@p cp.async.bulk.commit_group;\n}\n" ::"l"(tmap),
      "r"(src), "r"(x), "r"(y), "r"((uint32_t)pred)
      : "memory");
}

struct UnitIter {
  int64_t q_begin, q_end;
  int nqb, maxseg;
  int S;                      // column stride
  const int32_t* blist;       // block-list mode when not null
  int nlist;
  int u, stride;
  // current unit
  int64_t t0;
  int tile_begin, tile_end;
  // columns of the block row of query t: the pools p < elig(t) with p % S == 0
  __device__ int64_t ncols(int64_t t) const { return S == 1 ? elig(t) : (elig(t) + S - 1) / S; }
  __device__ int ntiles(int qb, int BN, int BM) const {
    int64_t t_last = q_begin + (int64_t)qb * BN + BN - 1;
    if (t_last >= q_end) t_last = q_end - 1;
    return (int)((ncols(t_last) + BM - 1) / BM);
  }
  template <int BN, int BM, int SEG>
  __device__ bool next() {
    const int nb = blist ? nlist : nqb;
    while (u < nb * maxseg) {
      const int seg = u / nb;
      const int qb = blist ? blist[u % nb] : nqb - 1 - (u % nb);
      u += stride;
      const int nt = ntiles(qb, BN, BM);
      if (seg * SEG >= nt) continue;
      t0 = q_begin + (int64_t)qb * BN;
      tile_begin = seg * SEG;
      tile_end = tile_begin + SEG < nt ? tile_begin + SEG : nt;
      return true;
    }
    return false;
  }
};

template <int HI, int DI, bool EMIT>
__global__ void __launch_bounds__(IdxCfg<HI, DI>::THREADS, 1)
    indexer_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_kp,
                      const __grid_constant__ CUtensorMap tmap_s, const IdxArgs a) {
  using C = IdxCfg<HI, DI>;
  const float* __restrict__ w = a.w;
  float* __restrict__ scores = a.scores;
  const int64_t P = a.P_cols, q_begin = a.q_begin, q_count = a.q_count;
  const int tma_store = a.tma_store;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~static_cast<uintptr_t>(1023));
  const uint32_t sA = smem_u32(smem + C::OFF_A);
  const uint32_t sB = smem_u32(smem + C::OFF_B);
  float* w_s = reinterpret_cast<float*>(smem + C::OFF_W);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  // barrier slots: full_a[4] empty_a[4] full_b[2] empty_b[2] tfull[2] tempty[2]
  const uint32_t bar0 = smem_u32(bars);
  auto full_a = [&](int s) { return bar0 + 8u * s; };
  auto empty_a = [&](int s) { return bar0 + 8u * (4 + s); };
  auto full_b = [&](int s) { return bar0 + 8u * (8 + s); };
  auto empty_b = [&](int s) { return bar0 + 8u * (10 + s); };
  auto tfull = [&](int s) { return bar0 + 8u * (12 + s); };
  auto tempty = [&](int s) { return bar0 + 8u * (14 + s); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 17);
  const uint32_t drain_bar = bar0 + 8u * 18;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t q_end = q_begin + q_count;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NSA; ++s) {
      mbar_init(full_a(s), 1);
      mbar_init(empty_a(s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(full_b(s), 1);
      mbar_init(empty_b(s), 1);
      mbar_init(tfull(s), 1);
      mbar_init(tempty(s), C::NEPI);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap_q);
    prefetch_tmap(&tmap_kp);
    if (tma_store) prefetch_tmap(&tmap_s);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  UnitIter it;
  it.q_begin = q_begin;
  it.q_end = q_end;
  it.nqb = (int)((q_count + C::BN - 1) / C::BN);
  it.S = a.col_stride;
  it.blist = a.blist;
  it.nlist = a.blist ? (int)*a.blist_n : 0;
  {
    const int nt_last = it.ntiles(it.nqb - 1, C::BN, C::BM);
    it.maxseg = (nt_last + C::SEG - 1) / C::SEG;
  }
  it.u = (int)blockIdx.x;
  it.stride = (int)gridDim.x;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t a_iter = 0, b_iter = 0;
      bool ok = true;
      while (ok && it.next<C::BN, C::BM, C::SEG>()) {
        const int bb = b_iter & 1;
        if (!(ok = mbar_wait(empty_b(bb), ((b_iter >> 1) & 1) ^ 1, abort_flag))) break;
        mbar_arrive_expect_tx(full_b(bb), C::B_BYTES);
        for (int c = 0; c < C::KC; ++c)
          tma_load_3d(sB + bb * C::B_BYTES + c * C::B_CHUNK, &tmap_q, full_b(bb), 64 * c, (int32_t)it.t0, 0);
        ++b_iter;
        for (int tile = it.tile_begin; tile < it.tile_end; ++tile) {
          const int s = a_iter % C::NSA;
          if (!(ok = mbar_wait(empty_a(s), ((a_iter / C::NSA) & 1) ^ 1, abort_flag))) break;
          mbar_arrive_expect_tx(full_a(s), C::A_BYTES);
          for (int c = 0; c < C::KC; ++c)
            tma_load_2d(sA + s * C::A_BYTES + c * C::A_CHUNK, &tmap_kp, full_a(s), 64 * c,
                        (int32_t)(tile * C::BM));
          ++a_iter;
        }
      }
      // On abort, wait (bounded) for the loads this thread issued last into
      // each buffer, so no TMA write lands after the CTA has exited.
      if (!ok) {
        for (uint32_t i = (a_iter > (uint32_t)C::NSA ? a_iter - C::NSA : 0); i < a_iter; ++i)
          mbar_wait(full_a(i % C::NSA), (i / C::NSA) & 1, nullptr);
        for (uint32_t i = (b_iter > 2u ? b_iter - 2 : 0); i < b_iter; ++i) mbar_wait(full_b(i & 1), (i >> 1) & 1, nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(C::BM, C::NCOL);
      uint32_t a_iter = 0, b_iter = 0, acc_iter = 0;
      bool ok = true;
      while (ok && it.next<C::BN, C::BM, C::SEG>()) {
        const int bb = b_iter & 1;
        if (!(ok = mbar_wait(full_b(bb), (b_iter >> 1) & 1, abort_flag))) break;
        for (int tile = it.tile_begin; tile < it.tile_end; ++tile) {
          const int s = a_iter % C::NSA;
          const int ab = acc_iter & 1;
          if (!(ok = mbar_wait(full_a(s), (a_iter / C::NSA) & 1, abort_flag))) break;
          if (!(ok = mbar_wait(tempty(ab), ((acc_iter >> 1) & 1) ^ 1, abort_flag))) break;
          tc_fence_after();
          const uint32_t d_base = tmem_base + ab * C::ACC_COLS;
#pragma unroll
          for (int c = 0; c < C::KC; ++c) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t adesc = smem_desc_sw128(sA + s * C::A_BYTES + c * C::A_CHUNK + kk * 32);
              const uint64_t bdesc = smem_desc_sw128(sB + bb * C::B_BYTES + c * C::B_CHUNK + kk * 32);
              tc_mma_f16(d_base, adesc, bdesc, idesc, (c | kk) != 0);
            }
          }
          tc_commit(empty_a(s));
          tc_commit(tfull(ab));
          ++a_iter;
          ++acc_iter;
        }
        if (!ok) break;
        tc_commit(empty_b(bb));
        ++b_iter;
      }
      // Drain: wait (bounded) until every MMA this thread issued has finished,
      // so tensor memory is never freed under a running MMA.
      tc_commit(drain_bar);
      mbar_wait(drain_bar, 0, nullptr);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int ew = warp - 2;                 // 0 .. NEPI-1
    const int quarter = warp & 3;            // TMEM lanes this warp may access
    const int qg = ew >> 2;                  // which QPW of the 32 queries
    const int lane_base = quarter * 32;
    uint32_t acc_iter = 0;
    bool ok = true;
    float* w_mine = w_s + ew * C::QPW * HI;  // this warp's HI heads x QPW queries (head-major)
    // emit mode, per query of this warp (8 words): [0] tau, [4] sub-list
    // capacity, [5..6] sub-list base (64-bit), [7] sub-list length so far
    // (words 4..7 are read as one 16-byte vector).  The lengths live in
    // shared memory rather than registers: they persist across tiles, and
    // registers are what the epilogue's scoring math is short of.
    uint32_t* emit_mine = reinterpret_cast<uint32_t*>(smem + C::OFF_EMIT) + ew * C::QPW * 8;
    const uint32_t emit_sa = smem_u32(emit_mine);
    const uint32_t w_mine_s = smem_u32(w_mine);
    uint32_t stg_iter = 0;
    static_assert(C::QPW == 8, "a warp's queries of one head are one 8-column TMEM load");
    while (ok && it.next<C::BN, C::BM, C::SEG>()) {
      __syncwarp();
      for (int i = lane; i < C::QPW * HI; i += 32) {
        const int64_t t = it.t0 + qg * C::QPW + i % C::QPW;
        w_mine[i] = t < q_end ? __ldg(w + t * HI + i / C::QPW) : 0.f;
      }
      // emit mode: the threshold and this warp's sub-list of each of its
      // queries for this unit (segment seg, lane quarter `quarter`); +inf and
      // capacity 0 past the range
      if constexpr (EMIT) {
        if (lane < C::QPW) {
          const int64_t t = it.t0 + qg * C::QPW + lane;
          const int64_t seg = it.tile_begin / C::SEG;
          float th = INFINITY;
          uint32_t cap = 0u;
          int64_t base = 0;
          if (t < q_end) {
            th = __ldg(a.tau + (t - q_begin));
            const int64_t e = elig(t);
            const int64_t nseg = e > kSegPools ? (e + kSegPools - 1) / kSegPools : 1;
            cap = (uint32_t)(a.cand_stride / (4 * nseg));
            base = (t - q_begin) * a.cand_stride + (seg * 4 + quarter) * (int64_t)cap;
          }
          emit_mine[8 * lane] = __float_as_uint(th);
          emit_mine[8 * lane + 4] = cap;
          emit_mine[8 * lane + 5] = (uint32_t)base;
          emit_mine[8 * lane + 6] = (uint32_t)(base >> 32);
          emit_mine[8 * lane + 7] = 0u;
        }
      }
      __syncwarp();
      for (int tile = it.tile_begin; tile < it.tile_end; ++tile) {
        const int ab = acc_iter & 1;
        if (!(ok = mbar_wait(tfull(ab), (acc_iter >> 1) & 1, abort_flag))) break;
        tc_fence_after();
        // this thread: pool (lane_base + lane), queries qg*QPW .. +QPW-1 of head
        // h in columns h*BN + qg*QPW .. +QPW-1 -- all loaded before one wait
        const uint32_t taddr = tmem_base + ((uint32_t)lane_base << 16) + ab * C::ACC_COLS + qg * C::QPW;
        float v[HI][C::QPW];
#pragma unroll
        for (int h = 0; h < HI; ++h) tmem_ld8(taddr + h * C::BN, v[h]);
        tmem_ld_wait();
        // the accumulator is in registers: hand it back to the MMA warp
        tc_fence_before();
        __syncwarp();
        mbar_arrive_if(tempty(ab), lane == 0);
        const int64_t p = (int64_t)tile * C::BM + lane_base + lane;
        // acc[j] = fma(relu(s_h), w_h, acc[j]) over heads h = 0..Hi-1 in order,
        // two queries per packed FMA
        float2 acc2[C::QPW / 2];
#pragma unroll
        for (int jp = 0; jp < C::QPW / 2; ++jp) acc2[jp] = make_float2(0.f, 0.f);
#pragma unroll
        for (int h = 0; h < HI; ++h) {
          // weights of head h for the warp's queries (broadcast, explicit shared loads)
          const float4 wa = ld_shared_v4(w_mine_s + 4 * (h * C::QPW));
          const float4 wb = ld_shared_v4(w_mine_s + 4 * (h * C::QPW + 4));
          const float2 w2[4] = {make_float2(wa.x, wa.y), make_float2(wa.z, wa.w), make_float2(wb.x, wb.y),
                                make_float2(wb.z, wb.w)};
#pragma unroll
          for (int jp = 0; jp < C::QPW / 2; ++jp)
            acc2[jp] = __ffma2_rn(make_float2(fmaxf(v[h][2 * jp], 0.f), fmaxf(v[h][2 * jp + 1], 0.f)), w2[jp],
                                  acc2[jp]);
        }
        float acc[C::QPW];
#pragma unroll
        for (int jp = 0; jp < C::QPW / 2; ++jp) {
          acc[2 * jp] = acc2[jp].x;
          acc[2 * jp + 1] = acc2[jp].y;
        }
        if constexpr (EMIT) {
          // candidates: every eligible score >= the row's threshold goes to
          // this warp's sub-list of the row (no atomics: the warp alone fills
          // it, with a warp-uniform running length); entries past the
          // capacity are counted but not stored (the row then takes the
          // score-block path)
          const uint32_t below = (1u << lane) - 1u;
          const int pe = (int)p;
#pragma unroll
          const int tq0 = (int)(it.t0 + qg * C::QPW);   // this warp's first query
          for (int j = 0; j < C::QPW; ++j) {
            uint32_t th;
            asm volatile("ld.shared.u32 %0, [%1];\n" : "=r"(th) : "r"(emit_sa + 32 * j));
            const bool take = pe < ((tq0 + j + 1) >> 2) && acc[j] >= __uint_as_float(th);
            // the ballot also orders this lane-0 read-modify-write of the
            // length after every lane's earlier reads of it
            const uint32_t m = __ballot_sync(0xffffffffu, take);
            if (m != 0u) {   // warp-uniform
              uint32_t cap, blo, bhi, len;
              asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];\n"
                           : "=r"(cap), "=r"(blo), "=r"(bhi), "=r"(len)
                           : "r"(emit_sa + 32 * j + 16));
              const uint32_t pos = len + (uint32_t)__popc(m & below);
              if (take && pos < cap) {
                const int64_t base = (int64_t)(((uint64_t)bhi << 32) | blo);
                a.cand[base + pos] = make_uint2(__float_as_uint(acc[j]), (uint32_t)pe);
              }
              __syncwarp();
              if (lane == 0)
                asm volatile("st.shared.u32 [%0], %1;\n" ::"r"(emit_sa + 32 * j + 28), "r"(len + (uint32_t)__popc(m)));
            }
          }
          __syncwarp();
        } else if (tma_store) {
          // stage this warp's QPW queries x 32 pools and store them with one
          // TMA box; entries past a query's causal prefix inside the box are
          // written too (the top-k never reads them)
          const int sb = stg_iter % C::NSTG;
          const uint32_t stg = smem_u32(smem + C::OFF_STG) + (ew * C::NSTG + sb) * C::STG_BYTES;
          bulk_wait_read_if<C::NSTG - 1>(lane == 0 && stg_iter >= C::NSTG);
          __syncwarp();
#pragma unroll
          for (int j = 0; j < C::QPW; ++j)
            asm volatile("st.shared.f32 [%0], %1;\n" ::"r"(stg + (j * 32 + lane) * 4), "f"(acc[j]) : "memory");
          fence_proxy_async_shared();
          __syncwarp();
          tma_store_2d_commit_if(&tmap_s, stg, (int32_t)(tile * C::BM + lane_base),
                                 (int32_t)(it.t0 - q_begin + qg * C::QPW), lane == 0);
          ++stg_iter;
        } else {
#pragma unroll
          for (int j = 0; j < C::QPW; ++j) {
            const int64_t t = it.t0 + qg * C::QPW + j;
            // streaming store: the score block is read once, by the top-k
            if (t < q_end && p < it.ncols(t)) __stcs(scores + (t - q_begin) * P + p, acc[j]);
          }
        }
        ++acc_iter;
      }
      if constexpr (EMIT) {
        // the unit's sub-list lengths (lane j: query j)
        __syncwarp();
        const uint32_t mine = lane < C::QPW ? emit_mine[8 * lane + 7] : 0u;
        const int64_t t = it.t0 + qg * C::QPW + lane;
        if (ok && lane < C::QPW && t < q_end)
          a.cntq[((t - q_begin) * a.nseg_max + it.tile_begin / C::SEG) * 4 + quarter] = mine;
      }
    }
    if (!ok) *abort_flag = 1;
    // every score store of this warp has finished before the CTA exits
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// --------------------------------------------------------------------- host
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

template <int HI, int DI>
static cudaError_t launch_tc(int64_t L, const void* q_idx, const void* kpool, IdxArgs a, bool emit,
                             cudaStream_t s) {
  using C = IdxCfg<HI, DI>;
  const int64_t P = L / 4;
  const int S = a.col_stride;
  const int64_t P_src = (P + S - 1) / S;   // kpool rows the launch reads (every S-th pool)
  auto enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap tq, tk;
  {
    // q_I [L, Hi, di] seen as (di, t, h): a box of 32 queries x Hi heads lands
    // head-major in shared memory (row h*32 + t)
    const cuuint64_t dims[3] = {(cuuint64_t)DI, (cuuint64_t)L, (cuuint64_t)HI};
    const cuuint64_t strides[2] = {(cuuint64_t)HI * DI * 2, (cuuint64_t)DI * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)C::BN, (cuuint32_t)HI};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (enc(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q_idx), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    // row j of this view is pool j*S
    const cuuint64_t dims[2] = {(cuuint64_t)DI, (cuuint64_t)P_src};
    const cuuint64_t strides[1] = {(cuuint64_t)DI * 2 * (cuuint64_t)S};
    const cuuint32_t box[2] = {64, (cuuint32_t)C::BM};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(kpool), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  // Score tiles go out through TMA when the row pitch allows it (P_cols*4 a
  // multiple of 16 bytes); otherwise with plain stores.
  CUtensorMap ts = tk;  // unused unless a TMA store map is made below
  a.tma_store = 0;
  if (!emit && (a.P_cols % 4) == 0) {
    const cuuint64_t dims[2] = {(cuuint64_t)a.P_cols, (cuuint64_t)a.q_count};
    const cuuint64_t strides[1] = {(cuuint64_t)a.P_cols * 4};
    const cuuint32_t box[2] = {32, (cuuint32_t)C::QPW};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&ts, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, a.scores, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    a.tma_store = 1;
  }
  auto kern = emit ? indexer_tc_kernel<HI, DI, true> : indexer_tc_kernel<HI, DI, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int64_t nqb = (a.q_count + C::BN - 1) / C::BN;
  const int64_t t_last = a.q_begin + a.q_count - 1;
  const int64_t nt_last = ((((t_last + 1) >> 2) + S - 1) / S + C::BM - 1) / C::BM;
  const int64_t units = nqb * ((nt_last + C::SEG - 1) / C::SEG);
  if (units == 0) return cudaSuccess;
  int64_t grid = device_sm_count();
  if (a.blist == nullptr && grid > units) grid = units;   // a block list's length is known on the device only
  kern<<<(unsigned)grid, C::THREADS, C::SMEM_BYTES, s>>>(tq, tk, ts, a);
  return cudaGetLastError();
}

cudaError_t launch_indexer_tc_bf16_ex(int64_t L, int Hi, int di, const void* q_idx, const void* kpool,
                                      const IdxArgs& a, bool emit, cudaStream_t s) {
  if (Hi == 8 && di == 64) return launch_tc<8, 64>(L, q_idx, kpool, a, emit, s);
  if (Hi == 8 && di == 128) return launch_tc<8, 128>(L, q_idx, kpool, a, emit, s);
  if (Hi == 4 && di == 64) return launch_tc<4, 64>(L, q_idx, kpool, a, emit, s);
  if (Hi == 4 && di == 128) return launch_tc<4, 128>(L, q_idx, kpool, a, emit, s);
  return cudaErrorNotSupported;
}

cudaError_t launch_indexer_tc_bf16(int64_t L, int Hi, int di, const void* q_idx, const void* kpool,
                                   const float* w, int64_t q_begin, int64_t q_count, float* scores,
                                   cudaStream_t s) {
  IdxArgs a{};
  a.w = w;
  a.scores = scores;
  a.P_cols = L / 4;
  a.q_begin = q_begin;
  a.q_count = q_count;
  a.col_stride = 1;
  return launch_indexer_tc_bf16_ex(L, Hi, di, q_idx, kpool, a, false, s);
}

}  // namespace dsa
