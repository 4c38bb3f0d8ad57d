// attn_fwd_tc.cu -- sparse attention forward on the tcgen05 tensor cores
// (bf16, head dim 128, 16 or 32 query heads).
//
// Page "SkyRL extends GLM-5.3-Flash training context to 1 million tokens",
// section "Model and bottleneck" (about 2048 keys read per query) and section
// "1. DSA truly sparse" (a truly sparse kernel; 2051 = 4*512+3 keys).  Same
// definition as attn_fwd.cu: the keys of query t are the tokens of the pools
// in idx[t,:] (entries < 0 skipped) plus its own partial pool
// 4*floor(t/4) .. t when t%4 != 3; O = softmax(scale Q K^T) V, LSE in natural
// log.
//
// Design: one persistent CTA per SM walks queries (late first); all Hq heads
// of a query share its keys, so the heads are the N side of the MMAs and the
// keys the M side:
//   * a key tile is 32 pool slots = 128 keys.  Producer warps gather it with
//     16-byte cp.async copies (lanes along a pool's contiguous 1 KB of K or
//     V rows) straight into the canonical K-major layout with the 128-byte
//     swizzle; an empty or out-of-range slot is zero-filled.  The copies
//     arrive on the stage's barrier by themselves when they land, and the MMA
//     thread fences them into the async proxy after its wait.  (TMA box
//     loads of the same 512-byte pieces were tried first: one producer warp
//     issued them at about 50 cycles per box, five times too slow.)  K and V
//     have separate stage rings: a K stage is free once S is formed, a V
//     stage only after P.V.  Q, one contiguous box per query, comes by TMA.
//   * one thread issues S^T = K_tile . Q^T (M = 128 keys, N = Hq, fp32 in
//     tensor memory) and O^T += V_tile^T . P (M = 128 head dims, N = Hq; V
//     read as an MN-major operand, P from shared memory).  O^T stays in
//     tensor memory for the whole query.
//   * four softmax warps own one key each per TMEM lane: they read S^T,
//     apply the causal/validity mask, and form P = 2^(s*scale*log2e - base)
//     with a per-head base that moves lazily (only when a tile's score
//     exceeds it by more than 2^8, decided CTA-wide with one barrier
//     reduction per tile); moving it rescales the running sums and O^T in
//     tensor memory.  P is written as bf16 (with an o_acc buffer, as bf16
//     hi + lo: two MMAs, P carried to about 2^-17).  Row sums stay in
//     per-thread fp32 partials until the end of the query.
//   * the partial pool's (at most 3) keys are scored on the CUDA cores at the
//     start of the query (they seed the base) and added to O and the row sums
//     in fp32 at the end.
// Every wait is bounded; on expiry the CTA records a timeout and unwinds,
// waiting for its own copies and MMAs before it frees tensor memory.
//
// Measured against the warp-level kernel (attn_fwd.cu) at L = 131072, Hq = 16,
// k = 512: 33.3 ms against 10.2 ms with o_acc, 28.1 against 8.2 without.  A
// clock64 breakdown shows the gather keeping up and the MMA thread busy
// issuing: a one-thread loop of back-to-back M = 128, K = 16 bf16 MMAs takes
// 189 cycles per MMA whatever N is (16 to 256) and however many independent
// accumulators it cycles through, so an N = 16 MMA does 1/16 of the work of
// an N = 256 one in the same time.  A tile needs 16 to 24 of them (8 more
// with o_acc cost 5.2 ms in this kernel).  Only the Hq heads of one query
// share its keys, so N cannot grow; the warp-level kernel stays the default
// and this one is the alternative route.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "launch.h"

namespace dsa {

template <int HQ>
struct FtcCfg {
  static constexpr int D = 128;
  static constexpr int TK = 128;                  // keys per tile (MMA M, TMEM lanes)
  static constexpr int SLOTS = TK / 4;            // pool slots per tile (one producer lane each)
  static constexpr int CB = TK * 128;             // one 64-column block of a K or V tile
  static constexpr int KV_TILE = 2 * CB;          // 32 KB
  static constexpr int NKS = 3;                   // K stages
  static constexpr int NVS = 3;                   // V stages
  static constexpr int NPB = HQ == 16 ? 2 : 1;    // P buffers
  static constexpr int Q_CB = HQ * 128;           // one 64-column block of the Q tile
  static constexpr int Q_TILE = 2 * Q_CB;
  static constexpr int P_CB = HQ * 128;           // 64 keys of P^T (rows = heads)
  static constexpr int P_TERM = 2 * P_CB;         // P^T of one tile, one bf16 term
  static constexpr int P_BUF = 2 * P_TERM;        // hi + lo
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + NKS * KV_TILE;
  static constexpr int OFF_Q = OFF_V + NVS * KV_TILE;
  static constexpr int OFF_P = OFF_Q + 2 * Q_TILE;
  static constexpr int OFF_PART = OFF_P + NPB * P_BUF;   // [4][HQ] fp32: partial-pool scores
  static constexpr int OFF_RED = OFF_PART + 4 * HQ * 4;  // [4][HQ] fp32: tile maxima per warp
  static constexpr int OFF_SUM = OFF_RED + 4 * HQ * 4;   // [4][HQ] fp32: row sums per warp
  static constexpr int OFF_BAR = OFF_SUM + 4 * HQ * 4;
  static constexpr int NBAR = 2 * NKS + 2 * NVS + 16 + 1;   // rings, 8 pairs, drain
  static constexpr int SMEM_BYTES = OFF_BAR + NBAR * 8 + 16 + 1024;   // + alignment slack
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
  static constexpr int TMEM_COLS = 4 * HQ;        // S^T x2, O^T x2
  // producer warps: four at 16 heads; two at 32 (seven warps leave the
  // softmax threads 255 registers for their 3 x 32 per-head values)
  static constexpr int NPW = HQ == 16 ? 4 : 2;
  static constexpr int SPW = SLOTS / NPW;         // pool slots per producer warp and tile
  static constexpr int THREADS = 32 * (5 + NPW);  // softmax warps 0-3, MMA warp 4, producers 5..
  static constexpr int TPH = 128 / HQ;            // partial pool: threads per head
  static constexpr int EPT = D / TPH;             // partial pool: elements per thread
};

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, uint32_t bar, int32_t x, int32_t y,
                                            int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
      "[%2];\n" ::"r"(dst),
      "l"(tmap), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}
// Arrive on the mbarrier once every cp.async this thread issued so far has
// landed (the barrier's expected count includes this arrival).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void softmax_bar() { asm volatile("bar.sync 1, 128;\n" ::: "memory"); }
// barrier over the 128 softmax threads that also ORs a predicate across them
__device__ __forceinline__ bool softmax_bar_any(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\nbarrier.cta.red.or.pred q, 1, 128, p;\nselp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
      "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
      "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;\n" ::"r"(addr), "h"(v) : "memory");
}
// Shared-memory descriptor of an MN-major operand with the 128-byte swizzle:
// 64 MN-elements (128 bytes) per row, one row per K index, 8-row groups
// `sbo` bytes apart along K and 64-element MN blocks `lbo` bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sw128_mn(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t desc = 0;
  desc |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  desc |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  desc |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  desc |= (uint64_t)1u << 46;
  desc |= (uint64_t)2u << 61;
  return desc;
}
// TMEM load of n consecutive fp32 columns (n = 16 or 32) of this thread's lane.
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[N]) {
#pragma unroll
  for (int c = 0; c < N / 16; ++c) tmem_ld16(taddr + 16 * c, *reinterpret_cast<float(*)[16]>(&v[16 * c]));
}
template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const float (&v)[N]) {
#pragma unroll
  for (int c = 0; c < N / 16; ++c) tmem_st16(taddr + 16 * c, *reinterpret_cast<const float(*)[16]>(&v[16 * c]));
}

struct FtcArgs {
  const __nv_bfloat16* Q;
  const __nv_bfloat16* K;
  const __nv_bfloat16* V;
  const int32_t* idx;
  __nv_bfloat16* O;
  float* LSE;
  float* Oacc;
  int64_t L;
  int k;
  float scale_log2;
};

template <int HQ, bool ACC>
__global__ void __launch_bounds__(FtcCfg<HQ>::THREADS, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const FtcArgs a) {
  using C = FtcCfg<HQ>;
  constexpr float kLazy = 8.f;   // the base lags the running max by at most this (log2 units)
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~static_cast<uintptr_t>(1023));
  const uint32_t sK = smem_u32(smem + C::OFF_K), sV = smem_u32(smem + C::OFF_V);
  const uint32_t sQ = smem_u32(smem + C::OFF_Q), sP = smem_u32(smem + C::OFF_P);
  float* part = reinterpret_cast<float*>(smem + C::OFF_PART);
  float* red = reinterpret_cast<float*>(smem + C::OFF_RED);
  float* rsum = reinterpret_cast<float*>(smem + C::OFF_SUM);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  const uint32_t bar0 = smem_u32(bars);
  // barrier slots: kfull kfree [NKS], vfull vfree [NVS], then qfull qfree sfull
  // sfree pfull pvdone ofull ofree [2 each], then the drain barrier
  auto kfull = [&](int s) { return bar0 + 8u * s; };
  auto kfree = [&](int s) { return bar0 + 8u * (C::NKS + s); };
  auto vfull = [&](int s) { return bar0 + 8u * (2 * C::NKS + s); };
  auto vfree = [&](int s) { return bar0 + 8u * (2 * C::NKS + C::NVS + s); };
  constexpr int B2 = 2 * C::NKS + 2 * C::NVS;
  auto qfull = [&](int s) { return bar0 + 8u * (B2 + s); };
  auto qfree = [&](int s) { return bar0 + 8u * (B2 + 2 + s); };
  auto sfull = [&](int s) { return bar0 + 8u * (B2 + 4 + s); };
  auto sfree = [&](int s) { return bar0 + 8u * (B2 + 6 + s); };
  auto pfull = [&](int s) { return bar0 + 8u * (B2 + 8 + s); };
  auto pvdone = [&](int s) { return bar0 + 8u * (B2 + 10 + s); };
  auto ofull = [&](int s) { return bar0 + 8u * (B2 + 12 + s); };
  auto ofree = [&](int s) { return bar0 + 8u * (B2 + 14 + s); };
  const uint32_t drain_bar = bar0 + 8u * (B2 + 16);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + C::NBAR) + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t L = a.L;
  const int k = a.k;
  const int T = (k + C::SLOTS - 1) / C::SLOTS;   // key tiles per query

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NKS; ++s) {
      mbar_init(kfull(s), 32 * C::NPW);   // every producer thread
      mbar_init(kfree(s), 1);
    }
    for (int s = 0; s < C::NVS; ++s) {
      mbar_init(vfull(s), 32 * C::NPW);
      mbar_init(vfree(s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(qfull(s), 1);
      mbar_init(qfree(s), 1);
      mbar_init(sfull(s), 1);
      mbar_init(sfree(s), 4);
      mbar_init(pfull(s), 4);
      mbar_init(pvdone(s), 1);
      mbar_init(ofull(s), 1);
      mbar_init(ofree(s), 4);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap_q);
  }
  if (warp == 4) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp >= 5) {
    // ---------------------------------------------------- cp.async producers
    // Producer warp pw gathers pool slots SPW*pw .. SPW*pw+SPW-1 of every
    // tile: per slot two 16-byte copies per lane for K (rows 2u, 2u+1, lanes
    // along the 256-byte rows) and two for V, written straight into the
    // swizzled canonical layout.  V of tile g goes out after K of tile g+1 (V
    // is needed one softmax later).  Each thread's copies of a stage arrive on
    // the stage's full barrier by themselves when they land
    // (cp.async.mbarrier.arrive.noinc), so a producer only ever waits for a
    // free stage; the MMA thread fences them into the async proxy.
    const int pw = warp - 5;
    const int rlo = lane >> 4, j16 = lane & 15, cblk = j16 >> 3, jj = j16 & 7;
    const uint32_t src_off = (uint32_t)(rlo * 256 + j16 * 16);
    uint32_t dst_off[2][2];   // [slot parity][copy]
#pragma unroll
    for (int par = 0; par < 2; ++par)
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int r = 2 * u + rlo;
        dst_off[par][u] = (uint32_t)(cblk * C::CB + r * 128 + ((jj ^ (4 * par + r)) << 4));
      }
    const char* Kb = reinterpret_cast<const char*>(a.K);
    const char* Vb = reinterpret_cast<const char*>(a.V);
    uint32_t g = 0;   // tiles issued
    bool ok = true, bad = false;
    // copies of one tensor's SPW slots of a tile into `stage`; `mine` is the
    // pool of slot SPW*pw + lane (lanes 0..SPW-1), -1 for none
    auto gather = [&](const char* base, uint32_t stage, int mine) {
#pragma unroll
      for (int i = 0; i < C::SPW; ++i) {
        const int pool = __shfl_sync(0xffffffffu, mine, i);
        const uint32_t bytes = pool >= 0 ? 16u : 0u;
        const char* src = base + (int64_t)(pool >= 0 ? pool : 0) * 1024 + src_off;
        const uint32_t dst = stage + (uint32_t)(C::SPW * pw + i) * 512u;
#pragma unroll
        for (int u = 0; u < 2; ++u) cp_async16(dst + dst_off[i & 1][u], src + u * 512, bytes);
      }
    };
    auto wait_free = [&](uint32_t bar, uint32_t parity) -> bool {
      bool w = true;
      if (lane == 0) w = mbar_wait(bar, parity, abort_flag);
      return __shfl_sync(0xffffffffu, (int)w, 0) != 0;
    };
    int pool_prev = -1;   // this lane's slot of the previous tile (for its V)
    for (int64_t i = blockIdx.x; ok && i < L; i += gridDim.x) {
      const int64_t t = L - 1 - i;
      const int64_t el = elig(t);
      const int32_t* irow = a.idx + t * (int64_t)k;
      auto pool_of = [&](int j) -> int {   // this lane's slot of tile j of this query
        const int slot = j * C::SLOTS + C::SPW * pw + (lane & (C::SPW - 1));
        const int p = slot < k ? __ldg(irow + slot) : -1;
        bad |= p >= el;
        return (p >= 0 && p < el) ? p : -1;
      };
      int pool_next = pool_of(0);
      for (int j = 0; j < T; ++j) {
        const int pool_cur = pool_next;
        if (j + 1 < T) pool_next = pool_of(j + 1);   // a tile ahead of its use
        const int ks = g % C::NKS;
        if (!(ok = wait_free(kfree(ks), ((g / C::NKS) & 1) ^ 1))) break;
        gather(Kb, sK + ks * C::KV_TILE, pool_cur);
        cp_async_arrive_noinc(kfull(ks));
        if (g >= 1) {
          const int vs = (g - 1) % C::NVS;
          if (!(ok = wait_free(vfree(vs), (((g - 1) / C::NVS) & 1) ^ 1))) break;
          gather(Vb, sV + vs * C::KV_TILE, pool_prev);
          cp_async_arrive_noinc(vfull(vs));
        }
        pool_prev = pool_cur;
        ++g;
      }
    }
    if (ok && g >= 1) {
      const int vs = (g - 1) % C::NVS;
      if ((ok = wait_free(vfree(vs), (((g - 1) / C::NVS) & 1) ^ 1))) {
        gather(Vb, sV + vs * C::KV_TILE, pool_prev);
        cp_async_arrive_noinc(vfull(vs));
      }
    }
    // every copy of this thread has landed before the CTA can exit
    cp_async_commit();
    cp_async_wait<0>();
    if (__any_sync(0xffffffffu, bad) && lane == 0) record_error(DSA_DEV_ERR_BAD_INDEX);
    if (!ok) *abort_flag = 1;
  } else if (warp == 4) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(C::TK, HQ);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(C::D, HQ) | (1u << 15);   // A (V^T) MN-major
      uint32_t gk = 0, gp = 0, nq = 0, nqi = 0;   // nqi: Q tiles issued
      bool ok = true;
      // Q tile of the CTA's n-th query (row t) into buffer n & 1, once the
      // S MMAs of query n-2 have finished reading that buffer
      auto load_q = [&](uint32_t n, int64_t t) -> bool {
        if (!mbar_wait(qfree(n & 1), ((n >> 1) & 1) ^ 1, abort_flag)) return false;
        mbar_arrive_expect_tx(qfull(n & 1), C::Q_TILE);
        tma_load_3d(sQ + (n & 1) * C::Q_TILE, &tmap_q, qfull(n & 1), 0, 0, (int32_t)t);
        tma_load_3d(sQ + (n & 1) * C::Q_TILE + C::Q_CB, &tmap_q, qfull(n & 1), 64, 0, (int32_t)t);
        ++nqi;
        return true;
      };
      if (blockIdx.x < L) ok = load_q(0, L - 1 - (int64_t)blockIdx.x);
      // O^T += V^T P for tile gp (the first tile of a query starts the accumulator)
      auto pv = [&](bool first) -> bool {
        const int vs = gp % C::NVS, pb = gp & 1, ob = nq & 1;   // pb: pfull/pvdone barrier
        if (!mbar_wait(vfull(vs), (gp / C::NVS) & 1, abort_flag)) return false;
        if (!mbar_wait(pfull(pb), (gp >> 1) & 1, abort_flag)) return false;
        if (first && !mbar_wait(ofree(ob), ((nq >> 1) & 1) ^ 1, abort_flag)) return false;
        fence_proxy_async_shared();   // the producers' copies, seen through the barrier
        tc_fence_after();
        const uint32_t d_o = tmem_base + 2 * HQ + ob * HQ;
        const uint32_t vt = sV + vs * C::KV_TILE, pt = sP + (gp % C::NPB) * C::P_BUF;
#pragma unroll
        for (int kk = 0; kk < C::TK / 16; ++kk) {
          const uint64_t ad = smem_desc_sw128_mn(vt + kk * 16 * 128, C::CB, 1024);
          const uint64_t bd = smem_desc_sw128(pt + (kk >> 2) * C::P_CB + (kk & 3) * 32);
          tc_mma_f16(d_o, ad, bd, idesc_pv, (first && kk == 0) ? 0u : 1u);
        }
        if constexpr (ACC) {
#pragma unroll
          for (int kk = 0; kk < C::TK / 16; ++kk) {
            const uint64_t ad = smem_desc_sw128_mn(vt + kk * 16 * 128, C::CB, 1024);
            const uint64_t bd = smem_desc_sw128(pt + C::P_TERM + (kk >> 2) * C::P_CB + (kk & 3) * 32);
            tc_mma_f16(d_o, ad, bd, idesc_pv, 1u);
          }
        }
        tc_commit(vfree(vs));
        tc_commit(pvdone(pb));
        ++gp;
        return true;
      };
      for (int64_t i = blockIdx.x; ok && i < L; i += gridDim.x, ++nq) {
        const int qb = nq & 1;
        if (!(ok = mbar_wait(qfull(qb), (nq >> 1) & 1, abort_flag))) break;
        for (int j = 0; j < T; ++j) {
          const int s = gk % C::NKS, sb = gk & 1;
          if (!(ok = mbar_wait(kfull(s), (gk / C::NKS) & 1, abort_flag))) break;
          if (!(ok = mbar_wait(sfree(sb), ((gk >> 1) & 1) ^ 1, abort_flag))) break;
          fence_proxy_async_shared();   // the producers' copies, seen through the barrier
          tc_fence_after();
          const uint32_t kt = sK + s * C::KV_TILE, qt = sQ + qb * C::Q_TILE;
#pragma unroll
          for (int kk = 0; kk < C::D / 16; ++kk) {
            const uint64_t ad = smem_desc_sw128(kt + (kk >> 2) * C::CB + (kk & 3) * 32);
            const uint64_t bd = smem_desc_sw128(qt + (kk >> 2) * C::Q_CB + (kk & 3) * 32);
            tc_mma_f16(tmem_base + sb * HQ, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
          }
          tc_commit(kfree(s));
          tc_commit(sfull(sb));
          ++gk;
          if (j == T - 1) {
            tc_commit(qfree(qb));
            const int64_t inext = i + gridDim.x;
            if (inext < L && !(ok = load_q(nq + 1, L - 1 - inext))) break;
          }
          if (j >= 1 && !(ok = pv(j == 1))) break;
        }
        if (!ok) break;
        if (!(ok = pv(T == 1))) break;
        tc_commit(ofull(nq & 1));
      }
      if (!ok) {
        *abort_flag = 1;
        // no TMA write may land after the CTA has exited
        for (uint32_t n = (nqi > 2u ? nqi - 2 : 0); n < nqi; ++n) mbar_wait(qfull(n & 1), (n >> 1) & 1, nullptr);
      }
      // Drain: every MMA this thread issued has finished before TMEM is freed.
      tc_commit(drain_bar);
      mbar_wait(drain_bar, 0, nullptr);
    }
  } else {
    // ---------------------------------------------------------- softmax warps
    // The four warps meet at named barriers, so none of them may leave the
    // loop alone: a failed (bounded) wait only clears `ok`, the warp carries
    // on with whatever data it has, and the decision to stop is taken by all
    // of them together at the next barrier reduction.
    const int key = warp * 32 + lane;            // this thread's key of a tile / head dim of O^T
    const uint32_t lane_addr = (uint32_t)(warp * 32) << 16;
    const int tid = threadIdx.x;                  // 0 .. 127
    uint32_t gk = 0, nq = 0;
    bool ok = true;
    const float sl2 = a.scale_log2;
    for (int64_t i = blockIdx.x; i < L; i += gridDim.x, ++nq) {
      // every thread is done with the previous query's part[] and rsum[]
      if (softmax_bar_any(!ok || *abort_flag != 0)) break;
      const int64_t t = L - 1 - i;
      const int64_t el = elig(t);
      const int npart = (t & 3) != 3 ? (int)(t & 3) + 1 : 0;
      const int64_t prow = 4 * (t >> 2);          // first token of the partial pool
      const int32_t* irow = a.idx + t * (int64_t)k;
      // partial-pool scores (log2 units): head h = tid / TPH, elements
      // (tid % TPH) * EPT .. +EPT-1, reduced over the TPH lanes of the head
      if (npart > 0) {
        const int h = tid / C::TPH, sub = tid % C::TPH;
        const uint4* q4 = reinterpret_cast<const uint4*>(a.Q + (t * HQ + h) * C::D + sub * C::EPT);
        uint4 qv[C::EPT / 8];
#pragma unroll
        for (int c = 0; c < C::EPT / 8; ++c) qv[c] = __ldg(q4 + c);
        for (int r = 0; r < npart; ++r) {
          const uint4* k4 = reinterpret_cast<const uint4*>(a.K + (prow + r) * C::D + sub * C::EPT);
          float acc = 0.f;
#pragma unroll
          for (int c = 0; c < C::EPT / 8; ++c) {
            const uint4 kv = __ldg(k4 + c);
            const uint32_t qw[4] = {qv[c].x, qv[c].y, qv[c].z, qv[c].w};
            const uint32_t kw[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              acc = fmaf(__uint_as_float(qw[e] << 16), __uint_as_float(kw[e] << 16), acc);
              acc = fmaf(__uint_as_float(qw[e] & 0xFFFF0000u), __uint_as_float(kw[e] & 0xFFFF0000u), acc);
            }
          }
#pragma unroll
          for (int o = 1; o < C::TPH; o <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
          if (sub == 0) part[r * HQ + h] = acc * sl2;
        }
      }
      softmax_bar();
      float base[HQ], lsum[HQ];
#pragma unroll
      for (int h = 0; h < HQ; ++h) {
        float b = -INFINITY;
        for (int r = 0; r < npart; ++r) b = fmaxf(b, part[r * HQ + h]);
        base[h] = b;
        lsum[h] = 0.f;
      }
      const int ob = nq & 1;
      const uint32_t o_cols = tmem_base + lane_addr + 2 * HQ + ob * HQ;
      int pnext = (key >> 2) < k ? __ldg(irow + (key >> 2)) : -1;   // this key's idx entry, a tile ahead
      bool stop = false;
      for (int j = 0; j < T; ++j) {
        const int sb = gk & 1;
        const int p = pnext;
        {
          const int slot = (j + 1) * C::SLOTS + (key >> 2);
          pnext = (j + 1 < T && slot < k) ? __ldg(irow + slot) : -1;
        }
        const bool valid = p >= 0 && p < el;
        ok &= mbar_wait(sfull(sb), (gk >> 1) & 1, abort_flag);
        tc_fence_after();
        float x[HQ];
        tmem_ld_cols<HQ>(tmem_base + lane_addr + sb * HQ, x);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(sfree(sb));
        bool exc = false;
#pragma unroll
        for (int h = 0; h < HQ; ++h) {
          x[h] = valid ? x[h] * sl2 : -INFINITY;
          exc |= x[h] > base[h] + kLazy;
        }
        const bool halt = !ok || *abort_flag != 0;
        if (softmax_bar_any(exc || halt)) {
          if (softmax_bar_any(halt)) {
            stop = true;
            break;
          }
          // move the base of every head whose tile maximum is above it by more
          // than kLazy to that maximum; rescale the row sums and O^T
#pragma unroll
          for (int h = 0; h < HQ; ++h) {
            float m = x[h];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            if (lane == 0) red[warp * HQ + h] = m;
          }
          softmax_bar();
          float alpha[HQ];
          bool any_a = false;
#pragma unroll
          for (int h = 0; h < HQ; ++h) {
            const float mt = fmaxf(fmaxf(red[h], red[HQ + h]), fmaxf(red[2 * HQ + h], red[3 * HQ + h]));
            alpha[h] = 1.f;
            if (mt > base[h] + kLazy) {
              alpha[h] = base[h] == -INFINITY ? 0.f : ex2_approx(base[h] - mt);
              base[h] = mt;
              any_a = true;
            }
            lsum[h] *= alpha[h];
          }
          if (any_a && j > 0) {
            // O^T holds P.V of tiles 0..j-1 once the last of them has finished
            ok &= mbar_wait(pvdone((gk - 1) & 1), ((gk - 1) >> 1) & 1, abort_flag);
            tc_fence_after();
            float o[HQ];
            tmem_ld_cols<HQ>(o_cols, o);
            tmem_ld_wait();
#pragma unroll
            for (int h = 0; h < HQ; ++h) o[h] *= alpha[h];
            tmem_st_cols<HQ>(o_cols, o);
            tmem_st_wait();
          }
        }
        // the P buffer of this tile was last read by P.V NPB tiles ago
        if (gk >= (uint32_t)C::NPB)
          ok &= mbar_wait(pvdone((gk - C::NPB) & 1), ((gk - C::NPB) >> 1) & 1, abort_flag);
        const uint32_t pt =
            sP + (gk % C::NPB) * C::P_BUF + (key >> 6) * C::P_CB + (((key & 63) >> 3) << 4) + (key & 7) * 2;
#pragma unroll
        for (int h = 0; h < HQ; ++h) {
          const float bh = base[h] == -INFINITY ? 0.f : base[h];
          const float pf = ex2_approx(x[h] - bh);
          lsum[h] += pf;
          const uint32_t row = pt + h * 128;
          const uint32_t sw = (uint32_t)(h & 7) << 4;   // 128-byte swizzle of row h
          const __nv_bfloat16 hi = __float2bfloat16_rn(pf);
          st_shared_u16(row ^ sw, __bfloat16_as_ushort(hi));
          if constexpr (ACC) {
            const __nv_bfloat16 lo = __float2bfloat16_rn(pf - __bfloat162float(hi));
            st_shared_u16((row + C::P_TERM) ^ sw, __bfloat16_as_ushort(lo));
          }
        }
        fence_proxy_async_shared();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(pfull(sb));
        ++gk;
      }
      if (stop) break;
      // ---- end of the query: row sums, partial pool, O and LSE
#pragma unroll
      for (int h = 0; h < HQ; ++h) {
        float s = lsum[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) rsum[warp * HQ + h] = s;
      }
      softmax_bar();
      float l[HQ];
#pragma unroll
      for (int h = 0; h < HQ; ++h) {
        l[h] = (rsum[h] + rsum[HQ + h]) + (rsum[2 * HQ + h] + rsum[3 * HQ + h]);
        const float bh = base[h] == -INFINITY ? 0.f : base[h];
        for (int r = 0; r < npart; ++r) l[h] += ex2_approx(part[r * HQ + h] - bh);
      }
      ok &= mbar_wait(ofull(ob), (nq >> 1) & 1, abort_flag);
      tc_fence_after();
      float o[HQ];
      tmem_ld_cols<HQ>(o_cols, o);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ofree(ob));
      const int dcol = key;   // TMEM lane of O^T = head dimension
      for (int r = 0; r < npart; ++r) {
        const float vv = __bfloat162float(a.V[(prow + r) * C::D + dcol]);
#pragma unroll
        for (int h = 0; h < HQ; ++h) {
          const float bh = base[h] == -INFINITY ? 0.f : base[h];
          o[h] = fmaf(ex2_approx(part[r * HQ + h] - bh), vv, o[h]);
        }
      }
      __nv_bfloat16* orow = a.O + t * HQ * C::D + dcol;
#pragma unroll
      for (int h = 0; h < HQ; ++h) {
        const float inv = 1.f / l[h];
        orow[h * C::D] = __float2bfloat16_rn(o[h] * inv);
        if constexpr (ACC) __stcs(a.Oacc + (t * HQ + h) * C::D + dcol, o[h] * inv);
      }
      constexpr float kLn2 = 0.6931471805599453f;
#pragma unroll
      for (int h = 0; h < HQ; ++h)
        if (tid == h) a.LSE[t * HQ + h] = (base[h] + log2f(l[h])) * kLn2;
    }
    if (!ok) *abort_flag = 1;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// --------------------------------------------------------------------- host
static PFN_cuTensorMapEncodeTiled_v12000 ftc_encode_fn() {
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

template <int HQ, bool ACC>
static cudaError_t launch_ftc(const FtcArgs& a, cudaStream_t s) {
  using C = FtcCfg<HQ>;
  auto enc = ftc_encode_fn();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap tq;
  const cuuint32_t estr[3] = {1, 1, 1};
  {
    // Q: [L, HQ, 128]; a box is one query's HQ heads x 64 columns
    const cuuint64_t dims[3] = {(cuuint64_t)C::D, (cuuint64_t)HQ, (cuuint64_t)a.L};
    const cuuint64_t strides[2] = {(cuuint64_t)C::D * 2, (cuuint64_t)HQ * C::D * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)HQ, 1};
    if (enc(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<__nv_bfloat16*>(a.Q), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  auto kern = attn_fwd_tc_kernel<HQ, ACC>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  int64_t grid = device_sm_count();
  if (grid > a.L) grid = a.L;
  kern<<<(unsigned)grid, C::THREADS, C::SMEM_BYTES, s>>>(tq, a);
  return cudaGetLastError();
}

bool attn_fwd_tc_supported(int Hq, int d) { return d == 128 && (Hq == 16 || Hq == 32); }

cudaError_t launch_attn_fwd_tc_bf16(int64_t L, int Hq, int d, int k, float scale, const void* q, const void* kk,
                                    const void* v, const int32_t* idx, void* o, float* lse, float* o_acc,
                                    cudaStream_t s) {
  if (!attn_fwd_tc_supported(Hq, d)) return cudaErrorNotSupported;
  FtcArgs a;
  a.Q = static_cast<const __nv_bfloat16*>(q);
  a.K = static_cast<const __nv_bfloat16*>(kk);
  a.V = static_cast<const __nv_bfloat16*>(v);
  a.idx = idx;
  a.O = static_cast<__nv_bfloat16*>(o);
  a.LSE = lse;
  a.Oacc = o_acc;
  a.L = L;
  a.k = k;
  a.scale_log2 = scale * 1.4426950408889634f;
  if (Hq == 16) return o_acc ? launch_ftc<16, true>(a, s) : launch_ftc<16, false>(a, s);
  return o_acc ? launch_ftc<32, true>(a, s) : launch_ftc<32, false>(a, s);
}

}  // namespace dsa
