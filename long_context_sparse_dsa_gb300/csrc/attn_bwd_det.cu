// attn_bwd_det.cu -- the deterministic (key-major) sparse attention backward.
//
// Page "SkyRL extends GLM-5.3-Flash training context to 1 million tokens",
// section "1. DSA truly sparse" (the sparse kernel runs forward and backward)
// and section "Real data" (the trainer's and the inference engine's log-probs
// are compared, which wants gradients that do not change run to run).
//
// Same gradients as attn_bwd.cu (dQ, dK, dV of softmax attention over keys(t);
// no gradient to the indexer inputs), but dK and dV are summed in a fixed
// order, so every run gives the same bits:
//   1. dQ (query-major): attn_bwd.cu's kernel without its dK/dV part; it also
//      stores D[t,h] = dO . O for step 4.
//   2. the selection inverted: for every pool, the queries that selected it,
//      in ascending order (a CSR).  Counts per (pool, 1024-query block), an
//      exclusive scan in (pool, block) order, then a fill in which each CTA
//      walks its block's queries in order with shared-memory cursors, one
//      barrier per query -- so the list order is fixed, not decided by atomics.
//   3. per band of kBand queries (their Q and dO stay in L2), work items of at
//      most kCH queries of one pool's list: a warp loads the pool's 4 K and V
//      rows once and, for each query, its Q and dO rows (all heads) through a
//      3-stage cp.async ring, recomputes S and dP, and accumulates
//      dV^T += dO^T P and dK^T += scale Q^T dS with mma.sync (d on M, the 4
//      keys padded to N = 8, heads on K; P and dS as bf16 hi + lo; each
//      query's product joins the sums with fp32 adds, not inside the MMA's
//      accumulator).  The
//      query's own partial pool counts as a prefix of its pool's stream.  Each
//      item writes its partial sums to its own slot;
//   4. per band, one warp per pool adds its items' partials to dK/dV in item
//      order (chunk 0, 1, ...), after the previous band's.
// Nothing is added with atomics, so the result is bitwise reproducible; the
// order is "band, then chunk, then query", fixed by the selection alone.
#include "common.cuh"
#include "launch.h"

namespace dsa {

constexpr int kDetQB = 1024;      // queries per CSR block
constexpr int kDetPR = 16384;     // pools per CSR CTA (its shared-memory counters: 64 KB)
constexpr int kDetBand = 4096;    // queries per key-major band (a multiple of kDetQB)
constexpr int kDetCH = 128;       // queries per key-major work item
constexpr int kDetNST = 3;        // cp.async stages per key-major warp
constexpr int kScanTile = 4096;   // elements per CTA of the scan

static_assert(kDetBand % kDetQB == 0, "a band is a whole number of CSR blocks");

__host__ __device__ __forceinline__ int64_t lmin(int64_t a, int64_t b) { return a < b ? a : b; }

// ------------------------------------------------------------------ CSR
// cnt[p * nblk + b] = number of queries t of block b with p in idx[t].
__global__ void __launch_bounds__(512) det_csr_count_kernel(const int32_t* __restrict__ idx, int64_t L, int k,
                                                            int64_t P, int nblk, int32_t* __restrict__ cnt) {
  extern __shared__ int32_t det_ctr[];
  const int b = blockIdx.x;
  const int64_t p0 = (int64_t)blockIdx.y * kDetPR;
  const int np = (int)lmin(kDetPR, P - p0);
  for (int i = threadIdx.x; i < np; i += blockDim.x) det_ctr[i] = 0;
  __syncthreads();
  const int64_t t0 = (int64_t)b * kDetQB, t1 = lmin(L, t0 + kDetQB);
  for (int64_t t = t0; t < t1; ++t) {
    const int64_t e = elig(t);
    for (int s = threadIdx.x; s < k; s += blockDim.x) {
      const int32_t p = __ldg(idx + t * k + s);
      if (p >= 0 && p < e && p >= p0 && p < p0 + np) atomicAdd(&det_ctr[p - p0], 1);
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < np; i += blockDim.x) cnt[(p0 + i) * nblk + b] = det_ctr[i];
}

// Three-phase exclusive scan of n int32 values in place; x[n] receives the
// total.  Phase 1: per-tile sums.
__global__ void __launch_bounds__(1024) det_scan_sums_kernel(const int32_t* __restrict__ x, int64_t n,
                                                             int32_t* __restrict__ sums) {
  __shared__ int32_t wsum[32];
  const int64_t base = (int64_t)blockIdx.x * kScanTile;
  int v = 0;
  for (int i = threadIdx.x; i < kScanTile; i += 1024) {
    const int64_t j = base + i;
    v += j < n ? x[j] : 0;
  }
  v = __reduce_add_sync(0xffffffffu, v);
  if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    const int w = __reduce_add_sync(0xffffffffu, wsum[threadIdx.x]);
    if (threadIdx.x == 0) sums[blockIdx.x] = w;
  }
}

// Block-wide exclusive scan of one value per thread (1024 threads).
__device__ __forceinline__ int det_block_scan(int v, int32_t* wbuf, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wbuf[w] = incl;
  __syncthreads();
  if (w == 0) {
    int x = wbuf[lane];
    int xi = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, xi, o);
      if (lane >= o) xi += y;
    }
    wbuf[lane] = xi - x;
    if (lane == 31) wbuf[32] = xi;
  }
  __syncthreads();
  const int r = wbuf[w] + incl - v;
  *total = wbuf[32];
  __syncthreads();
  return r;
}

// Phase 2 (one CTA): exclusive scan of the tile sums, in passes of 1024.
__global__ void __launch_bounds__(1024) det_scan_offsets_kernel(int32_t* __restrict__ sums, int ntiles) {
  __shared__ int32_t wbuf[33];
  int carry = 0;
  for (int base = 0; base < ntiles; base += 1024) {
    const int i = base + threadIdx.x;
    const int v = i < ntiles ? sums[i] : 0;
    int total;
    const int ex = det_block_scan(v, wbuf, &total);
    if (i < ntiles) sums[i] = carry + ex;
    carry += total;
  }
  if (threadIdx.x == 0) sums[ntiles] = carry;
}

// Phase 3: each tile's exclusive scan plus its offset; x[n] = total.
__global__ void __launch_bounds__(1024) det_scan_apply_kernel(int32_t* __restrict__ x, int64_t n,
                                                              const int32_t* __restrict__ offs, int ntiles) {
  __shared__ int32_t wbuf[33];
  constexpr int PER = kScanTile / 1024;
  const int64_t base = (int64_t)blockIdx.x * kScanTile + (int64_t)threadIdx.x * PER;
  int v[PER], sum = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    v[j] = base + j < n ? x[base + j] : 0;
    sum += v[j];
  }
  int total;
  int run = offs[blockIdx.x] + det_block_scan(sum, wbuf, &total);
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    if (base + j < n) x[base + j] = run;
    run += v[j];
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) x[n] = offs[ntiles];
}

// list[base[p*nblk+b] + r] = the r-th query of block b (ascending) that
// selected pool p.  One barrier per query keeps the order.
__global__ void __launch_bounds__(512) det_csr_fill_kernel(const int32_t* __restrict__ idx, int64_t L, int k,
                                                           int64_t P, int nblk, const int32_t* __restrict__ base,
                                                           int32_t* __restrict__ list) {
  extern __shared__ int32_t det_ctr[];
  const int b = blockIdx.x;
  const int64_t p0 = (int64_t)blockIdx.y * kDetPR;
  const int np = (int)lmin(kDetPR, P - p0);
  for (int i = threadIdx.x; i < np; i += blockDim.x) det_ctr[i] = base[(p0 + i) * nblk + b];
  const int64_t t0 = (int64_t)b * kDetQB, t1 = lmin(L, t0 + kDetQB);
  for (int64_t t = t0; t < t1; ++t) {
    __syncthreads();
    const int64_t e = elig(t);
    for (int s = threadIdx.x; s < k; s += blockDim.x) {
      const int32_t p = __ldg(idx + t * k + s);
      if (p >= 0 && p < e && p >= p0 && p < p0 + np) {
        // the pools of one query are distinct, so no other thread touches
        // this counter before the next barrier
        const int pos = det_ctr[p - p0];
        det_ctr[p - p0] = pos + 1;
        list[pos] = (int32_t)t;
      }
    }
  }
}

// ------------------------------------------------------------ work items
// The stream of pool p in band [bt0, bt1): its own partial-pool queries
// 4p..4p+2 that lie in the band (a prefix), then list[s .. e).
struct DetBand {
  int64_t bt0, bt1;   // query range of the band
  int b0, b1;         // its CSR blocks
};

__device__ __forceinline__ void det_stream(const int32_t* __restrict__ base, int nblk, int64_t L, int64_t p,
                                           const DetBand& bd, int& npart, int& s, int& e) {
  s = base[p * nblk + bd.b0];
  e = base[p * nblk + bd.b1];   // b1 may be nblk: that is the next pool's first entry (or the total)
  const int64_t tp = 4 * p;
  npart = (tp >= bd.bt0 && tp < bd.bt1) ? (int)lmin(3, L - tp) : 0;
}

// items[i] = (pool, chunk) for every kDetCH-query chunk of every pool's band
// stream; first[p] = the item of the pool's chunk 0, nch[p] = its chunks.
__global__ void __launch_bounds__(256) det_items_kernel(const int32_t* __restrict__ base, int nblk, int64_t L,
                                                        int64_t P, DetBand bd, int2* __restrict__ items,
                                                        uint32_t* __restrict__ nitems, int32_t* __restrict__ first,
                                                        int32_t* __restrict__ nch) {
  const int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (p >= P) return;
  int npart, s, e;
  det_stream(base, nblk, L, p, bd, npart, s, e);
  const int n = npart + (e - s);
  const int c = (n + kDetCH - 1) / kDetCH;
  nch[p] = c;
  if (c == 0) return;
  const int f = (int)atomicAdd(nitems, (uint32_t)c);
  first[p] = f;
  for (int i = 0; i < c; ++i) items[f + i] = make_int2((int)p, i);
}

// ------------------------------------------------------------ key-major
template <int D, int HG>
struct DetCfg {
  static constexpr int ROW_BYTES = D * 2;
  static constexpr int CHUNKS = D / 8;                 // 16-byte chunks per row
  static constexpr int TILE = 16 * ROW_BYTES;          // 16 heads x D, one tensor, one head group
  static constexpr int AUX = 2 * 16 * 4 * HG + 16;     // LSE and D of every head; the query and its rows
  static constexpr int STAGE = 2 * HG * TILE + AUX;    // Q and dO of all heads, LSE, D
  static constexpr int KV = 2 * 8 * ROW_BYTES;         // K and V rows of the pool (8 rows: 4 keys + zero padding)
  static constexpr int WARP_BYTES = kDetNST * STAGE + KV;
  static constexpr int WARPS = (220 * 1024) / WARP_BYTES >= 8 ? 8 : (220 * 1024) / WARP_BYTES;
  static constexpr int SMEM = WARPS * WARP_BYTES;
  static_assert(STAGE % 16 == 0 && WARP_BYTES % 16 == 0, "16-byte alignment");
};

// Partial sums of one item: [2][4][D] fp32 (0: dV, 1: dK; keys of the pool).
template <int D, int HG>
__global__ void __launch_bounds__(32 * DetCfg<D, HG>::WARPS) det_keymajor_kernel(
    const __nv_bfloat16* __restrict__ Q, const __nv_bfloat16* __restrict__ K, const __nv_bfloat16* __restrict__ V,
    const __nv_bfloat16* __restrict__ dO, const float* __restrict__ LSE, const float* __restrict__ Dbuf,
    const int32_t* __restrict__ base, const int32_t* __restrict__ list, int nblk, int64_t L, DetBand bd,
    const int2* __restrict__ items, const uint32_t* __restrict__ nitems, float* __restrict__ part, float scale,
    float scale_log2) {
  using C = DetCfg<D, HG>;
  constexpr int Hq = 16 * HG;
  extern __shared__ __align__(128) unsigned char det_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, qi = lane & 3;
  const uint32_t wbase = smem_u32(det_smem) + warp * C::WARP_BYTES;
  const uint32_t kvs = wbase + kDetNST * C::STAGE;   // K rows then V rows
  unsigned char* kvp = det_smem + warp * C::WARP_BYTES + kDetNST * C::STAGE;
  // K/V rows 4..7 stay zero (the N padding of the MMAs)
  for (int i = lane; i < C::KV / 16; i += 32) {
    const int row = (i / C::CHUNKS) % 8;
    if (row >= 4) reinterpret_cast<uint4*>(kvp)[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  __syncwarp();
  constexpr float kLog2e = 1.4426950408889634f;
  const uint32_t n_items = *nitems;
  const int64_t gw = (int64_t)blockIdx.x * C::WARPS + warp, nw = (int64_t)gridDim.x * C::WARPS;
  for (int64_t it = gw; it < n_items; it += nw) {
    const int2 pc = __ldg(items + it);
    const int64_t p = pc.x;
    int npart, s, e;
    det_stream(base, nblk, L, p, bd, npart, s, e);
    const int n = npart + (e - s);
    const int j0 = pc.y * kDetCH, j1 = min(n, j0 + kDetCH);
    // the pool's K and V rows (swizzled: chunk c of row r at c ^ (r & 7))
    for (int i = lane; i < 2 * 4 * C::CHUNKS; i += 32) {
      const int tn = i / (4 * C::CHUNKS), rem = i % (4 * C::CHUNKS);
      const int row = rem / C::CHUNKS, ch = rem % C::CHUNKS;
      const __nv_bfloat16* src = (tn ? V : K) + (4 * p + row) * D + ch * 8;
      cp_async16(kvs + tn * 8 * C::ROW_BYTES + row * C::ROW_BYTES + ((ch ^ row) << 4), src, 16);
    }
    // element j of the stream: query t and its visible rows of the pool
    auto elem = [&](int j, int64_t& t, int& nrows) {
      if (j < npart) {
        t = 4 * p + j;
        nrows = j + 1;
      } else {
        t = __ldg(list + s + (j - npart));
        nrows = (t >= 4 * p + 3 && t < L) ? 4 : 0;   // a list entry is always eligible; anything else is skipped
        if (nrows == 0) t = 4 * p;                   // a valid address, rows masked
      }
    };
    // Q and dO of all heads of query t, then its LSE and D, into stage st
    auto fetch = [&](int j, int st) {
      int64_t t;
      int nr;
      elem(j, t, nr);
      const uint32_t sb = wbase + st * C::STAGE;
#pragma unroll
      for (int tn = 0; tn < 2; ++tn) {
        const __nv_bfloat16* src = (tn ? dO : Q) + t * Hq * D;
        for (int i = lane; i < HG * 16 * C::CHUNKS; i += 32) {
          const int row = i / C::CHUNKS, ch = i % C::CHUNKS;   // row = head (all head groups)
          cp_async16(sb + tn * HG * C::TILE + row * C::ROW_BYTES + ((ch ^ (row & 7)) << 4),
                     src + row * D + ch * 8, 16);
        }
      }
      if (lane < 2 * 4 * HG) {   // 16-byte chunks of LSE (first 4*HG) and D
        const int which = lane / (4 * HG), ch = lane % (4 * HG);
        cp_async16(sb + 2 * HG * C::TILE + which * 64 * HG + ch * 16, (which ? Dbuf : LSE) + t * Hq + ch * 4, 16);
      }
      // the element's query and visible rows, for the step that consumes it
      // (so no global load sits on that step's critical path); the stage's
      // previous reader finished before this warp's last __syncwarp
      if (lane == 0) {
        int* meta = reinterpret_cast<int*>(det_smem + (sb - smem_u32(det_smem)) + 2 * HG * C::TILE + 2 * 64 * HG);
        meta[0] = (int)t;
        meta[1] = nr;
      }
    };
    float accv[HG][D / 16][4], acck[HG][D / 16][4];
#pragma unroll
    for (int hg = 0; hg < HG; ++hg)
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
        for (int c = 0; c < 4; ++c) accv[hg][mt][c] = acck[hg][mt][c] = 0.f;
    // prologue: the first two elements (the K/V copies join the first group)
    if (j0 < j1) fetch(j0, 0);
    cp_async_commit();
    if (j0 + 1 < j1) fetch(j0 + 1, 1);
    cp_async_commit();
    for (int j = j0; j < j1; ++j) {
      const int st = (j - j0) % kDetNST;
      if (j + 2 < j1) fetch(j + 2, (j + 2 - j0) % kDetNST);
      cp_async_commit();
      cp_async_wait<2>();
      __syncwarp();
      const uint32_t sb = wbase + st * C::STAGE;
      const float* aux = reinterpret_cast<const float*>(det_smem + (sb - smem_u32(det_smem)) + 2 * HG * C::TILE);
      const int nrows = reinterpret_cast<const int*>(aux + 2 * 16 * HG)[1];
#pragma unroll
      for (int hg = 0; hg < HG; ++hg) {
        const uint32_t qs = sb + hg * 16 * C::ROW_BYTES;                 // heads hg*16 .. +15 of Q
        const uint32_t ds = sb + HG * C::TILE + hg * 16 * C::ROW_BYTES;  // and of dO
        // S = Q K^T and dP = dO V^T: heads x 8 keys (keys 4..7 are zero rows),
        // even and odd k-steps in two chains added at the end -- the same
        // arithmetic as the query-major kernel, so S, P, dP and dS are the
        // same values there and here
        float sc[4] = {0.f, 0.f, 0.f, 0.f}, dp[4] = {0.f, 0.f, 0.f, 0.f};
        float sc2[4] = {0.f, 0.f, 0.f, 0.f}, dp2[4] = {0.f, 0.f, 0.f, 0.f};
        {
          const int arow = lane & 15, ach = lane >> 4;
          const int brow = lane & 7, bch = lane >> 3;
#pragma unroll
          for (int ks = 0; ks < D / 16; ks += 2) {
            uint32_t a[2][4], q2[2][4], kb[4], vb[4];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int ch = 2 * (ks + u) + ach;
              ldsm_x4(qs + arow * C::ROW_BYTES + ((ch ^ (arow & 7)) << 4), a[u][0], a[u][1], a[u][2], a[u][3]);
              ldsm_x4(ds + arow * C::ROW_BYTES + ((ch ^ (arow & 7)) << 4), q2[u][0], q2[u][1], q2[u][2], q2[u][3]);
            }
            const int chb = 2 * ks + bch;   // chunks 2ks .. 2ks+3 (two k-steps)
            ldsm_x4(kvs + brow * C::ROW_BYTES + ((chb ^ brow) << 4), kb[0], kb[1], kb[2], kb[3]);
            ldsm_x4(kvs + 8 * C::ROW_BYTES + brow * C::ROW_BYTES + ((chb ^ brow) << 4), vb[0], vb[1], vb[2], vb[3]);
            mma_bf16_16816(sc, a[0][0], a[0][1], a[0][2], a[0][3], kb[0], kb[1]);
            mma_bf16_16816(dp, q2[0][0], q2[0][1], q2[0][2], q2[0][3], vb[0], vb[1]);
            mma_bf16_16816(sc2, a[1][0], a[1][1], a[1][2], a[1][3], kb[2], kb[3]);
            mma_bf16_16816(dp2, q2[1][0], q2[1][1], q2[1][2], q2[1][3], vb[2], vb[3]);
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            sc[e] += sc2[e];
            dp[e] += dp2[e];
          }
        }
        // P and dS (rows g, g+8 = heads; cols 2qi, 2qi+1 = keys)
        const float lse_g = aux[hg * 16 + g] * kLog2e, lse_g8 = aux[hg * 16 + g + 8] * kLog2e;
        const float d_g = aux[16 * HG + hg * 16 + g], d_g8 = aux[16 * HG + hg * 16 + g + 8];
        const bool v0 = 2 * qi < nrows, v1 = 2 * qi + 1 < nrows;
        const float p0 = ex2_approx(v0 ? sc[0] * scale_log2 - lse_g : -INFINITY);
        const float p1 = ex2_approx(v1 ? sc[1] * scale_log2 - lse_g : -INFINITY);
        const float p2 = ex2_approx(v0 ? sc[2] * scale_log2 - lse_g8 : -INFINITY);
        const float p3 = ex2_approx(v1 ? sc[3] * scale_log2 - lse_g8 : -INFINITY);
        const float s0 = scale * p0 * (dp[0] - d_g), s1 = scale * p1 * (dp[1] - d_g);
        const float s2 = scale * p2 * (dp[2] - d_g8), s3 = scale * p3 * (dp[3] - d_g8);
        // B operands (k = head, n = key) of P and scale*dS, hi and lo parts:
        // the transposes of the accumulator's 8x8 blocks
        uint32_t pb[2][2], db[2][2];
        {
          uint32_t hi, lo;
          hi = pack_bf16(p0, p1);
          lo = pack_bf16(p0 - __uint_as_float(hi << 16), p1 - __uint_as_float(hi & 0xFFFF0000u));
          pb[0][0] = movmatrix_t(hi);
          pb[1][0] = movmatrix_t(lo);
          hi = pack_bf16(p2, p3);
          lo = pack_bf16(p2 - __uint_as_float(hi << 16), p3 - __uint_as_float(hi & 0xFFFF0000u));
          pb[0][1] = movmatrix_t(hi);
          pb[1][1] = movmatrix_t(lo);
          hi = pack_bf16(s0, s1);
          lo = pack_bf16(s0 - __uint_as_float(hi << 16), s1 - __uint_as_float(hi & 0xFFFF0000u));
          db[0][0] = movmatrix_t(hi);
          db[1][0] = movmatrix_t(lo);
          hi = pack_bf16(s2, s3);
          lo = pack_bf16(s2 - __uint_as_float(hi << 16), s3 - __uint_as_float(hi & 0xFFFF0000u));
          db[0][1] = movmatrix_t(hi);
          db[1][1] = movmatrix_t(lo);
        }
        // dV^T += dO^T P and dK^T += Q^T (scale dS): d on M (tiles of 16), heads on K
        {
          const int mtx = lane >> 3, r = lane & 7;
          const int hrow = (mtx >> 1) * 8 + r;
#pragma unroll
          for (int mt = 0; mt < D / 16; ++mt) {
            const int ch = 2 * mt + (mtx & 1);
            uint32_t ao[4], aq[4];
            ldsm_x4_t(ds + hrow * C::ROW_BYTES + ((ch ^ (hrow & 7)) << 4), ao[0], ao[1], ao[2], ao[3]);
            ldsm_x4_t(qs + hrow * C::ROW_BYTES + ((ch ^ (hrow & 7)) << 4), aq[0], aq[1], aq[2], aq[3]);
            // each query's product starts from zero and joins the running
            // sums with ordinary fp32 adds: the tensor core's own fp32
            // accumulation does not round like an add, and over a pool's
            // whole list (113k queries for the most-selected pool at 128k)
            // its error builds up
            float tv[4] = {0.f, 0.f, 0.f, 0.f}, tk[4] = {0.f, 0.f, 0.f, 0.f};
            mma_bf16_16816(tv, ao[0], ao[1], ao[2], ao[3], pb[0][0], pb[0][1]);
            mma_bf16_16816(tk, aq[0], aq[1], aq[2], aq[3], db[0][0], db[0][1]);
            mma_bf16_16816(tv, ao[0], ao[1], ao[2], ao[3], pb[1][0], pb[1][1]);
            mma_bf16_16816(tk, aq[0], aq[1], aq[2], aq[3], db[1][0], db[1][1]);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              accv[hg][mt][c] += tv[c];
              acck[hg][mt][c] += tk[c];
            }
          }
        }
      }
      __syncwarp();
    }
    cp_async_wait<0>();
    __syncwarp();
    // the item's partial sums: lanes with qi < 2 hold keys 2qi, 2qi+1; head
    // groups are added here (a fixed order)
    float* dst = part + it * (int64_t)(2 * 4 * D);
    if (qi < 2) {
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        float v[4], kk[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          v[c] = accv[0][mt][c];
          kk[c] = acck[0][mt][c];
        }
#pragma unroll
        for (int hg = 1; hg < HG; ++hg)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            v[c] += accv[hg][mt][c];
            kk[c] += acck[hg][mt][c];
          }
        const int dd = mt * 16 + g;
        const int k0 = 2 * qi, k1 = 2 * qi + 1;
        dst[(0 * 4 + k0) * D + dd] = v[0];
        dst[(0 * 4 + k1) * D + dd] = v[1];
        dst[(0 * 4 + k0) * D + dd + 8] = v[2];
        dst[(0 * 4 + k1) * D + dd + 8] = v[3];
        dst[(1 * 4 + k0) * D + dd] = kk[0];
        dst[(1 * 4 + k1) * D + dd] = kk[1];
        dst[(1 * 4 + k0) * D + dd + 8] = kk[2];
        dst[(1 * 4 + k1) * D + dd + 8] = kk[3];
      }
    }
    __syncwarp();
  }
}

// dK/dV of every pool with items in this band += the items' partials, in
// chunk order (one warp per pool; each lane owns D/8 consecutive values of
// each of the 8 rows).
template <int D>
__global__ void __launch_bounds__(128) det_combine_kernel(const int32_t* __restrict__ first,
                                                          const int32_t* __restrict__ nch, int64_t P,
                                                          const float* __restrict__ part, float* __restrict__ dK,
                                                          float* __restrict__ dV) {
  const int64_t p = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
  if (p >= P) return;
  const int lane = threadIdx.x & 31;
  const int c = nch[p];
  if (c == 0) return;
  const int f = first[p];
  constexpr int PER = 2 * 4 * D / 32;   // values per lane
  float acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  for (int ch = 0; ch < c; ++ch) {
    const float4* src = reinterpret_cast<const float4*>(part + (int64_t)(f + ch) * (2 * 4 * D)) + lane * (PER / 4);
#pragma unroll
    for (int i = 0; i < PER / 4; ++i) {
      const float4 x = __ldg(src + i);
      acc[4 * i] += x.x;
      acc[4 * i + 1] += x.y;
      acc[4 * i + 2] += x.z;
      acc[4 * i + 3] += x.w;
    }
  }
  // lane's values: flat index lane*PER .. +PER-1 of [2][4][D]
  const int flat = lane * PER;
  const int tn = flat / (4 * D), rem = flat % (4 * D);
  const int key = rem / D, dd = rem % D;
  float* dst = (tn ? dK : dV) + (4 * p + key) * D + dd;
#pragma unroll
  for (int i = 0; i < PER; ++i) dst[i] += acc[i];
}

// ------------------------------------------------------------------ host
namespace {
size_t al256(size_t b) { return (b + 255) & ~(size_t)255; }

struct DetWs {
  float* dbuf;        // [L, Hq]
  int32_t* cnt;       // [P * nblk + 1]  counts, then offsets
  int32_t* sums;      // [ntiles + 1]
  int32_t* list;      // [L * k]
  int2* items;        // [max items per band]
  uint32_t* nitems;   // [1]
  int32_t* first;     // [P]
  int32_t* nch;       // [P]
  float* part;        // [max items per band][2][4][d]
  size_t bytes;
};

DetWs det_carve(void* ws, int64_t L, int Hq, int d, int k) {
  DetWs w{};
  const int64_t P = L / 4;
  const int nblk = (int)((L + kDetQB - 1) / kDetQB);
  const int64_t n = P * nblk;
  const int ntiles = (int)((n + kScanTile - 1) / kScanTile);
  const int64_t max_items = ((int64_t)kDetBand * (k + 1) + kDetCH - 1) / kDetCH + P;
  char* p = static_cast<char*>(ws);
  size_t off = 0;
  auto take = [&](size_t b) {
    char* q = p ? p + off : nullptr;
    off += al256(b);
    return q;
  };
  w.dbuf = reinterpret_cast<float*>(take((size_t)L * Hq * 4));
  w.cnt = reinterpret_cast<int32_t*>(take((size_t)(n + 1) * 4));
  w.sums = reinterpret_cast<int32_t*>(take((size_t)(ntiles + 1) * 4));
  w.list = reinterpret_cast<int32_t*>(take((size_t)L * k * 4));
  w.items = reinterpret_cast<int2*>(take((size_t)max_items * 8));
  w.nitems = reinterpret_cast<uint32_t*>(take(16));
  w.first = reinterpret_cast<int32_t*>(take((size_t)P * 4));
  w.nch = reinterpret_cast<int32_t*>(take((size_t)P * 4));
  w.part = reinterpret_cast<float*>(take((size_t)max_items * 2 * 4 * d * 4));
  w.bytes = off;
  return w;
}

template <int D, int HG>
cudaError_t launch_keymajor(const __nv_bfloat16* q, const __nv_bfloat16* kk, const __nv_bfloat16* v,
                            const __nv_bfloat16* dout, const float* lse, const DetWs& w, int nblk, int64_t L,
                            const DetBand& bd, float scale, cudaStream_t s) {
  using C = DetCfg<D, HG>;
  auto kern = det_keymajor_kernel<D, HG>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)device_sm_count(), 32 * C::WARPS, C::SMEM, s>>>(q, kk, v, dout, lse, w.dbuf, w.cnt, w.list, nblk,
                                                                  L, bd, w.items, w.nitems, w.part, scale,
                                                                  scale * 1.4426950408889634f);
  return cudaGetLastError();
}
}  // namespace

size_t det_bwd_ws_bytes(int64_t L, int Hq, int d, int k) { return det_carve(nullptr, L, Hq, d, k).bytes; }

cudaError_t launch_attn_bwd_det_bf16(int64_t L, int Hq, int d, int k, float scale, const void* q, const void* kk,
                                     const void* v, const int32_t* idx, const float* lse, const void* dout,
                                     const float* oacc, float* dq, float* dk, float* dv, void* ws, cudaStream_t s) {
  if (!((d == 128 || d == 64) && (Hq == 16 || Hq == 32))) return cudaErrorNotSupported;
  const DetWs w = det_carve(ws, L, Hq, d, k);
  const int64_t P = L / 4;
  const int nblk = (int)((L + kDetQB - 1) / kDetQB);
  const int64_t n = P * nblk;
  const int ntiles = (int)((n + kScanTile - 1) / kScanTile);
  const int nrange = (int)((P + kDetPR - 1) / kDetPR);
  // 1. dQ, and D for the key-major half
  cudaError_t e = launch_attn_bwd_dq_bf16(L, Hq, d, k, scale, q, kk, v, idx, lse, dout, oacc, w.dbuf, dq, s);
  if (e != cudaSuccess) return e;
  // 2. the selection inverted
  const int ctr_bytes = kDetPR * 4;
  if ((e = cudaFuncSetAttribute(det_csr_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, ctr_bytes)) !=
      cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(det_csr_fill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, ctr_bytes)) !=
      cudaSuccess)
    return e;
  det_csr_count_kernel<<<dim3((unsigned)nblk, (unsigned)nrange), 512, ctr_bytes, s>>>(idx, L, k, P, nblk, w.cnt);
  det_scan_sums_kernel<<<(unsigned)ntiles, 1024, 0, s>>>(w.cnt, n, w.sums);
  det_scan_offsets_kernel<<<1, 1024, 0, s>>>(w.sums, ntiles);
  det_scan_apply_kernel<<<(unsigned)ntiles, 1024, 0, s>>>(w.cnt, n, w.sums, ntiles);
  det_csr_fill_kernel<<<dim3((unsigned)nblk, (unsigned)nrange), 512, ctr_bytes, s>>>(idx, L, k, P, nblk, w.cnt,
                                                                                       w.list);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // 3-4. per band: items, key-major partials, ordered combine
  if ((e = cudaMemsetAsync(dk, 0, (size_t)L * d * 4, s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(dv, 0, (size_t)L * d * 4, s)) != cudaSuccess) return e;
  auto qp = static_cast<const __nv_bfloat16*>(q);
  auto kp = static_cast<const __nv_bfloat16*>(kk);
  auto vp = static_cast<const __nv_bfloat16*>(v);
  auto gp = static_cast<const __nv_bfloat16*>(dout);
  for (int64_t bt0 = 0; bt0 < L; bt0 += kDetBand) {
    DetBand bd;
    bd.bt0 = bt0;
    bd.bt1 = lmin(L, bt0 + kDetBand);
    bd.b0 = (int)(bt0 / kDetQB);
    bd.b1 = (int)lmin(nblk, (bt0 + kDetBand) / kDetQB);
    if ((e = cudaMemsetAsync(w.nitems, 0, 4, s)) != cudaSuccess) return e;
    det_items_kernel<<<(unsigned)((P + 255) / 256), 256, 0, s>>>(w.cnt, nblk, L, P, bd, w.items, w.nitems, w.first,
                                                                 w.nch);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (d == 128)
      e = Hq == 16 ? launch_keymajor<128, 1>(qp, kp, vp, gp, lse, w, nblk, L, bd, scale, s)
                   : launch_keymajor<128, 2>(qp, kp, vp, gp, lse, w, nblk, L, bd, scale, s);
    else
      e = Hq == 16 ? launch_keymajor<64, 1>(qp, kp, vp, gp, lse, w, nblk, L, bd, scale, s)
                   : launch_keymajor<64, 2>(qp, kp, vp, gp, lse, w, nblk, L, bd, scale, s);
    if (e != cudaSuccess) return e;
    if (d == 128)
      det_combine_kernel<128><<<(unsigned)((P + 3) / 4), 128, 0, s>>>(w.first, w.nch, P, w.part, dk, dv);
    else
      det_combine_kernel<64><<<(unsigned)((P + 3) / 4), 128, 0, s>>>(w.first, w.nch, P, w.part, dk, dv);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace dsa
