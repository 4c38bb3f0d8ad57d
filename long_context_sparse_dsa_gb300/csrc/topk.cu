// topk.cu -- per-query top-k pool selection by radix select over fp32 bits.
//
// Page "SkyRL extends GLM-5.3-Flash training context to 1 million tokens",
// section "Model and bottleneck" (about 2048 keys = 512 pools per query) and
// section "1. DSA truly sparse" (selected pool indices are int32).
//
// For query t only the causal prefix p < elig(t) of its score row is read.
// If elig(t) <= k every eligible pool is kept.  Otherwise the k-th largest
// score is found exactly by three radix rounds (11 + 11 + 10 bits) over an
// order-preserving uint32 key of the fp32 score (-0 is folded into +0 so the
// two tie), and an ordered selection keeps every score above that threshold
// plus the lowest-indexed ties at it.  The output is in ascending pool order
// and padded with -1; the result depends only on the scores (no atomics
// decide order), so it is bitwise reproducible.  Scores are taken to be
// finite (the indexer gives finite scores for finite inputs): a NaN score has
// no defined rank.
//
// One CTA of kTopkThreads threads per row, one read of the row in the
// common case:
//   1. 1024 evenly spaced samples give a threshold tau: the lower edge of the
//      22-bit key bin of the r-th largest sample (two radix rounds),
//      r = mu + 4 sqrt(mu) + 2 with mu = k * 1024 / n the expected
//      number of samples at or above the k-th score, so that tau lies below
//      the k-th score with high probability while few scores pass it (rows of
//      at most kCandCap scores skip this and keep every score);
//   2. one pass over the row copies every score >= tau, with its index, into
//      shared memory; each warp compacts its own contiguous segment in index
//      order, so the candidates come out in ascending pool order with no
//      block-wide scan;
//   3. the exact radix select and the ordered selection run on those
//      candidates.
// Scores equal to tau are counted but not stored.  When fewer than k scores
// are above tau and the ties at tau make up the rest, the k-th score is tau
// itself: the row keeps every stored score plus the lowest-indexed ties, which
// the warps holding them collect in a short second scan of their segments.
// Rows of small integer scores (thousands of exact ties at the k-th value)
// take this path instead of the fallback.
// If the candidates number fewer than k (tau too high) or overflow the
// buffer, the row falls back to the exact two-pass path:
// a histogram pass, then an ordered compaction of the threshold bin and
// above, or -- when even that overflows -- rounds and selection over the
// whole row.
#include "common.cuh"
#include "launch.h"

namespace dsa {

constexpr int kTopkThreads = 256;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kCandCap = 4096;                        // candidate keys + indices in SMEM (32 KB)
constexpr int kWarpCap = kCandCap / kTopkWarps;       // per-warp compaction region
constexpr int kSamples = 1024;
constexpr int kStreamUnroll = 4;                      // 128-score groups a warp loads per iteration
constexpr int kTieUnroll = 8;                         // 32-score groups per iteration when collecting ties

// Exclusive block-wide scan of one int per thread.  Returns the exclusive
// prefix; *total receives the block sum.  Contains __syncthreads().
__device__ __forceinline__ int block_excl_scan(int v, int* warp_buf, int* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_buf[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    int x = lane < kTopkWarps ? warp_buf[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane < kTopkWarps) warp_buf[lane] = x;
  }
  __syncthreads();
  const int base = wid ? warp_buf[wid - 1] : 0;
  *total = warp_buf[kTopkWarps - 1];
  __syncthreads();
  return base + incl - v;
}

// Predicated shared-memory writes: one instruction each, no branch around
// them (a predicated-off instruction does not touch its address).
__device__ __forceinline__ void st_shared_u32_if(uint32_t addr, uint32_t v, bool pred) {
  asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %2, 0;\n@p st.shared.u32 [%0], %1;\n}\n" ::"r"(addr), "r"(v),
               "r"((uint32_t)pred)
               : "memory");
}
__device__ __forceinline__ void red_shared_add_if(uint32_t addr, uint32_t v, bool pred) {
  asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %2, 0;\n@p red.shared.add.u32 [%0], %1;\n}\n" ::"r"(addr),
               "r"(v), "r"((uint32_t)pred)
               : "memory");
}
__device__ __forceinline__ void st_global_s32_if(int32_t* addr, int32_t v, bool pred) {
  asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %2, 0;\n@p st.global.s32 [%0], %1;\n}\n" ::"l"(addr), "r"(v),
               "r"((uint32_t)pred)
               : "memory");
}

// Histogram add: one shared-memory atomic add per key (bin < 0: none).
// Aggregating equal bins across the warp first (match_any, then one add per
// group) was slower at 128k (4.74 against 4.37 ms per step) and even on the
// tie-heavy 1M rows it was written for (189 against 173 ms).
__device__ __forceinline__ void hist_add(int* hist, int bin) {
  red_shared_add_if(smem_u32(hist) + 4u * (uint32_t)bin, 1u, bin >= 0);
}

// Find, scanning bins from the top, the bin where the running count reaches
// `need`.  Writes the bin and the count strictly above it to sel[0], sel[1].
// NBINS is 1024 or 2048: each thread owns 4 or 8 consecutive bins, read as
// int4 vectors into registers.
template <int NBINS>
__device__ __forceinline__ void find_bin(const int* hist, int need, int* warp_buf, int* sel) {
  constexpr int PER = NBINS / kTopkThreads;
  static_assert(PER == 4 || PER == 8, "4 or 8 bins per thread");
  // thread i owns the bins NBINS-PER*(i+1) .. NBINS-1-PER*i (thread 0 the highest)
  const int lo = NBINS - PER * (threadIdx.x + 1);
  int h[PER];
#pragma unroll
  for (int v = 0; v < PER / 4; ++v) {
    const int4 x = reinterpret_cast<const int4*>(hist + lo)[v];
    h[4 * v] = x.x;
    h[4 * v + 1] = x.y;
    h[4 * v + 2] = x.z;
    h[4 * v + 3] = x.w;
  }
  int local = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) local += h[j];
  int total;
  int cum = block_excl_scan(local, warp_buf, &total);
  if (cum < need && cum + local >= need) {
#pragma unroll
    for (int j = PER - 1; j >= 0; --j) {   // from the highest bin down
      if (cum < need && cum + h[j] >= need) {
        sel[0] = lo + j;
        sel[1] = cum;
      }
      cum += h[j];
    }
  }
  __syncthreads();
}

// Zero the first NBINS histogram bins (int4 stores).
template <int NBINS>
__device__ __forceinline__ void zero_hist(int* hist) {
  for (int b = threadIdx.x; b < NBINS / 4; b += kTopkThreads) reinterpret_cast<int4*>(hist)[b] = make_int4(0, 0, 0, 0);
}

// `need`-th largest key among keys[0..m) (need <= m) by radix rounds of
// 11, 11 and 10 bits.  With ROUNDS = 3 it returns that key exactly and sets
// *above = how many keys are > it.  With ROUNDS = 2 it returns the lower edge
// of the 22-bit bin holding that key (a threshold at or below it).
template <int ROUNDS = 3>
__device__ __forceinline__ uint32_t select_kth(const uint32_t* keys, int m, int need, int* hist, int* warp_buf,
                                               int* sel, int* above) {
  const int m_round = (m + kTopkThreads - 1) / kTopkThreads * kTopkThreads;
  uint32_t prefix = 0;
  int got_above = 0;
  const int shifts[3] = {21, 10, 0};
  const int widths[3] = {11, 11, 10};
#pragma unroll
  for (int round = 0; round < ROUNDS; ++round) {
    const int nb = 1 << widths[round];
    if (round < 2)
      zero_hist<2048>(hist);
    else
      zero_hist<1024>(hist);
    __syncthreads();
    const int sh = shifts[round];
    const int hi = sh + widths[round];   // bits above this digit must equal the prefix
    for (int i = threadIdx.x; i < m_round; i += kTopkThreads) {
      int bin = -1;
      if (i < m) {
        const uint32_t key = keys[i];
        const bool match = hi >= 32 ? true : ((key >> hi) == prefix);
        if (match) bin = (int)((key >> sh) & (uint32_t)(nb - 1));
      }
      hist_add(hist, bin);
    }
    __syncthreads();
    if (round < 2)
      find_bin<2048>(hist, need, warp_buf, sel);
    else
      find_bin<1024>(hist, need, warp_buf, sel);
    prefix = (prefix << widths[round]) | (uint32_t)sel[0];
    need -= sel[1];
    got_above += sel[1];
  }
  *above = got_above;
  return ROUNDS == 3 ? prefix : (prefix << 10);
}

// One tile of the ordered selection: keep keys > T and the first `need_eq`
// keys == T in index order.  Positions come from block-wide scans, so the
// output is in ascending index order.  `ids` maps tile positions to pool
// indices (nullptr: the position is the pool index).
__device__ __forceinline__ void select_tile(const uint32_t (&kk)[4], int base, int n, uint32_t T, int need_eq,
                                            int& eq_seen, int& taken, int* warp_buf, const int32_t* ids,
                                            int32_t* out) {
  int n_eq = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) n_eq += (base + j < n && kk[j] == T);
  int eq_total;
  int eq_rank = eq_seen + block_excl_scan(n_eq, warp_buf, &eq_total);
  bool take[4];
  int n_take = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const bool valid = base + j < n;
    const bool gt = valid && kk[j] > T;
    const bool eq = valid && kk[j] == T;
    take[j] = gt || (eq && eq_rank < need_eq);
    eq_rank += eq;
    n_take += take[j];
  }
  int take_total;
  int pos = taken + block_excl_scan(n_take, warp_buf, &take_total);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    // ids[] is read for every valid position (taken or not) so the store can be predicated
    const int32_t v = ids ? (base + j < n ? ids[base + j] : 0) : base + j;
    st_global_s32_if(out + pos, v, take[j]);
    pos += take[j];
  }
  eq_seen += eq_total;
  taken += take_total;
}

// Ordered selection of the top k over candidates (keys, ids) in index order.
__device__ __forceinline__ void select_from_candidates(const uint32_t* cand_key, const int32_t* cand_idx, int m,
                                                       int k, int* hist, int* warp_buf, int* sel, int32_t* out) {
  int above;
  const uint32_t T = select_kth(cand_key, m, k, hist, warp_buf, sel, &above);
  const int need_eq = k - above;
  const int c_round = (m + 4 * kTopkThreads - 1) / (4 * kTopkThreads) * (4 * kTopkThreads);
  int eq_seen = 0, taken = 0;
  for (int base = threadIdx.x * 4; base < c_round && taken < k; base += 4 * kTopkThreads) {
    uint32_t kk[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) kk[j] = (base + j < m) ? cand_key[base + j] : 0u;
    select_tile(kk, base, m, T, need_eq, eq_seen, taken, warp_buf, cand_idx, out);
  }
}

// The selection of one row (row r of the score block, query q_begin + r),
// done by the whole CTA.
__device__ __forceinline__ void topk_row(const float* __restrict__ scores, int64_t P, int k, int64_t q_begin,
                                         int64_t r, int32_t* __restrict__ idx) {
  __shared__ __align__(16) int hist[2048];
  __shared__ int warp_buf[32];
  __shared__ int sel[4];
  __shared__ int warp_cnt[kTopkWarps];
  __shared__ int warp_eq[kTopkWarps];
  __shared__ int flag_overflow;
  __shared__ __align__(16) uint32_t cand_key[kCandCap];
  __shared__ __align__(16) int32_t cand_idx[kCandCap];
  __shared__ uint32_t samples[kSamples];

  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int64_t t = q_begin + r;
  const int64_t n64 = elig(t);
  int32_t* out = idx + t * (int64_t)k;
  if (n64 <= k) {
    for (int i = threadIdx.x; i < k; i += kTopkThreads) out[i] = i < n64 ? i : -1;
    return;
  }
  const int n = (int)n64;
  const float* row = scores + r * P;
  const bool vec4 = ((P & 3) == 0) && ((reinterpret_cast<uintptr_t>(scores) & 15) == 0);

  // ---- 1. threshold from evenly spaced samples ------------------------------
  uint32_t tau = 0u;   // every key is >= 0
  if (n > kCandCap) {
    for (int i = threadIdx.x; i < kSamples; i += kTopkThreads)
      samples[i] = order_key(__ldg(row + (int)(((int64_t)i * n) / kSamples)));
    __syncthreads();
    // mu = expected samples at or above the true k-th score; take 4 sigma more
    const float mu = (float)k * (float)kSamples / (float)n;
    int rank = (int)(mu + 4.f * sqrtf(mu)) + 2;
    if (rank > kSamples) rank = kSamples;
    int above_s;
    tau = select_kth<2>(samples, kSamples, rank, hist, warp_buf, sel, &above_s);
  }

  // ---- 2. one pass: warp-segmented ordered compaction of keys > tau --------
  // A warp reads kStreamUnroll x 128 consecutive scores per iteration, all
  // loads issued before the first compaction, so several of its loads are in
  // flight at once; the 128-score groups are then compacted in index order.
  // Scores equal to tau are only counted: when the k-th score is tau itself
  // (rows with many exact ties) the stored scores plus the lowest-indexed ties
  // are the answer, and the ties need not occupy the candidate buffer.
  if (threadIdx.x == 0) flag_overflow = 0;
  const int seg = ((n + kTopkWarps - 1) / kTopkWarps + 127) & ~127;   // multiple of 128 elements
  const int w_begin = wid * seg;
  const int w_end = min(n, w_begin + seg);
  int wcount = 0, weq = 0;
  bool overflow = false;
  const uint32_t my_key_s = smem_u32(cand_key + wid * kWarpCap);
  const uint32_t my_idx_s = smem_u32(cand_idx + wid * kWarpCap);
  // For a finite score x, order_key(x) > tau exactly when x > key_value(tau),
  // and the keys are equal exactly when x == key_value(tau) (also for -0 and
  // +0), so the pass compares the floats themselves and keeps their raw bits;
  // the keys are formed for the candidates only, when the warp regions are
  // merged.  tau == 0 (no sampling) keeps every score.
  const bool keep_all = tau == 0u;
  const float tau_f = keep_all ? 0.f : key_value(tau);
  for (int base = w_begin; base < w_end && !overflow; base += 128 * kStreamUnroll) {
    float xx[kStreamUnroll][4];
#pragma unroll
    for (int u = 0; u < kStreamUnroll; ++u) {
      const int e = base + u * 128 + 4 * lane;
      if (vec4 && e + 3 < w_end) {
        const float4 f = __ldg(reinterpret_cast<const float4*>(row + e));
        xx[u][0] = f.x;
        xx[u][1] = f.y;
        xx[u][2] = f.z;
        xx[u][3] = f.w;
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) xx[u][j] = (e + j < w_end) ? __ldg(row + e + j) : 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < kStreamUnroll; ++u) {
      const int e = base + u * 128 + 4 * lane;
      bool f[4];
      int c = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        f[j] = (e + j < w_end) && (keep_all || xx[u][j] > tau_f);
        weq += (e + j < w_end) && !keep_all && xx[u][j] == tau_f;
        c += f[j];
      }
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int tot = __shfl_sync(0xffffffffu, incl, 31);
      if (overflow || wcount + tot > kWarpCap) {   // warp-uniform
        overflow = true;
        continue;
      }
      int pos = wcount + incl - c;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        st_shared_u32_if(my_key_s + 4u * pos, __float_as_uint(xx[u][j]), f[j]);   // raw bits
        st_shared_u32_if(my_idx_s + 4u * pos, (uint32_t)(e + j), f[j]);
        pos += f[j];
      }
      wcount += tot;
    }
  }
  weq = __reduce_add_sync(0xffffffffu, weq);
  if (lane == 0) {
    warp_cnt[wid] = wcount;
    warp_eq[wid] = weq;
    if (overflow) flag_overflow = 1;
  }
  __syncthreads();
  int m = 0, eq_total = 0;
  for (int w = 0; w < kTopkWarps; ++w) {
    m += warp_cnt[w];
    eq_total += warp_eq[w];
  }
  // fast: the k-th score is above tau, so every selected score is stored;
  // tie: fewer than k scores are above tau but with the ties at tau there are
  // enough, so the k-th score is tau itself (k <= kCandCap holds for k <= 1024)
  const bool fast = !flag_overflow && m >= k;
  const bool tie = !flag_overflow && !fast && m + eq_total >= k && k <= kCandCap;
  if (fast || tie) {
    // close the gaps between the warp regions (in warp order = index order):
    // every thread reads its compacted positions i = tid + j*threads from
    // their regions into registers, then, after one barrier, writes them
    int pre[kTopkWarps];
    {
      int acc = 0;
#pragma unroll
      for (int w = 0; w < kTopkWarps; ++w) {
        pre[w] = acc;
        acc += warp_cnt[w];
      }
    }
    // in passes of J*threads positions; a candidate's source position is
    // never below its destination, so a later pass reads nothing an earlier
    // pass wrote
    constexpr int J = 8;
    for (int pass0 = 0; pass0 < m; pass0 += J * kTopkThreads) {
      uint32_t kv[J];
      int32_t iv[J];
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const int i = pass0 + threadIdx.x + j * kTopkThreads;
        kv[j] = 0u;
        iv[j] = 0;
        if (pass0 + j * kTopkThreads >= m) break;   // block-uniform
        if (i < m) {
          int src = i;
#pragma unroll
          for (int w = 1; w < kTopkWarps; ++w)
            if (i >= pre[w]) src = i - pre[w] + w * kWarpCap;
          kv[j] = order_key(__uint_as_float(cand_key[src]));   // raw bits -> key
          iv[j] = cand_idx[src];
        }
      }
      __syncthreads();
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const int i = pass0 + threadIdx.x + j * kTopkThreads;
        if (pass0 + j * kTopkThreads >= m) break;   // block-uniform
        if (i < m) {
          cand_key[i] = kv[j];
          cand_idx[i] = iv[j];
        }
      }
      __syncthreads();
    }
    if (fast) {
      select_from_candidates(cand_key, cand_idx, m, k, hist, warp_buf, sel, out);
      return;
    }
    // tie: all m stored scores are taken, plus the need_eq lowest-indexed
    // scores equal to tau.  Each warp owning some of those ties collects them
    // from its own segment (warp order is index order) into the buffer after
    // the stored ones, then the two index-sorted lists are merged by rank.
    const int need_eq = k - m;
    int eq_before = 0;
    for (int w = 0; w < wid; ++w) eq_before += warp_eq[w];
    const int quota = max(0, min(warp_eq[wid], need_eq - eq_before));
    int32_t* eq_list = cand_idx + m;
    const uint32_t lanes_below = (1u << lane) - 1u;
    int got = 0;
    for (int base = w_begin; base < w_end && got < quota; base += 32 * kTieUnroll) {
      float xq[kTieUnroll];
#pragma unroll
      for (int u = 0; u < kTieUnroll; ++u) {
        const int e = base + u * 32 + lane;
        xq[u] = e < w_end ? __ldg(row + e) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kTieUnroll; ++u) {
        const int e = base + u * 32 + lane;
        const bool q = e < w_end && xq[u] == tau_f;
        const uint32_t ball = __ballot_sync(0xffffffffu, q);
        const int rnk = got + __popc(ball & lanes_below);
        if (q && rnk < quota) eq_list[eq_before + rnk] = e;
        got += __popc(ball);
      }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < k; i += kTopkThreads) {
      const bool stored = i < m;
      const int32_t v = stored ? cand_idx[i] : eq_list[i - m];
      const int32_t* other = stored ? eq_list : cand_idx;
      int lo = 0, hi = stored ? need_eq : m;   // entries of the other list below v
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (other[mid] < v)
          lo = mid + 1;
        else
          hi = mid;
      }
      out[(stored ? i : i - m) + lo] = v;
    }
    return;
  }

  // ---- fallback: histogram pass, then the threshold bin and above ---------
  const int n_round = (n + 4 * kTopkThreads - 1) / (4 * kTopkThreads) * (4 * kTopkThreads);
  auto load4 = [&](int base, uint32_t (&kk)[4]) {
    if (vec4 && base + 3 < n) {
      const float4 f = __ldg(reinterpret_cast<const float4*>(row + base));
      kk[0] = order_key(f.x);
      kk[1] = order_key(f.y);
      kk[2] = order_key(f.z);
      kk[3] = order_key(f.w);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) kk[j] = (base + j < n) ? order_key(__ldg(row + base + j)) : 0u;
    }
  };
  zero_hist<2048>(hist);
  __syncthreads();
  for (int base = threadIdx.x * 4; base < n_round; base += 4 * kTopkThreads) {
    uint32_t kk[4];
    load4(base, kk);
#pragma unroll
    for (int j = 0; j < 4; ++j) hist_add(hist, base + j < n ? (int)(kk[j] >> 21) : -1);
  }
  __syncthreads();
  find_bin<2048>(hist, k, warp_buf, sel);
  const uint32_t b0 = (uint32_t)sel[0];
  const int n_cand = sel[1] + hist[b0];
  __syncthreads();
  if (n_cand <= kCandCap) {
    int written = 0;
    for (int base = threadIdx.x * 4; base < n_round; base += 4 * kTopkThreads) {
      uint32_t kk[4];
      load4(base, kk);
      bool f[4];
      int cnt = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        f[j] = (base + j < n) && (kk[j] >> 21) >= b0;
        cnt += f[j];
      }
      int tot;
      int pos = written + block_excl_scan(cnt, warp_buf, &tot);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        st_shared_u32_if(smem_u32(cand_key) + 4u * pos, kk[j], f[j]);
        st_shared_u32_if(smem_u32(cand_idx) + 4u * pos, (uint32_t)(base + j), f[j]);
        pos += f[j];
      }
      written += tot;
    }
    __syncthreads();
    select_from_candidates(cand_key, cand_idx, n_cand, k, hist, warp_buf, sel, out);
    return;
  }
  // tie-heavy: rounds 1 and 2 over the row, then the ordered selection over the row
  const int need1 = k - sel[1];
  zero_hist<2048>(hist);
  __syncthreads();
  for (int base = threadIdx.x * 4; base < n_round; base += 4 * kTopkThreads) {
    uint32_t kk[4];
    load4(base, kk);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      hist_add(hist, (base + j < n && (kk[j] >> 21) == b0) ? (int)((kk[j] >> 10) & 0x7FFu) : -1);
  }
  __syncthreads();
  find_bin<2048>(hist, need1, warp_buf, sel);
  const uint32_t pre1 = (b0 << 11) | (uint32_t)sel[0];
  const int need2 = need1 - sel[1];
  zero_hist<1024>(hist);
  __syncthreads();
  for (int base = threadIdx.x * 4; base < n_round; base += 4 * kTopkThreads) {
    uint32_t kk[4];
    load4(base, kk);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      hist_add(hist, (base + j < n && (kk[j] >> 10) == pre1) ? (int)(kk[j] & 0x3FFu) : -1);
  }
  __syncthreads();
  find_bin<1024>(hist, need2, warp_buf, sel);
  const uint32_t T = (pre1 << 10) | (uint32_t)sel[0];
  const int need_eq = need2 - sel[1];
  int eq_seen = 0, taken = 0;
  for (int base = threadIdx.x * 4; base < n_round && taken < k; base += 4 * kTopkThreads) {
    uint32_t kk[4];
    load4(base, kk);
    select_tile(kk, base, n, T, need_eq, eq_seen, taken, warp_buf, nullptr, out);
  }
}

// Four CTAs per SM (64 registers a thread).  Five fit in shared memory
// (about 45 KB each), but the 48-register cap that five need spills, and four
// measured faster on long rows (1M tokens: -20%) and no slower at 128k.
__global__ void __launch_bounds__(kTopkThreads, 4) topk_kernel(const float* __restrict__ scores, int64_t P, int k,
                                                            int64_t q_begin, int64_t q_count,
                                                            int32_t* __restrict__ idx) {
  // Longer rows (later queries) first.
  topk_row(scores, P, k, q_begin, q_count - 1 - (int64_t)blockIdx.x, idx);
}

// The same selection for the rows listed in rlist[0 .. *rlist_n) (the rows
// the fused indexer + top-k could not settle from their candidates), by a
// persistent grid; with an empty list every CTA returns at once.
__global__ void __launch_bounds__(kTopkThreads, 4) topk_list_kernel(const float* __restrict__ scores, int64_t P,
                                                                 int k, int64_t q_begin,
                                                                 const int32_t* __restrict__ rlist,
                                                                 const uint32_t* __restrict__ rlist_n,
                                                                 int32_t* __restrict__ idx) {
  const uint32_t n = *rlist_n;
  for (uint32_t b = blockIdx.x; b < n; b += gridDim.x) {
    topk_row(scores, P, k, q_begin, rlist[b], idx);
    __syncthreads();   // the shared arrays are reused by the next row
  }
}

cudaError_t launch_topk(int64_t L, int k, const float* scores, int64_t q_begin, int64_t q_count, int32_t* idx,
                        cudaStream_t s) {
  const int64_t P = L / 4;
  topk_kernel<<<(unsigned)q_count, kTopkThreads, 0, s>>>(scores, P, k, q_begin, q_count, idx);
  return cudaGetLastError();
}

cudaError_t launch_topk_list(int64_t L, int k, const float* scores, int64_t q_begin, int64_t max_rows,
                             const int32_t* rlist, const uint32_t* rlist_n, int32_t* idx, cudaStream_t s) {
  const int64_t P = L / 4;
  int64_t grid = (int64_t)device_sm_count() * 4;
  if (grid > max_rows) grid = max_rows;
  if (grid < 1) grid = 1;
  topk_list_kernel<<<(unsigned)grid, kTopkThreads, 0, s>>>(scores, P, k, q_begin, rlist, rlist_n, idx);
  return cudaGetLastError();
}

}  // namespace dsa
