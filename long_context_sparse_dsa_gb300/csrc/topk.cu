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
// decide order), so it is bitwise reproducible.
//
// One CTA of kTopkThreads threads per row.  Global traffic is two passes
// over the row: pass 1 builds the top-11-bit histogram; pass 2 copies every
// key in the threshold bin or above (at most k-1 + that bin) with its index,
// in index order, into shared memory; the remaining rounds and the selection
// run there.  Rows up to kRowCap scores are also staged in shared memory in
// pass 1, so pass 2 reads SMEM.  Tie-heavy rows whose threshold bin overflows
// the candidate buffer fall back to rounds and selection over the row.
#include "common.cuh"
#include "launch.h"

namespace dsa {

constexpr int kTopkThreads = 512;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kRowCap = 12288;   // scores staged in SMEM (48 KB)
constexpr int kCandCap = 6144;   // candidate keys + indices kept in SMEM (48 KB)

__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t u = __float_as_uint(x);
  if (u == 0x80000000u) u = 0u;  // -0 ties with +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

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

// Histogram add with warp aggregation (many equal keys in tie-heavy rows).
__device__ __forceinline__ void hist_add(int* hist, int bin) {
  const unsigned peers = __match_any_sync(0xffffffffu, bin);
  const int leader = __ffs(peers) - 1;
  if ((int)(threadIdx.x & 31) == leader && bin >= 0) atomicAdd(&hist[bin], __popc(peers));
}

// Find, scanning bins from the top, the bin where the running count reaches
// `need`.  Writes the bin and the count strictly above it to sel[0], sel[1].
__device__ __forceinline__ void find_bin(const int* hist, int nbins, int need, int* warp_buf, int* sel) {
  const int per = (nbins + kTopkThreads - 1) / kTopkThreads;  // 4 or 2
  int local = 0;
  for (int j = 0; j < per; ++j) {
    const int b = nbins - 1 - (threadIdx.x * per + j);
    if (b >= 0) local += hist[b];
  }
  int total;
  int cum = block_excl_scan(local, warp_buf, &total);
  for (int j = 0; j < per; ++j) {
    const int b = nbins - 1 - (threadIdx.x * per + j);
    if (b < 0) break;
    const int h = hist[b];
    if (cum < need && cum + h >= need) {
      sel[0] = b;
      sel[1] = cum;
    }
    cum += h;
  }
  __syncthreads();
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
  for (int j = 0; j < 4; ++j)
    if (take[j]) out[pos++] = ids ? ids[base + j] : base + j;
  eq_seen += eq_total;
  taken += take_total;
}

template <bool STAGE>
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const float* __restrict__ scores, int64_t P, int k,
                                                            int64_t q_begin, int64_t q_count,
                                                            int32_t* __restrict__ idx) {
  extern __shared__ __align__(16) unsigned char topk_smem[];
  int* hist = reinterpret_cast<int*>(topk_smem);                     // [2048]
  int* warp_buf = hist + 2048;                                       // [32]
  int* sel = warp_buf + 32;                                          // [4]
  uint32_t* cand_key = reinterpret_cast<uint32_t*>(sel + 4);         // [kCandCap]
  int32_t* cand_idx = reinterpret_cast<int32_t*>(cand_key + kCandCap);  // [kCandCap]
  uint32_t* row_keys = reinterpret_cast<uint32_t*>(cand_idx + kCandCap);  // [kRowCap] when STAGE

  // Longer rows (later queries) first.
  const int64_t r = q_count - 1 - (int64_t)blockIdx.x;
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
  const int n_round = (n + 4 * kTopkThreads - 1) / (4 * kTopkThreads) * (4 * kTopkThreads);

  // Four consecutive keys of the row starting at `base` (0 past the end).
  auto load4 = [&](int base, uint32_t (&kk)[4]) {
    if (STAGE) {
#pragma unroll
      for (int j = 0; j < 4; ++j) kk[j] = (base + j < n) ? row_keys[base + j] : 0u;
    } else if (vec4 && base + 3 < n) {
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

  // ---- pass 1: histogram of the top 11 bits (and stage the row) -------------
  for (int b = threadIdx.x; b < 2048; b += kTopkThreads) hist[b] = 0;
  __syncthreads();
  for (int base = threadIdx.x * 4; base < n_round; base += 4 * kTopkThreads) {
    uint32_t kk[4];
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
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const bool valid = base + j < n;
      if (STAGE && valid) row_keys[base + j] = kk[j];
      hist_add(hist, valid ? (int)(kk[j] >> 21) : -1);
    }
  }
  __syncthreads();
  find_bin(hist, 2048, k, warp_buf, sel);
  const uint32_t b0 = (uint32_t)sel[0];
  const int above0 = sel[1];
  const int need1 = k - above0;
  const int n_cand = above0 + hist[b0];
  __syncthreads();

  if (n_cand <= kCandCap) {
    // ---- pass 2: ordered compaction of every key in bins >= b0 -------------
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
      for (int j = 0; j < 4; ++j)
        if (f[j]) {
          cand_key[pos] = kk[j];
          cand_idx[pos] = base + j;
          ++pos;
        }
      written += tot;
    }
    __syncthreads();
    // ---- rounds 1 and 2 on the candidates ------------------------------------
    for (int b = threadIdx.x; b < 2048; b += kTopkThreads) hist[b] = 0;
    __syncthreads();
    const int m_round = (n_cand + kTopkThreads - 1) / kTopkThreads * kTopkThreads;
    for (int i = threadIdx.x; i < m_round; i += kTopkThreads) {
      int bin = -1;
      if (i < n_cand && (cand_key[i] >> 21) == b0) bin = (int)((cand_key[i] >> 10) & 0x7FFu);
      hist_add(hist, bin);
    }
    __syncthreads();
    find_bin(hist, 2048, need1, warp_buf, sel);
    const uint32_t pre1 = (b0 << 11) | (uint32_t)sel[0];
    const int need2 = need1 - sel[1];
    for (int b = threadIdx.x; b < 1024; b += kTopkThreads) hist[b] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < m_round; i += kTopkThreads) {
      int bin = -1;
      if (i < n_cand && (cand_key[i] >> 10) == pre1) bin = (int)(cand_key[i] & 0x3FFu);
      hist_add(hist, bin);
    }
    __syncthreads();
    find_bin(hist, 1024, need2, warp_buf, sel);
    const uint32_t T = (pre1 << 10) | (uint32_t)sel[0];
    const int need_eq = need2 - sel[1];
    // ---- ordered selection over the candidates (already in index order) -----
    const int c_round = (n_cand + 4 * kTopkThreads - 1) / (4 * kTopkThreads) * (4 * kTopkThreads);
    int eq_seen = 0, taken = 0;
    for (int base = threadIdx.x * 4; base < c_round && taken < k; base += 4 * kTopkThreads) {
      uint32_t kk[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) kk[j] = (base + j < n_cand) ? cand_key[base + j] : 0u;
      select_tile(kk, base, n_cand, T, need_eq, eq_seen, taken, warp_buf, cand_idx, out);
    }
    return;
  }

  // ---- fallback (tie-heavy rows): refine over the row, select over the row --
  for (int b = threadIdx.x; b < 2048; b += kTopkThreads) hist[b] = 0;
  __syncthreads();
  for (int base = threadIdx.x * 4; base < n_round; base += 4 * kTopkThreads) {
    uint32_t kk[4];
    load4(base, kk);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      hist_add(hist, (base + j < n && (kk[j] >> 21) == b0) ? (int)((kk[j] >> 10) & 0x7FFu) : -1);
  }
  __syncthreads();
  find_bin(hist, 2048, need1, warp_buf, sel);
  const uint32_t pre1 = (b0 << 11) | (uint32_t)sel[0];
  const int need2 = need1 - sel[1];
  for (int b = threadIdx.x; b < 1024; b += kTopkThreads) hist[b] = 0;
  __syncthreads();
  for (int base = threadIdx.x * 4; base < n_round; base += 4 * kTopkThreads) {
    uint32_t kk[4];
    load4(base, kk);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      hist_add(hist, (base + j < n && (kk[j] >> 10) == pre1) ? (int)(kk[j] & 0x3FFu) : -1);
  }
  __syncthreads();
  find_bin(hist, 1024, need2, warp_buf, sel);
  const uint32_t T = (pre1 << 10) | (uint32_t)sel[0];
  const int need_eq = need2 - sel[1];
  int eq_seen = 0, taken = 0;
  for (int base = threadIdx.x * 4; base < n_round && taken < k; base += 4 * kTopkThreads) {
    uint32_t kk[4];
    load4(base, kk);
    select_tile(kk, base, n, T, need_eq, eq_seen, taken, warp_buf, nullptr, out);
  }
}

cudaError_t launch_topk(int64_t L, int k, const float* scores, int64_t q_begin, int64_t q_count, int32_t* idx,
                        cudaStream_t s) {
  const int64_t P = L / 4;
  const int64_t max_elig = (q_begin + q_count) / 4;
  const size_t base_smem = (2048 + 32 + 4) * sizeof(int) + (size_t)kCandCap * 8;
  if (max_elig <= kRowCap) {
    const size_t smem = base_smem + (size_t)kRowCap * sizeof(uint32_t);
    cudaError_t e = cudaFuncSetAttribute(topk_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    topk_kernel<true><<<(unsigned)q_count, kTopkThreads, smem, s>>>(scores, P, k, q_begin, q_count, idx);
  } else {
    cudaError_t e =
        cudaFuncSetAttribute(topk_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)base_smem);
    if (e != cudaSuccess) return e;
    topk_kernel<false><<<(unsigned)q_count, kTopkThreads, base_smem, s>>>(scores, P, k, q_begin, q_count, idx);
  }
  return cudaGetLastError();
}

}  // namespace dsa
