// fused_topk.cu -- indexer scores and top-k selection without the score block.
//
// Page "SkyRL extends GLM-5.3-Flash training context to 1 million tokens",
// section "Model and bottleneck" (the indexer scores every causal pool for
// every query: the layer's quadratic part) and section "1. DSA truly sparse"
// (the indexer is scored in query chunks and hands only int32 pool indices to
// the sparse kernel).  The result is the selection of the unfused pair
// (indexer_score then topk) bit for bit; only the route differs.  Route 1
// (the default) is that pair, with the score block in the workspace.  Route 0
// never writes the score block:
//
//   1. sampled scores: the tensor-core indexer scores every kSampleStride-th
//      pool (a strided view of kpool, 1/32 of the work) into a small block;
//   2. thresholds (one warp per row): tau = the lower edge of the 24-bit key
//      bin of the r-th largest sample, r = mu + 4 sqrt(mu) + 2 with
//      mu = k * n_samples / elig(t) the expected number of samples at or
//      above the k-th score, so that tau lies below the k-th score with high
//      probability while about r * kSampleStride scores pass it.  Rows with
//      at most kKeepAll eligible pools keep every score (tau = -inf); rows
//      with elig(t) <= k need no candidates (tau = +inf);
//   3. the indexer again, every pool, with an epilogue that appends each
//      eligible score >= tau to the row's candidates (no score block).  Each
//      epilogue warp owns a sub-list per (row, 2048-pool segment, lane
//      quarter) and fills it with a warp-uniform running length, so no
//      atomics are needed: a row's fused_cand_stride(P) entries are split
//      evenly over its 4 * nseg(t) sub-lists;
//   4. selection (one warp per row): if no sub-list overflowed and the row has
//      at least k candidates, every score at or above the k-th score is among
//      them (tau <= k-th score), so the exact k-th score and the
//      lowest-indexed ties at it are found among the candidates by radix
//      select, and the k pools are written in ascending order.  Otherwise the
//      row and its 32-query block are put on fallback lists;
//   5. fallback: the indexer writes the full score rows of the listed blocks,
//      and the unfused top-k selects the listed rows from them.  Both launches
//      read their list's length on the device and do nothing when it is empty.
//
// The candidate order depends on atomics; the selection does not (it depends
// only on the set of candidates), so the output is bitwise reproducible.
#include "common.cuh"
#include "launch.h"

namespace dsa {

constexpr int kSampleStride = 32;   // the sampled pass scores pools 0, 32, 64, ...
constexpr int kKeepAll = 2048;      // rows of at most this many eligible pools keep every score
constexpr int kFkWarps = 8;         // rows (one per warp) per CTA of the threshold and select kernels
constexpr int kMaxSel = 1024;       // largest k

// A keep-all row has one segment: each of its 4 sub-lists must hold the
// 512 pools of a lane quarter.
static_assert(kKeepAll <= kSegPools && 4096 / 4 >= kSegPools / 4, "a keep-all row must fit its sub-lists");

// Scanning a per-warp 256-bin histogram from bin 255 down, the bin where the
// running count reaches `need` (1 <= need <= total), and the count strictly
// above it.  Lane L owns bins 255-8L .. 248-8L.
__device__ __forceinline__ void warp_find_digit(const int* hist, int need, int& digit, int& above) {
  const int lane = threadIdx.x & 31;
  int h[8], sum = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    h[i] = hist[255 - 8 * lane - i];
    sum += h[i];
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const int excl = incl - sum;
  const bool mine = excl < need && incl >= need;
  int d = 0, a = 0;
  if (mine) {
    int cum = excl;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (cum + h[i] >= need) {
        d = 255 - 8 * lane - i;
        a = cum;
        break;
      }
      cum += h[i];
    }
  }
  const uint32_t b = __ballot_sync(0xffffffffu, mine);
  const int src = b ? __ffs(b) - 1 : 31;   // b == 0 only if need exceeds the total
  digit = __shfl_sync(0xffffffffu, d, src);
  above = __shfl_sync(0xffffffffu, a, src);
}

// hist[bin] += 1 when bin >= 0.
__device__ __forceinline__ void warp_hist_add(int* hist, int bin) {
  if (bin >= 0) atomicAdd(&hist[bin], 1);
}

__device__ __forceinline__ void warp_zero_hist(int* hist) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < 8; ++i) hist[lane + 32 * i] = 0;
  __syncwarp();
}

// Thresholds, candidate counters and fallback flags of one chunk.
__global__ void __launch_bounds__(32 * kFkWarps) fused_tau_kernel(const float* __restrict__ samples, int64_t P_s,
                                                                  int k, int64_t q_begin, int64_t q_count,
                                                                  float* __restrict__ tau,
                                                                  uint32_t* __restrict__ bflag,
                                                                  uint32_t* __restrict__ counters) {
  __shared__ int hist_all[kFkWarps][256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (blockIdx.x == 0 && threadIdx.x < 2) counters[threadIdx.x] = 0u;   // fallback list lengths
  const int64_t r = (int64_t)blockIdx.x * kFkWarps + warp;
  if (r >= q_count) return;
  int* hist = hist_all[warp];
  if (lane == 0 && (r & 31) == 0) bflag[r >> 5] = 0u;
  const int64_t e = elig(q_begin + r);
  float th;
  if (e <= k) {
    th = INFINITY;             // every eligible pool is selected; no candidates needed
  } else if (e <= kKeepAll) {
    th = -INFINITY;            // every eligible score is a candidate
  } else {
    const int ns = (int)((e + kSampleStride - 1) / kSampleStride);
    const float mu = (float)k * (float)ns / (float)e;
    int rank = (int)(mu + 4.f * sqrtf(mu)) + 2;
    if (rank > ns) rank = ns;
    const float* row = samples + r * P_s;
    uint32_t prefix = 0;
    int need = rank;
    for (int round = 0; round < 3; ++round) {
      const int shift = 24 - 8 * round;
      warp_zero_hist(hist);
      for (int j = lane; j < ns; j += 32) {
        const uint32_t key = order_key(__ldg(row + j));
        if (round == 0 || (key >> (shift + 8)) == prefix) warp_hist_add(hist, (int)((key >> shift) & 255u));
      }
      __syncwarp();
      int digit, above;
      warp_find_digit(hist, need, digit, above);
      prefix = (prefix << 8) | (uint32_t)digit;
      need -= above;
      __syncwarp();
    }
    th = key_value(prefix << 8);   // the lower edge of the r-th sample's 24-bit bin
  }
  if (lane == 0) tau[r] = th;
}

// Calls f(key, pool) for every candidate of a row held in its nsub
// sub-lists (lengths len[s], capacity cap each); key = order_key(score).
// With many sub-lists each lane walks whole sub-lists; with few, the lanes
// share each sub-list.  A lane meets the entries in the same order on every
// call.
template <typename F>
__device__ __forceinline__ void for_each_listed(const uint2* __restrict__ cr, const uint32_t* __restrict__ len,
                                                int nsub, int cap, F f) {
  const int lane = threadIdx.x & 31;
  if (nsub >= 32) {
    for (int sb = lane; sb < nsub; sb += 32) {
      const int n = (int)__ldg(len + sb);
      const uint2* e = cr + (int64_t)sb * cap;
      for (int i = 0; i < n; ++i) {
        const uint2 v = __ldg(e + i);
        f(order_key(__uint_as_float(v.x)), v.y);
      }
    }
  } else {
    for (int sb = 0; sb < nsub; ++sb) {
      const int n = (int)__ldg(len + sb);
      const uint2* e = cr + (int64_t)sb * cap;
      for (int i = lane; i < n; i += 32) {
        const uint2 v = __ldg(e + i);
        f(order_key(__uint_as_float(v.x)), v.y);
      }
    }
  }
}

// The selection proper.  `each` enumerates the c candidates, calling
// f(key, pool) for each (key = order_key(score)); keys_and/keys_or are the
// AND and OR of all their keys.  The k-th largest key K is found by 8-bit
// radix rounds that start at the highest bit where the keys differ (the bits
// above it are shared by every candidate and need no round), the ties at K by
// rounds over the tied pools from the low end (bins reversed).  The k
// selected pools are then compacted into sel, sorted ascending (bitonic, in
// shared memory) and written to out.
template <typename Each>
__device__ __forceinline__ void select_core(Each each, uint32_t keys_and, uint32_t keys_or, int c, int k,
                                            int* hist, int32_t* sel, int32_t* out) {
  const int lane = threadIdx.x & 31;
  const uint32_t diff = keys_and ^ keys_or;
  uint32_t K = keys_or;   // every candidate has this key when they all agree
  int need = k, n_eq = c;
  if (diff != 0u) {
    // rounds of 8-bit digits ending at bit 0, as few as cover the highest
    // differing bit; the bits above the first digit are shared by all keys
    const int top = 31 - __clz(diff);
    const int rounds = (top + 8) / 8;
    K = rounds >= 4 ? 0u : (keys_or >> (8 * rounds));
    for (int rd = 0; rd < rounds; ++rd) {
      const int sh = 8 * (rounds - 1 - rd);
      const uint32_t pre = K;
      warp_zero_hist(hist);
      each([&](uint32_t key, uint32_t) {
        if (sh + 8 >= 32 || (key >> (sh + 8)) == pre) warp_hist_add(hist, (int)((key >> sh) & 255u));
      });
      __syncwarp();
      int digit, above;
      warp_find_digit(hist, need, digit, above);
      K = (K << 8) | (uint32_t)digit;
      need -= above;
      n_eq = hist[digit];
      __syncwarp();
    }
  }
  uint32_t Ip = 0xFFFFFFFFu;
  if (need < n_eq) {
    uint32_t pre = 0;
    int nd = need;
    for (int round = 0; round < 4; ++round) {
      const int psh = 24 - 8 * round;
      warp_zero_hist(hist);
      each([&](uint32_t key, uint32_t pool) {
        if (key == K && (round == 0 || (pool >> (psh + 8)) == pre))
          warp_hist_add(hist, (int)(255u - ((pool >> psh) & 255u)));
      });
      __syncwarp();
      int digit, above;
      warp_find_digit(hist, nd, digit, above);
      pre = (pre << 8) | (uint32_t)(255 - digit);
      nd -= above;
      __syncwarp();
    }
    Ip = pre;
  }
  int mine = 0;
  each([&](uint32_t key, uint32_t pool) { mine += key > K || (key == K && pool <= Ip); });
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  int pos = incl - mine;
  each([&](uint32_t key, uint32_t pool) {
    if (key > K || (key == K && pool <= Ip)) {
      if (pos < kMaxSel) sel[pos] = (int32_t)pool;
      ++pos;
    }
  });
  int n = 32;
  while (n < k) n <<= 1;
  for (int i = k + lane; i < n; i += 32) sel[i] = 0x7FFFFFFF;
  __syncwarp();
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = lane; i < n / 2; i += 32) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const int32_t x = sel[lo], y = sel[hi];
        if ((x > y) == ((lo & size) == 0)) {
          sel[lo] = y;
          sel[hi] = x;
        }
      }
      __syncwarp();
    }
  }
  for (int i = lane; i < k; i += 32) out[i] = sel[i];
}

constexpr int kSelWarps = 4;        // rows (one per warp) per CTA of the select kernel
constexpr int kStage = 2048;        // candidates a warp stages in shared memory

struct SelWarpSmem {
  uint32_t key[kStage];
  uint32_t pool[kStage];
  int hist[256];
  int32_t sel[kMaxSel];
};

// Selection from the candidate sub-lists (one warp per row).  A row's
// candidates are first copied into the warp's shared memory (keys formed
// once), so the radix rounds run on shared memory; rows with more than
// kStage candidates work from the sub-lists directly.
__global__ void __launch_bounds__(32 * kSelWarps) fused_select_kernel(
    const uint2* __restrict__ cand, const uint32_t* __restrict__ cntq, int64_t cand_stride, int64_t nseg_max, int k,
    int64_t q_begin, int64_t q_count, int32_t* __restrict__ idx, int32_t* __restrict__ rlist,
    int32_t* __restrict__ blist, uint32_t* __restrict__ bflag, uint32_t* __restrict__ counters) {
  extern __shared__ __align__(16) unsigned char sel_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * kSelWarps + warp;
  if (r >= q_count) return;
  SelWarpSmem& sm = reinterpret_cast<SelWarpSmem*>(sel_smem)[warp];
  const int64_t t = q_begin + r;
  const int64_t e = elig(t);
  int32_t* out = idx + t * (int64_t)k;
  if (e <= k) {
    for (int i = lane; i < k; i += 32) out[i] = i < e ? i : -1;
    return;
  }
  const int nseg = (int)(e > kSegPools ? (e + kSegPools - 1) / kSegPools : 1);
  const int nsub = 4 * nseg;
  const int cap = (int)(cand_stride / nsub);
  const uint32_t* len = cntq + r * nseg_max * 4;
  // lengths: this lane's share (whole sub-lists when there are many)
  int total = 0, my_total = 0;
  bool overflow = false;
  for (int sb = lane; sb < nsub; sb += 32) {
    const int n = (int)__ldg(len + sb);
    my_total += n;
    overflow |= n > cap;
  }
  total = __reduce_add_sync(0xffffffffu, my_total);
  overflow = __any_sync(0xffffffffu, overflow);
  if (overflow || total < k) {
    // tau missed or a sub-list overflowed: the fallback settles this row
    if (lane == 0) {
      rlist[atomicAdd(&counters[0], 1u)] = (int32_t)r;
      const int32_t b = (int32_t)(r >> 5);
      if (atomicExch(&bflag[b], 1u) == 0u) blist[atomicAdd(&counters[1], 1u)] = b;
    }
    return;
  }
  const uint2* cr = cand + r * cand_stride;
  if (total > kStage) {
    uint32_t kand = 0xFFFFFFFFu, kor = 0u;
    for_each_listed(cr, len, nsub, cap, [&](uint32_t key, uint32_t) {
      kand &= key;
      kor |= key;
    });
    kand = __reduce_and_sync(0xffffffffu, kand);
    kor = __reduce_or_sync(0xffffffffu, kor);
    select_core([&](auto f) { for_each_listed(cr, len, nsub, cap, f); }, kand, kor, total, k, sm.hist, sm.sel, out);
    return;
  }
  // stage the candidates: positions from a warp scan of the per-lane totals
  // (many sub-lists) or a running offset (few)
  if (nsub >= 32) {
    int incl = my_total;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int pos = incl - my_total;
    for (int sb = lane; sb < nsub; sb += 32) {
      const int n = (int)__ldg(len + sb);
      const uint2* src = cr + (int64_t)sb * cap;
      int i = 0;
      for (; i + 4 <= n; i += 4) {   // four loads in flight
        uint2 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = __ldg(src + i + u);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          sm.key[pos + u] = order_key(__uint_as_float(v[u].x));
          sm.pool[pos + u] = v[u].y;
        }
        pos += 4;
      }
      for (; i < n; ++i, ++pos) {
        const uint2 v = __ldg(src + i);
        sm.key[pos] = order_key(__uint_as_float(v.x));
        sm.pool[pos] = v.y;
      }
    }
  } else {
    int base = 0;
    for (int sb = 0; sb < nsub; ++sb) {
      const int n = (int)__ldg(len + sb);
      const uint2* src = cr + (int64_t)sb * cap;
      for (int i = lane; i < n; i += 32) {
        const uint2 v = __ldg(src + i);
        sm.key[base + i] = order_key(__uint_as_float(v.x));
        sm.pool[base + i] = v.y;
      }
      base += n;
    }
  }
  __syncwarp();
  const int c = total;
  uint32_t kand = 0xFFFFFFFFu, kor = 0u;
  for (int i = lane; i < c; i += 32) {
    kand &= sm.key[i];
    kor |= sm.key[i];
  }
  kand = __reduce_and_sync(0xffffffffu, kand);
  kor = __reduce_or_sync(0xffffffffu, kor);
  select_core(
      [&](auto f) {
        for (int i = lane; i < c; i += 32) f(sm.key[i], sm.pool[i]);
      },
      kand, kor, c, k, sm.hist, sm.sel, out);
}

// --------------------------------------------------------------------- host
namespace {
size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

struct FusedWs {
  float* scores;        // [C, P]  fallback score rows
  float* samples;       // [C, P_s]
  uint2* cand;          // [C, fused_cand_stride(P)] candidate sub-lists
  uint32_t* cntq;       // [C, fused_nseg_max(P), 4] sub-list lengths
  float* tau;           // [C]
  int32_t* rlist;       // [C]
  int32_t* blist;       // [ceil(C/32)]
  uint32_t* bflag;      // [ceil(C/32)]
  uint32_t* counters;   // [2]: rlist and blist lengths
  size_t bytes;
};

FusedWs carve(void* base, int64_t C, int64_t P) {
  FusedWs f{};
  const int64_t P_s = (P + kSampleStride - 1) / kSampleStride;
  const int64_t nb = (C + 31) / 32;
  char* p = static_cast<char*>(base);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* q = p ? p + off : nullptr;
    off += align256(bytes);
    return q;
  };
  f.scores = reinterpret_cast<float*>(take((size_t)C * P * 4));
  f.samples = reinterpret_cast<float*>(take((size_t)C * P_s * 4));
  f.cand = reinterpret_cast<uint2*>(take((size_t)C * fused_cand_stride(P) * 8));
  f.cntq = reinterpret_cast<uint32_t*>(take((size_t)C * fused_nseg_max(P) * 4 * 4));
  f.tau = reinterpret_cast<float*>(take((size_t)C * 4));
  f.rlist = reinterpret_cast<int32_t*>(take((size_t)C * 4));
  f.blist = reinterpret_cast<int32_t*>(take((size_t)nb * 4));
  f.bflag = reinterpret_cast<uint32_t*>(take((size_t)nb * 4));
  f.counters = reinterpret_cast<uint32_t*>(take(16));
  f.bytes = off;
  return f;
}
}  // namespace

size_t fused_indexer_topk_ws_bytes(int64_t L, int64_t rows) { return carve(nullptr, rows, L / 4).bytes; }

cudaError_t launch_indexer_topk_bf16(int64_t L, int Hi, int di, int k, const void* q_idx, const void* kpool,
                                     const float* w, int64_t q_begin, int64_t q_count, int32_t* idx, void* ws,
                                     int route, cudaStream_t s) {
  const int64_t P = L / 4;
  const int64_t P_s = (P + kSampleStride - 1) / kSampleStride;
  const FusedWs f = carve(ws, q_count, P);
  if (route == 1) {
    // the score block and the row-wise top-k (the unfused pair)
    IdxArgs a{};
    a.w = w;
    a.scores = f.scores;
    a.P_cols = P;
    a.q_begin = q_begin;
    a.q_count = q_count;
    a.col_stride = 1;
    cudaError_t e = launch_indexer_tc_bf16_ex(L, Hi, di, q_idx, kpool, a, false, s);
    if (e != cudaSuccess) return e;
    return launch_topk(L, k, f.scores, q_begin, q_count, idx, s);
  }
  const int64_t t_last = q_begin + q_count - 1;
  cudaError_t e = cudaSuccess;
  // 1. sampled scores (only rows with more than kKeepAll eligible pools use them)
  if (((t_last + 1) >> 2) > kKeepAll) {
    IdxArgs a{};
    a.w = w;
    a.scores = f.samples;
    a.P_cols = P_s;
    a.q_begin = q_begin;
    a.q_count = q_count;
    a.col_stride = kSampleStride;
    if ((e = launch_indexer_tc_bf16_ex(L, Hi, di, q_idx, kpool, a, false, s)) != cudaSuccess) return e;
  }
  // 2. thresholds
  const unsigned rows_grid = (unsigned)((q_count + kFkWarps - 1) / kFkWarps);
  fused_tau_kernel<<<rows_grid, 32 * kFkWarps, 0, s>>>(f.samples, P_s, k, q_begin, q_count, f.tau, f.bflag,
                                                       f.counters);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // 3. candidates
  {
    IdxArgs a{};
    a.w = w;
    a.P_cols = P;
    a.q_begin = q_begin;
    a.q_count = q_count;
    a.col_stride = 1;
    a.tau = f.tau;
    a.cand = f.cand;
    a.cntq = f.cntq;
    a.cand_stride = fused_cand_stride(P);
    a.nseg_max = fused_nseg_max(P);
    if ((e = launch_indexer_tc_bf16_ex(L, Hi, di, q_idx, kpool, a, true, s)) != cudaSuccess) return e;
  }
  // 4. selection
  {
    constexpr int smem = kSelWarps * (int)sizeof(SelWarpSmem);
    if ((e = cudaFuncSetAttribute(fused_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) !=
        cudaSuccess)
      return e;
    const unsigned sel_grid = (unsigned)((q_count + kSelWarps - 1) / kSelWarps);
    fused_select_kernel<<<sel_grid, 32 * kSelWarps, smem, s>>>(f.cand, f.cntq, fused_cand_stride(P),
                                                              fused_nseg_max(P), k, q_begin, q_count, idx, f.rlist,
                                                              f.blist, f.bflag, f.counters);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // 5. fallback for the listed rows (nothing to do when the lists are empty)
  {
    IdxArgs a{};
    a.w = w;
    a.scores = f.scores;
    a.P_cols = P;
    a.q_begin = q_begin;
    a.q_count = q_count;
    a.col_stride = 1;
    a.blist = f.blist;
    a.blist_n = f.counters + 1;
    if ((e = launch_indexer_tc_bf16_ex(L, Hi, di, q_idx, kpool, a, false, s)) != cudaSuccess) return e;
  }
  return launch_topk_list(L, k, f.scores, q_begin, q_count, f.rlist, f.counters, idx, s);
}

}  // namespace dsa
