// gather.cuh -- the 16-key K/V gather step shared by the attention kernels.
//
// A pool's 4 K rows (and its 4 V rows) are one contiguous block of 4*D bf16
// values, so one step of a warp gathers 4 pool slots = 16 keys: 2 tensors x
// 16 rows x D/8 16-byte chunks, spread over the 32 lanes.  The shared tile is
// [16 keys][D] per tensor with the 16-byte chunk c of row r stored at chunk
// position c ^ (r & 7), which makes the ldmatrix reads conflict-free.
//
// Everything that depends only on the lane is computed once (GatherLane);
// per step a lane needs the 4 pool indices of the step (one 32-bit shuffle
// each) and issues its copies with a single address add per copy.  Keys that
// are not visible (empty slot, or tokens after t in the partial pool) are
// zero-filled.
#pragma once

#include "common.cuh"

namespace dsa {

template <int D>
struct GatherCfg {
  static constexpr int CHUNKS = D / 8;                  // 16-byte chunks per row
  static constexpr int ROW_BYTES = D * 2;
  static constexpr int TILE_BYTES = 16 * ROW_BYTES;     // 16 keys of one tensor
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;    // K tile + V tile
  static constexpr int COPIES = 2 * 16 * CHUNKS / 32;   // 16-byte copies per lane per step
  static constexpr int LANES_PER_ROW = CHUNKS;          // lanes covering one row of one tensor
  static constexpr int ROWS_PER_COPY = 32 / CHUNKS;     // rows covered by one copy instruction (2 or 4)
};

// Copy i of a lane covers: slot sig(i), tensor ten(i), row = row_base(i) + lane / CHUNKS, chunk = lane % CHUNKS.
template <int D>
struct GatherLane {
  int ch;         // 16-byte chunk within a row
  int row_lo;     // lane / CHUNKS: row offset inside the copy's row group
};

template <int D>
__device__ __forceinline__ GatherLane<D> gather_lane(int lane) {
  GatherLane<D> g;
  g.ch = lane % GatherCfg<D>::CHUNKS;
  g.row_lo = lane / GatherCfg<D>::CHUNKS;
  return g;
}

// Pool of slot `slot` for query t (slot k = the own partial pool), -1 if none.
// A pool the query may not see is recorded as a bad index and skipped.
__device__ __forceinline__ int slot_pool32(const int32_t* irow, int k, int slot, int64_t t) {
  if (slot < k) {
    const int p = __ldg(irow + slot);
    if (p < 0) return -1;
    if ((int64_t)p >= elig(t)) {
      record_error(DSA_DEV_ERR_BAD_INDEX);
      return -1;
    }
    return p;
  }
  if (slot == k && (t & 3) != 3) return (int)(t >> 2);
  return -1;
}

// The 4 pools of step `grp` for every lane (lanes 0..3 read idx, then shuffle).
__device__ __forceinline__ void step_pools(const int32_t* irow, int k, int grp, int64_t t, int lane, int (&pools)[4]) {
  const int mine = lane < 4 ? slot_pool32(irow, k, grp * 4 + lane, t) : -1;
#pragma unroll
  for (int s = 0; s < 4; ++s) pools[s] = __shfl_sync(0xffffffffu, mine, s);
}

// Number of visible tokens of slot s (4 for a selected pool, 1..3 for the
// partial pool, 0 for an empty slot).
__device__ __forceinline__ int slot_rows(int pool, int slot, int k, int64_t t) {
  if (pool < 0) return 0;
  if (slot != k) return 4;
  return (int)(t - 4 * (int64_t)pool) + 1;
}

template <int D>
__device__ __forceinline__ void gather_step16(uint32_t stage, const __nv_bfloat16* __restrict__ K,
                                              const __nv_bfloat16* __restrict__ V, const int (&pools)[4],
                                              const GatherLane<D>& gl, int64_t t, int k, int grp) {
  using C = GatherCfg<D>;
#pragma unroll
  for (int i = 0; i < C::COPIES; ++i) {
    // copy i covers rows [row0, row0 + ROWS_PER_COPY) of one (slot, tensor)
    constexpr int per_slot = 2 * 4 / C::ROWS_PER_COPY;       // copies per slot (both tensors)
    const int sig = i / per_slot;
    const int ten = (i % per_slot) / (per_slot / 2);
    const int row = (i % (per_slot / 2)) * C::ROWS_PER_COPY + gl.row_lo;
    const int p = pools[sig];
    const int nrows = slot_rows(p, grp * 4 + sig, k, t);
    const bool valid = row < nrows;
    const __nv_bfloat16* base = ten ? V : K;
    const __nv_bfloat16* src = base + (valid ? ((int64_t)(4 * p + row) * D + gl.ch * 8) : 0);
    const int key = sig * 4 + row;
    const uint32_t dst = stage + ten * C::TILE_BYTES + key * C::ROW_BYTES + ((gl.ch ^ (key & 7)) << 4);
    cp_async16(dst, src, valid ? 16u : 0u);
  }
}

}  // namespace dsa
