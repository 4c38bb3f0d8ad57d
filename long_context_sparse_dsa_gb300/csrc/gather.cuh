// gather.cuh -- the 16-key K/V gather step shared by the attention kernels.
//
// A pool's 4 K rows (and its 4 V rows) are one contiguous block of 4*D bf16
// values, so one step of a warp gathers 4 pool slots = 16 keys: 2 tensors x
// 16 rows x D/8 16-byte chunks, spread over the 32 lanes.  The shared tile is
// [16 keys][D] per tensor with the 16-byte chunk c of row r stored at chunk
// position c ^ (r & 7), which makes the ldmatrix reads conflict-free.
//
// Everything that depends only on the lane is computed once (GatherLane);
// per step a lane reads one idx entry (the step's 4 packed pool slots then
// reach every lane by shuffles), forms one address per pool slot, and then
// one compare per copy.  Keys that are not visible (empty slot, or tokens
// after t in the partial pool) are zero-filled.  The backward uses a
// pool-interleaved variant of the tile (gather_step16_il).
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

// Lane constants of the gather.  Copy (sig, ten, rb) of a lane moves the
// 16-byte chunk `ch` of row  rb*ROWS_PER_COPY + row_lo  of slot sig, tensor
// ten (0 = K, 1 = V).  Within the step's shared tile that row is key
// sig*4 + row and its chunk lands at position ch ^ (key & 7); since key & 7 =
// (sig & 1)*4 + row, the destination offset depends on the lane only through
// dst_off[sig & 1][rb] (the sig*4 rows and the tensor add compile-time
// constants).
template <int D>
struct GatherLane {
  static constexpr int NRB = 4 / GatherCfg<D>::ROWS_PER_COPY;   // row blocks per slot (2 or 1)
  int row_lo;                  // lane / CHUNKS
  uint32_t src_off;            // row_lo * ROW_BYTES + ch * 16
  uint32_t dst_off[2][NRB];    // row * ROW_BYTES + ((ch ^ ((sig&1)*4 + row)) << 4)
};

template <int D>
__device__ __forceinline__ GatherLane<D> gather_lane(int lane) {
  using C = GatherCfg<D>;
  GatherLane<D> g;
  const int ch = lane % C::CHUNKS;
  g.row_lo = lane / C::CHUNKS;
  g.src_off = (uint32_t)(g.row_lo * C::ROW_BYTES + ch * 16);
#pragma unroll
  for (int a = 0; a < 2; ++a)
#pragma unroll
    for (int rb = 0; rb < GatherLane<D>::NRB; ++rb) {
      const int row = rb * C::ROWS_PER_COPY + g.row_lo;
      g.dst_off[a][rb] = (uint32_t)(row * C::ROW_BYTES + ((ch ^ (a * 4 + row)) << 4));
    }
  return g;
}

// The idx entry this lane decides for step `grp`: slot grp*4 + (lane & 3), or
// 0 when that slot is past the k selected ones.  Loaded a step ahead of its
// use, so its latency is hidden behind the current step.
__device__ __forceinline__ int slot_raw(const int32_t* irow, int k, int grp) {
  const int slot = grp * 4 + (int)(threadIdx.x & 3);
  return slot < k ? __ldg(irow + slot) : 0;
}

// The 4 pool slots of step `grp` (slots grp*4 .. grp*4+3; slot k is the own
// partial pool), each packed as (pool << 3) | visible rows: 4 for a selected
// pool, (t & 3) + 1 for the partial pool, and the value 0 (pool 0, no rows)
// for an empty slot, so that an empty slot still names a valid address and
// its rows are zero-filled.  Each lane decides slot (lane & 3) from `raw`
// (slot_raw of the same step) with selects (no lane-divergent branch), and
// the four results are shuffled to every lane.  An entry outside the causal
// range is skipped and sets `bad`, which the caller reports once.
__device__ __forceinline__ void step_pools_from(int raw, int k, int grp, int64_t t, uint32_t (&slots)[4],
                                                bool& bad) {
  const int el = (int)elig(t);
  const bool has_part = (t & 3) != 3;
  const uint32_t part = ((uint32_t)(t >> 2) << 3) | (uint32_t)((t & 3) + 1);
  const int slot = grp * 4 + (int)(threadIdx.x & 3);
  const bool sel = slot < k;
  const bool out = sel && raw >= el;
  bad |= out;
  const uint32_t mine =
      sel ? ((raw < 0 || out) ? 0u : (((uint32_t)raw << 3) | 4u)) : ((slot == k && has_part) ? part : 0u);
#pragma unroll
  for (int s = 0; s < 4; ++s) slots[s] = __shfl_sync(0xffffffffu, mine, s);
}
__device__ __forceinline__ void step_pools(const int32_t* irow, int k, int grp, int64_t t, uint32_t (&slots)[4],
                                           bool& bad) {
  step_pools_from(slot_raw(irow, k, grp), k, grp, t, slots, bad);
}
__device__ __forceinline__ int slot_pool(uint32_t v) { return (int)(v >> 3); }
__device__ __forceinline__ int slot_nrows(uint32_t v) { return (int)(v & 7u); }

template <int D>
__device__ __forceinline__ void gather_step16(uint32_t stage, const __nv_bfloat16* __restrict__ K,
                                              const __nv_bfloat16* __restrict__ V, const uint32_t (&slots)[4],
                                              const GatherLane<D>& gl) {
  using C = GatherCfg<D>;
  constexpr int NRB = GatherLane<D>::NRB;
  constexpr int POOL_BYTES = 4 * C::ROW_BYTES;
#pragma unroll
  for (int sig = 0; sig < 4; ++sig) {
    const int nrows = slot_nrows(slots[sig]);
    const int64_t pool_off = (int64_t)slot_pool(slots[sig]) * POOL_BYTES + gl.src_off;
    const char* srcK = reinterpret_cast<const char*>(K) + pool_off;
    const char* srcV = reinterpret_cast<const char*>(V) + pool_off;
#pragma unroll
    for (int rb = 0; rb < NRB; ++rb) {
      const uint32_t bytes = rb * C::ROWS_PER_COPY + gl.row_lo < nrows ? 16u : 0u;
      const uint32_t dst = stage + sig * POOL_BYTES + gl.dst_off[sig & 1][rb];
      cp_async16(dst, srcK + rb * C::ROWS_PER_COPY * C::ROW_BYTES, bytes);
      cp_async16(dst + C::TILE_BYTES, srcV + rb * C::ROWS_PER_COPY * C::ROW_BYTES, bytes);
    }
  }
}

// The same 16-key gather into a pool-interleaved tile: shared row m holds
// token (m >> 2) of slot (m & 3), so that row m of the tile, and column m of
// any product formed from it, belongs to slot m & 3.  The swizzle is the
// usual one (chunk c of row m at c ^ (m & 7)).  Since a lane's rows all have
// the same parity, (m & 7) = ((row & 1) << 2) | slot and the destination is a
// lane constant plus compile-time offsets, XOR the slot.
template <int D>
__device__ __forceinline__ void gather_step16_il(uint32_t stage, const __nv_bfloat16* __restrict__ K,
                                                 const __nv_bfloat16* __restrict__ V, const uint32_t (&slots)[4],
                                                 const GatherLane<D>& gl) {
  using C = GatherCfg<D>;
  constexpr int NRB = GatherLane<D>::NRB;
  constexpr int POOL_BYTES = 4 * C::ROW_BYTES;
  const int ch = (int)((gl.src_off % C::ROW_BYTES) >> 4);
  const uint32_t cpar = (uint32_t)(ch ^ ((gl.row_lo & 1) << 2));   // chunk position before the slot XOR
  const uint32_t row_base = stage + (uint32_t)(gl.row_lo * 4 * C::ROW_BYTES);
#pragma unroll
  for (int sig = 0; sig < 4; ++sig) {
    const int nrows = slot_nrows(slots[sig]);
    const int64_t pool_off = (int64_t)slot_pool(slots[sig]) * POOL_BYTES + gl.src_off;
    const char* srcK = reinterpret_cast<const char*>(K) + pool_off;
    const char* srcV = reinterpret_cast<const char*>(V) + pool_off;
    const uint32_t col = (cpar ^ (uint32_t)sig) << 4;
#pragma unroll
    for (int rb = 0; rb < NRB; ++rb) {
      const uint32_t bytes = rb * C::ROWS_PER_COPY + gl.row_lo < nrows ? 16u : 0u;
      // token row = rb*ROWS_PER_COPY + row_lo  ->  shared row 4*row + sig
      const uint32_t dst = row_base + (uint32_t)((rb * C::ROWS_PER_COPY * 4 + sig) * C::ROW_BYTES) + col;
      cp_async16(dst, srcK + rb * C::ROWS_PER_COPY * C::ROW_BYTES, bytes);
      cp_async16(dst + C::TILE_BYTES, srcV + rb * C::ROWS_PER_COPY * C::ROW_BYTES, bytes);
    }
  }
}

}  // namespace dsa
