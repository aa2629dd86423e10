// Shared definitions of the attention kernels: launch parameters, the mask
// predicate, and the tile ranges that causal / sliding-window skipping uses.
//
// Mask (page "mlx-bun 0.0.4: package/src/model/flash-attention.ts", forward
// shader): key j is hidden from query i when (causal && j > i) or
// (window > 0 && i >= j && i - j >= window). Keys at or beyond Tkv and queries
// at or beyond Tq (tile padding) are hidden as well.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "sm103_ptx.cuh"

namespace fa {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Rows of the query tile one MMA covers (M of tcgen05.mma, one TMEM lane each).
constexpr int kBM = 128;

struct AttnShape {
  int B, Hq, Hkv, Tq, Tkv;
  int causal, window;
  float scale_log2;  // scale * log2(e): scores are handled in the exp2 domain
};

struct WaitCfg {
  uint32_t* status;    // device status word
  uint64_t timeout_cycles;  // bound of every mbarrier wait, in SM clock cycles
};

// Order in which a 1-D grid visits (unit, tile) work items. A unit is a
// (batch, head) or (batch, KV group) whose tiles share an operand (K/V, or
// Q/dO); a tile is a row block. Blocks are dispatched roughly in linear order,
// so the grid walks `chunk` units at a time (their shared operands then stay
// resident in L2) and, inside a chunk, the heaviest tiles first (causal
// masking makes the work per tile uneven), round-robin over the units.
struct TileOrder {
  int units, tiles, chunk;
  int heavy_last;  // 1: the last tile index carries the most work
};

__device__ __forceinline__ void decode_tile(int linear, const TileOrder& o, int* unit, int* tile) {
  const int per_chunk = o.chunk * o.tiles;
  const int c = linear / per_chunk;
  const int r = linear - c * per_chunk;
  const int cu = min(o.chunk, o.units - c * o.chunk);  // units in this (maybe last) chunk
  const int t = r / cu;
  *unit = c * o.chunk + (r - t * cu);
  *tile = o.heavy_last ? o.tiles - 1 - t : t;
}

// Work items of a persistent CTA, handed out by cluster launch control: the
// CTA starts on item blockIdx.x and, instead of exiting after it, takes over
// the next CTA of the grid that has not started yet (in launch order, so the
// TileOrder is kept and faster SMs take more items). Warp 0 requests the
// response that names item k + 1 when it starts item k; every warp reads it
// once done with item k. Responses rotate through kClcSlots slots.
constexpr int kClcSlots = 4;

struct ItemQueue {
  uint32_t resp;   // kClcSlots responses of 16 bytes (shared address, 16-byte aligned)
  uint32_t full;   // kClcSlots barriers: arrival count 1, plus 16 transaction bytes
  uint32_t empty;  // kClcSlots barriers: arrival count = warps of the CTA
};

// Warp 0, whole warp: request the response for item k + 1 once slot k % S has
// been read by every warp (for item k + 1 - S).
__device__ __forceinline__ bool clc_request(const ItemQueue& q, int k, bool leader, uint64_t tmo,
                                            volatile int* abort, uint32_t* status) {
  const int slot = k % kClcSlots;
  if (k >= kClcSlots &&
      !mbar_wait_poll(q.empty + 8u * slot, ((k / kClcSlots) - 1) & 1, tmo, abort, status))
    return false;
  if (leader) {
    mbar_arrive_expect_tx(q.full + 8u * slot, 16);
    clc_try_cancel(q.resp + 16u * slot, q.full + 8u * slot);
  }
  __syncwarp();
  return true;
}

// Every warp, done with item k: the next item in *item, or false when the
// grid has none left (or a wait gave up).
__device__ __forceinline__ bool clc_next(const ItemQueue& q, int k, int lane, int* item,
                                         uint64_t tmo, volatile int* abort, uint32_t* status) {
  const int slot = k % kClcSlots;
  if (!mbar_wait(q.full + 8u * slot, (k / kClcSlots) & 1, tmo, abort, status)) return false;
  const bool got = clc_query(q.resp + 16u * slot, item);
  __syncwarp();
  if (lane == 0) mbar_arrive(q.empty + 8u * slot);
  return got;
}

__host__ __device__ __forceinline__ bool key_visible(int i, int j, int causal, int window) {
  if (causal && j > i) return false;
  if (window > 0 && i >= j && i - j >= window) return false;
  return true;
}

// Keys that any query in [q_lo, q_hi) can see: [first, last) (may be empty).
__host__ __device__ __forceinline__ void key_range(const AttnShape& s, int q_lo, int q_hi,
                                                   int* first, int* last) {
  int lo = 0, hi = s.Tkv;
  if (s.causal) hi = min(hi, q_hi);              // j <= i <= q_hi - 1
  if (s.window > 0) lo = max(0, q_lo - s.window + 1);
  *first = lo;
  *last = max(lo, hi);
}

// Queries that can see any key in [k_lo, k_hi): [first, last) (may be empty).
__host__ __device__ __forceinline__ void query_range(const AttnShape& s, int k_lo, int k_hi,
                                                     int* first, int* last) {
  int lo = 0, hi = s.Tq;
  if (s.causal) lo = k_lo;                        // i >= j >= k_lo
  if (s.window > 0) hi = min(hi, k_hi - 1 + s.window);  // i - j < window
  *first = min(lo, s.Tq);
  *last = max(*first, hi);
}

// True when every (query, key) pair of the block [q_lo, q_hi) x [k_lo, k_hi)
// is visible and in range, so the block needs no per-element mask.
__host__ __device__ __forceinline__ bool block_unmasked(const AttnShape& s, int q_lo, int q_hi,
                                                        int k_lo, int k_hi) {
  if (q_hi > s.Tq || k_hi > s.Tkv) return false;
  if (s.causal && k_hi - 1 > q_lo) return false;
  if (s.window > 0 && (q_hi - 1) - k_lo >= s.window) return false;
  return true;
}

}  // namespace fa
