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

// Forward calls with at most this many query rows per head take the
// split-key CUDA-core kernel (fa_decode.cuh) instead of the tile kernel.
constexpr int kDecodeMaxTq = 8;

struct AttnShape {
  int B, Hq, Hkv, Tq, Tkv;
  int causal, window;
  float scale_log2;  // scale * log2(e): scores are handled in the exp2 domain
};

struct WaitCfg {
  uint32_t* status;         // device status word
  uint64_t timeout_cycles;  // bound of every mbarrier wait, in SM clock cycles
  // Bound of the waits at exit after a wait gave up (copies still landing in
  // shared memory, MMAs still running before TMEM is freed): never shorter
  // than the default limit, so a short test limit cannot let a CTA leave with
  // work in flight.
  uint64_t drain_cycles;
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

// The same mask as intervals, for masking a tile with one compare-and-select
// per element (evaluating key_visible per element of a 128-wide unrolled row
// costs thousands of cycles per tile).
//
// Keys visible to query i, relative to key k0: [lo, hi) (may be empty or reach
// past either end of a tile); keys at or beyond Tkv are excluded.
__host__ __device__ __forceinline__ void visible_keys(const AttnShape& s, int i, int k0, int* lo,
                                                      int* hi) {
  const int h = s.causal ? min(i + 1, s.Tkv) : s.Tkv;
  const int l = s.window > 0 ? i - s.window + 1 : -(1 << 30);
  *lo = max(l - k0, -(1 << 30));
  *hi = h - k0;
}

// Queries that see key j, relative to query i0: [lo, hi) (queries at or beyond
// Tq are not excluded here).
__host__ __device__ __forceinline__ void visible_queries(const AttnShape& s, int j, int i0, int* lo,
                                                         int* hi) {
  *lo = s.causal ? j - i0 : -(1 << 30);
  *hi = s.window > 0 ? j + s.window - i0 : (1 << 30);
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

// After an abort, wait (bounded by `tmo`, the drain limit, whatever the abort
// flag says) until the last `nst` loads issued into a ring of `nst` slots have
// landed, so that no copy is still in flight into this CTA's shared memory
// when it exits.
__device__ __forceinline__ void drain_ring(uint32_t full_bar0, int nst, int issued,
                                           uint64_t tmo, uint32_t* status) {
  for (int i = issued > nst ? issued - nst : 0; i < issued; ++i)
    mbar_wait(full_bar0 + 8u * static_cast<uint32_t>(i % nst), (i / nst) & 1, tmo, nullptr, status);
}

// Store a 32-row x 8S-column block of an fp32 TMEM accumulator (the warp's
// TMEM lane quarter, columns [taddr, taddr + 8S)), scaled by `mul`, as 16-bit
// values to rows [0, rows_valid) of `base` (row r at base + r * ld). A thread
// holds one row, so storing it directly would make every 16-byte store of the
// warp touch 32 rows; instead the lanes first transpose 16-byte segments
// within groups of S lanes (log2 S butterfly exchange steps), after which each
// store instruction writes 32 / S whole 16S-byte row segments.
template <int S, bool BF16, class T16>
__device__ __forceinline__ void store_acc_block(uint32_t taddr, bool have_data, float mul,
                                                T16* base, int64_t ld, int rows_valid) {
  static_assert(S == 4 || S == 8, "segments per row");
  const int lane = threadIdx.x & 31;
  uint4 a[S];  // this lane's row: S segments of 8 values
#pragma unroll
  for (int h = 0; h < S / 2; ++h) {
    uint32_t v[16];
    if (have_data) {
      tmem_ld16(taddr + 16 * h, v);
      tmem_ld_wait();
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float x = have_data ? __uint_as_float(v[8 * q + 2 * e]) * mul : 0.f;
        const float y = have_data ? __uint_as_float(v[8 * q + 2 * e + 1]) * mul : 0.f;
        w[e] = pack2<BF16>(x, y);
      }
      a[2 * h + q] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  // after the exchange, lane c of a group holds in a[j] segment c of the
  // group's row j
#pragma unroll
  for (int k = S / 2; k >= 1; k >>= 1) {
    const bool hi = (lane & k) != 0;
#pragma unroll
    for (int e = 0; e < S; ++e) {
      if (e & k) continue;
      const uint4 send = hi ? a[e] : a[e ^ k];
      uint4 r;
      r.x = __shfl_xor_sync(0xffffffffu, send.x, k);
      r.y = __shfl_xor_sync(0xffffffffu, send.y, k);
      r.z = __shfl_xor_sync(0xffffffffu, send.z, k);
      r.w = __shfl_xor_sync(0xffffffffu, send.w, k);
      if (hi)
        a[e] = r;
      else
        a[e ^ k] = r;
    }
  }
  const int g = lane / S, c = lane % S;
#pragma unroll
  for (int j = 0; j < S; ++j) {
    const int r = S * g + j;
    if (r < rows_valid) *reinterpret_cast<uint4*>(base + r * ld + 8 * c) = a[j];
  }
}

}  // namespace fa
