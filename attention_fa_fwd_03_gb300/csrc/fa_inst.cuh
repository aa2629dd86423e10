// Launch helpers shared by the per-head-dimension instantiation units: build
// the TMA maps a kernel configuration needs and launch it on the caller's
// stream. Each fa_inst_d*.cu picks the tile configuration for its head dim.
#pragma once

#include <algorithm>
#include <atomic>
#include <type_traits>
#include <utility>

#include "fa_bwd.cuh"
#include "fa_bwd_d256.cuh"
#include "fa_bwd_pipelined.cuh"
#include "fa_decode.cuh"
#include "fa_fwd.cuh"
#include "fa_launch.h"

namespace fa {

// Every kernel is launched with programmatic stream serialisation: its launch
// and prologue overlap the end of the previous kernel in the stream, and it
// waits for that kernel (grid_wait_prior) before it touches global memory.
// Appends the attribute to cfg's attribute array `attrs`, which must have room.
inline void allow_early_launch(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attrs) {
  cudaLaunchAttribute& at = attrs[cfg->numAttrs++];
  at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at.val.programmaticStreamSerializationAllowed = 1;
  cfg->attrs = attrs;
}

// Launches kern on a 1-D grid of `grid` CTAs (in clusters of `cluster`).
template <class... P, class... A>
cudaError_t launch_kernel(void (*kern)(P...), int64_t grid, int threads, int smem,
                          cudaStream_t stream, unsigned cluster, A&&... args) {
  if (grid > INT32_MAX) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  if (cluster > 1) {
    attrs[0].id = cudaLaunchAttributeClusterDimension;
    attrs[0].val.clusterDim.x = cluster;
    attrs[0].val.clusterDim.y = 1;
    attrs[0].val.clusterDim.z = 1;
    cfg.numAttrs = 1;
  }
  allow_early_launch(&cfg, attrs);
  return cudaLaunchKernelEx(&cfg, kern, std::forward<A>(args)...);
}

// A kernel that moves registers between its warpgroups (setmaxnreg) may only
// be launched when its launch-time registers cover the new counts; otherwise
// an increase would wait forever. Checked once per kernel.
inline bool register_split_fits(const void* kern, int threads, int needed) {
  if (needed <= 0) return true;
  cudaFuncAttributes attr;
  if (cudaFuncGetAttributes(&attr, kern) != cudaSuccess) return false;
  return static_cast<int64_t>(attr.numRegs) * threads >= needed;
}

// Units per chunk so that the operands the units' tiles share stay in L2:
// about 32 MiB of them at a time (the L2 holds 126 MiB, and the streamed
// per-tile operands and outputs pass through it too), rounded to a multiple
// of `align` units.
inline TileOrder make_order(int units, int tiles, int64_t shared_bytes_per_unit, int align,
                            bool heavy_last, int64_t target = int64_t(32) << 20) {
  int64_t chunk = target / (shared_bytes_per_unit > 0 ? shared_bytes_per_unit : 1);
  chunk = chunk / align * align;
  if (chunk < align) chunk = align;
  if (chunk > units) chunk = units;
  TileOrder o;
  o.units = units;
  o.tiles = tiles;
  o.chunk = static_cast<int>(chunk);
  o.heavy_last = heavy_last ? 1 : 0;
  return o;
}

// Query-row blocks of one head share the group's K and V (reps heads each).
inline TileOrder query_block_order(const AttnShape& s, int rows_per_block, int D) {
  const int reps = s.Hq / s.Hkv;
  const int64_t kv_bytes = int64_t(s.Tkv) * D * 2 * 2;
  return make_order(s.B * s.Hq, (s.Tq + rows_per_block - 1) / rows_per_block, kv_bytes / reps,
                    reps, s.causal != 0);
}

// KV-row blocks of one group share its reps heads' Q and dO. The dK/dV kernel
// nevertheless runs best as one chunk over all groups (measured on the
// causal B4 Hq32 Hkv8 T4096 D128 shape: 0.71 ms against 0.81 ms with 32 MiB
// chunks): heaviest blocks first over the whole grid balances the SMs, and
// its tile loads are latency-bound rather than limited by L2 misses.
constexpr int64_t kDkvChunkBytes = int64_t(1) << 40;
// KV-row blocks of one group share its reps heads' Q and dO.
inline TileOrder kv_block_order(const AttnShape& s, int D) {
  const int reps = s.Hq / s.Hkv;
  const int64_t qdo_bytes = int64_t(reps) * s.Tq * D * 2 * 2;
  return make_order(s.B * s.Hkv, (s.Tkv + kBM - 1) / kBM, qdo_bytes, 1, false, kDkvChunkBytes);
}

template <class C>
cudaError_t run_fwd(const FwdLaunch& a) {
  const int bhq = a.s.B * a.s.Hq, bhkv = a.s.B * a.s.Hkv;
  CUtensorMap mq, mk, mv;
  if (!encode_tile_map(&mq, a.q, C::BF16, C::D, a.s.Tq, bhq, kBM) ||
      !encode_tile_map(&mk, a.k, C::BF16, C::D, a.s.Tkv, bhkv, C::BN) ||
      !encode_tile_map(&mv, a.v, C::BF16, C::D, a.s.Tkv, bhkv, C::BN))
    return cudaErrorInvalidValue;
  auto kern = fa_fwd_kernel<C>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  if (!register_split_fits(reinterpret_cast<const void*>(kern), C::THREADS, C::REG_NEEDED))
    return cudaErrorInvalidConfiguration;
  const TileOrder order = query_block_order(a.s, C::NQ * kBM, C::D);
  return launch_kernel(kern, int64_t(order.units) * order.tiles, C::THREADS, C::SMEM_BYTES, a.stream,
                       1, mq, mk, mv, a.o, a.lse, a.s, order, a.wc);
}

template <int D, bool BF16>
cudaError_t run_dvec(const BwdLaunch& a) {
  const int64_t nrows = static_cast<int64_t>(a.s.B) * a.s.Hq * a.s.Tq;
  constexpr int chunks = D / 8;
  constexpr int tpr = chunks <= 8 ? 8 : (chunks <= 16 ? 16 : 32);
  constexpr int rows_per_block = 256 / tpr;
  const int64_t want = (nrows + rows_per_block - 1) / rows_per_block;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
  const int blocks = static_cast<int>(want < cap ? want : cap);
  return launch_kernel(fa_bwd_dvec_kernel<D, BF16>, blocks, 256, 0, a.stream, 1,
                       static_cast<const uint4*>(a.o), static_cast<const uint4*>(a.dout), a.dvec,
                       nrows);
}

// Kernel configurations without a register split need no check.
template <class C, class = void>
struct RegSplit {
  static constexpr int needed = 0;
};
template <class C>
struct RegSplit<C, std::void_t<decltype(C::REG_NEEDED)>> {
  static constexpr int needed = C::REG_NEEDED;
};

template <class C, class Kern>
cudaError_t launch_dkv_with(const BwdLaunch& a, Kern kern) {
  const int bhq = a.s.B * a.s.Hq, bhkv = a.s.B * a.s.Hkv;
  CUtensorMap mq, mk, mv, mdo;
  if (!encode_tile_map(&mq, a.q, C::BF16, C::D, a.s.Tq, bhq, C::BMQ) ||
      !encode_tile_map(&mdo, a.dout, C::BF16, C::D, a.s.Tq, bhq, C::BMQ) ||
      !encode_tile_map(&mk, a.k, C::BF16, C::D, a.s.Tkv, bhkv, kBM) ||
      !encode_tile_map(&mv, a.v, C::BF16, C::D, a.s.Tkv, bhkv, kBM))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  if (!register_split_fits(reinterpret_cast<const void*>(kern), C::THREADS, RegSplit<C>::needed))
    return cudaErrorInvalidConfiguration;
  const TileOrder order = kv_block_order(a.s, C::D);
  return launch_kernel(kern, int64_t(order.units) * order.tiles, C::THREADS, C::SMEM_BYTES, a.stream,
                       1, mq, mk, mv, mdo, a.lse, a.dvec, a.dk, a.dv, a.scale, a.s, order, a.wc);
}

// dK/dV with each item's tiles split over the two CTAs of a cluster (one item
// per cluster, heaviest first): for grids with at most half as many items as
// SMs.
template <class C>
cudaError_t launch_dkv_split(const BwdLaunch& a) {
  const int bhq = a.s.B * a.s.Hq, bhkv = a.s.B * a.s.Hkv;
  CUtensorMap mq, mk, mv, mdo;
  if (!encode_tile_map(&mq, a.q, C::BF16, C::D, a.s.Tq, bhq, C::BMQ) ||
      !encode_tile_map(&mdo, a.dout, C::BF16, C::D, a.s.Tq, bhq, C::BMQ) ||
      !encode_tile_map(&mk, a.k, C::BF16, C::D, a.s.Tkv, bhkv, kBM) ||
      !encode_tile_map(&mv, a.v, C::BF16, C::D, a.s.Tkv, bhkv, kBM))
    return cudaErrorInvalidValue;
  auto kern = fa_bwd_dkv_kernel<C>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const TileOrder order = kv_block_order(a.s, C::D);
  return launch_kernel(kern, int64_t(C::SPLIT) * order.units * order.tiles, C::THREADS,
                       C::SMEM_BYTES, a.stream, C::SPLIT, mq, mk, mv, mdo, a.lse,
                       static_cast<const float*>(a.dvec), a.dk, a.dv, a.scale, a.s, order, a.wc);
}

// Split each KV block's query tiles over a two-CTA cluster when the blocks
// would leave half the SMs idle and a block has at least two tiles to split
// (with one, the second CTA has nothing to do and the cluster only adds its
// exchange: a folded 32-row block measured 17.5 against 10.3 us).
inline bool dkv_small_grid(const AttnShape& s) {
  const int64_t tiles_per_block = static_cast<int64_t>(s.Hq / s.Hkv) * ((s.Tq + kBM - 1) / kBM);
  return tiles_per_block >= 2 &&
         2 * static_cast<int64_t>(s.B) * s.Hkv * ((s.Tkv + kBM - 1) / kBM) <= device_sm_count();
}

// D = 256 dK/dV: one cluster of C::CLUSTER CTAs (one or two pairs) per
// 128-row KV block (fa_bwd_dkv_pair_kernel), non-persistent, heaviest blocks
// first.
template <class C>
cudaError_t launch_dkv_pair(const BwdLaunch& a) {
  const int bhq = a.s.B * a.s.Hq;
  CUtensorMap mq, mdo;
  if (!encode_tile_map(&mq, a.q, C::BF16, C::D, a.s.Tq, bhq, C::BMQ) ||
      !encode_tile_map(&mdo, a.dout, C::BF16, C::D, a.s.Tq, bhq, C::BMQ))
    return cudaErrorInvalidValue;
  auto kern = fa_bwd_dkv_pair_kernel<C>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const TileOrder order = kv_block_order(a.s, C::D);
  return launch_kernel(kern, int64_t(C::CLUSTER) * order.units * order.tiles, C::THREADS,
                       C::SMEM_BYTES, a.stream, C::CLUSTER, mq, mdo, a.k, a.v, a.lse,
                       static_cast<const float*>(a.dvec), a.dk, a.dv, a.scale, a.s, order, a.wc);
}

// D = 256 dK/dV: two pairs per KV block when the blocks fit twice over on the
// SMs' pairs (so one causal block's query tiles are not the critical path alone).
inline bool dkv_pair_halves(const AttnShape& s) {
  return 4 * static_cast<int64_t>(s.B) * s.Hkv * ((s.Tkv + kBM - 1) / kBM) <= 2 * device_sm_count();
}

// overlap_prior: the dK/dV launch of the same backward directly precedes this
// one on the stream (see fa_bwd_dq_kernel).
template <class C, class Kern>
cudaError_t launch_dq_with(const BwdLaunch& a, Kern kern, bool overlap_prior) {
  const int bhq = a.s.B * a.s.Hq, bhkv = a.s.B * a.s.Hkv;
  CUtensorMap mq, mk, mv, mdo;
  if (!encode_tile_map(&mq, a.q, C::BF16, C::D, a.s.Tq, bhq, kBM) ||
      !encode_tile_map(&mdo, a.dout, C::BF16, C::D, a.s.Tq, bhq, kBM) ||
      !encode_tile_map(&mk, a.k, C::BF16, C::D, a.s.Tkv, bhkv, C::BN) ||
      !encode_tile_map(&mv, a.v, C::BF16, C::D, a.s.Tkv, bhkv, C::BN))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  if (!register_split_fits(reinterpret_cast<const void*>(kern), C::THREADS, RegSplit<C>::needed))
    return cudaErrorInvalidConfiguration;
  const TileOrder order = query_block_order(a.s, kBM, C::D);
  return launch_kernel(kern, int64_t(order.units) * order.tiles, C::THREADS, C::SMEM_BYTES, a.stream,
                       1, mq, mk, mv, mdo, a.q, a.lse, a.dvec, a.dq, a.scale, a.s, order, a.wc,
                       overlap_prior ? 1 : 0);
}

// Softmax warpgroups of the pipelined backward kernels: four (32 score columns
// each) give every SM sub-partition four softmax warps to hide the TMEM and
// MUFU latencies with.
constexpr int kSoftmaxWarpgroups = 4;

// Backward for one head dim. D <= 128: the pipelined 128 x 128 kernels
// (fa_bwd_pipelined.cuh). D = 256: the dK and dV accumulators alone fill TMEM,
// so dV and dK are computed by the two CTAs of a pair that exchange P (two
// pairs per KV block on small grids; fa_bwd_d256.cuh), and dQ runs the
// pipelined kernel with 64-key tiles and Q in TMEM. Tq <= 8: the vector dK/dV
// and the split-key dQ (fa_decode.cuh).
// dQ of short query blocks on the split-key kernel (defined below)
template <int D, bool BF16>
cudaError_t run_dq_decode(const BwdLaunch& a, bool overlap_prior);

// dK / dV of short query blocks: the vector kernel, one CTA per (batch, KV
// group, kVecKeys keys), on the call's own row shape, in chunks of RC rows.
template <class C>
cudaError_t launch_dkv_vec(const BwdLaunch& a) {
  const AttnShape& s = a.s_rows;
  auto kern = fa_bwd_dkv_vec_kernel<C>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int64_t blocks =
      static_cast<int64_t>(s.B) * s.Hkv * ((s.Tkv + kVecKeys - 1) / kVecKeys);
  if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
  return launch_kernel(kern, blocks, kVecThreads, C::SMEM_BYTES, a.stream, 1,
                       static_cast<const uint16_t*>(a.q), static_cast<const uint16_t*>(a.k),
                       static_cast<const uint16_t*>(a.v), static_cast<const uint16_t*>(a.dout),
                       a.lse, a.dvec, static_cast<uint16_t*>(a.dk), static_cast<uint16_t*>(a.dv), s);
}

template <int D, bool BF16>
cudaError_t run_dkv_vec(const BwdLaunch& a) {
  const int rows = a.s_rows.Hq / a.s_rows.Hkv * a.s_rows.Tq;  // query rows per KV group
  if (rows <= 8) return launch_dkv_vec<DkvVecCfg<D, BF16, 8>>(a);
  if (rows <= 16) return launch_dkv_vec<DkvVecCfg<D, BF16, 16>>(a);
  return launch_dkv_vec<DkvVecCfg<D, BF16, 32>>(a);
}

// Short query blocks (Tq <= 8), masked or not: a tile per head would be almost
// all padding, and with a causal or window mask the heads' rows cannot share
// a tile (the mask depends on each row's position within its head). Measured
// per dK/dV launch at B2 Hq8 Hkv2 Tkv1024 D128 (ncu launch lists): 7.1 us at
// Tq = 1 and 12.7 us at Tq = 8 against 10.3 us for the heads' rows folded into
// one tile, and 12.4 against 19.9 us for a causal Tq = 8 call on one tile per
// head.
inline bool dkv_vector_path(const BwdLaunch& a) { return a.s_rows.Tq <= kDecodeMaxTq; }

// dQ starts beside dK/dV (fa_bwd_dq_kernel's overlap_prior) where dK/dV leaves
// SMs idle for long: masked grids, whose KV blocks carry unequal numbers of
// tiles so the SMs run dry one by one, and short query blocks, whose small
// vector and split-key CTAs share SMs. Unmasked tile grids finish their equal
// blocks together; there the dQ CTAs that start early only take a second
// block each while the rest start late, which measured slower (B2 Hq8 Hkv8
// T1024 D128: 62.2 against 58.2 us per fwd + bwd step; causal B2 Hq8 Hkv2
// T2048 D64: 80.5 against 104.7).
inline bool dq_overlaps_dkv(const BwdLaunch& a) {
  return a.s_rows.causal != 0 || a.s_rows.window > 0 || dkv_vector_path(a);
}

template <int D, bool BF16>
cudaError_t run_bwd(const BwdLaunch& a, int phases) {
  cudaError_t e = cudaSuccess;
  if (phases & kPhaseDvec) e = run_dvec<D, BF16>(a);
  if (e != cudaSuccess) return e;
  if (phases & kPhaseDkv) {
    if (dkv_vector_path(a)) {
      e = run_dkv_vec<D, BF16>(a);
    } else if constexpr (D <= 128) {
      using C = DkvCfg<D, BF16, kSoftmaxWarpgroups>;
      if (dkv_small_grid(a.s))
        e = launch_dkv_split<DkvCfg<D, BF16, kSoftmaxWarpgroups, 2>>(a);
      else
        e = launch_dkv_with<C>(a, fa_bwd_dkv_kernel<C>);
    } else {
      e = dkv_pair_halves(a.s) ? launch_dkv_pair<DkvPairCfg<BF16, 2>>(a)
                               : launch_dkv_pair<DkvPairCfg<BF16>>(a);
    }
  }
  if (e != cudaSuccess) return e;
  if (phases & kPhaseDq) {
    // dQ needs only the D-vector of the phases before it: right after this
    // call's dK/dV launch it may start without waiting for that grid
    const bool overlap = (phases & kPhaseDkv) != 0 && dq_overlaps_dkv(a);
    if (a.s_rows.Tq <= kDecodeMaxTq) return run_dq_decode<D, BF16>(a, overlap);
    if constexpr (D <= 128) {
      using C = DqCfg<D, BF16, kSoftmaxWarpgroups>;
      e = launch_dq_with<C>(a, fa_bwd_dq_kernel<C>, overlap);
    } else {
      // 64-key tiles, two softmax warpgroups, Q in TMEM, K / V rings 3 / 2
      using C = DqCfg<D, BF16, 2, 64, 3, 2, true>;
      e = launch_dq_with<C>(a, fa_bwd_dq_kernel<C>, overlap);
    }
  }
  return e;
}

// Short query blocks (Tq <= 8): the split-key kernels of fa_decode.cuh, one
// cluster of `split` CTAs per (batch, query head). The cluster size trades the
// keys each CTA walks (nk / split) against the waves the clusters need: the
// device runs at most M(split) such clusters at once (queried once per kernel,
// device and size, into `cache`), so the estimated time is
// ceil(clusters / M(split)) * (nk / split + fixed work). Slices are whole
// 32-key blocks; a cluster never has more CTAs than 32-key blocks to give them.
// `cfg` holds the block size, shared memory and stream; `attr` its cluster
// attribute, whose size is set here along with the grid.
inline void decode_split(const void* kern, cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr,
                         std::atomic<int> (*cache)[kDecodeMaxSplit + 1], int64_t units, int nk,
                         int* split_out,
                         int* per_out) {
  int dev = 0;
  cudaGetDevice(&dev);
  const int blocks32 = std::max(1, (nk + 31) / 32);
  int split = 1;
  double best = 0.0;
  for (int sz = 1; sz <= kDecodeMaxSplit; sz *= 2) {
    if (sz > 1 && sz > blocks32) break;
    int m = dev >= 0 && dev < 64 ? cache[dev][sz].load(std::memory_order_relaxed) : 0;
    if (m == 0) {
      cfg->gridDim = dim3(static_cast<unsigned>(sz), 1, 1);
      attr->val.clusterDim.x = static_cast<unsigned>(sz);
      if (cudaOccupancyMaxActiveClusters(&m, kern, cfg) != cudaSuccess || m < 1) {
        cudaGetLastError();  // clear; this size is not used
        continue;
      }
      if (dev >= 0 && dev < 64) cache[dev][sz].store(m, std::memory_order_relaxed);
    }
    const double waves = static_cast<double>((units + m - 1) / m);
    const double cost = waves * ((nk + sz - 1) / sz + 64);  // + per-CTA fixed work, in keys
    if (sz == 1 || cost < best) {
      best = cost;
      split = sz;
    }
  }
  int per = (nk + split - 1) / split;
  per = std::max(32, (per + 31) / 32 * 32);
  split = std::max(1, (nk + per - 1) / per);
  cfg->gridDim = dim3(static_cast<unsigned>(units * split), 1, 1);
  attr->val.clusterDim.x = static_cast<unsigned>(split);
  *split_out = split;
  *per_out = per;
}

// Launch configuration of a split-key kernel with cluster dimension x.
inline void decode_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, int smem,
                          cudaStream_t stream) {
  *cfg = cudaLaunchConfig_t{};
  cfg->blockDim = dim3(kDecodeThreads, 1, 1);
  cfg->dynamicSmemBytes = static_cast<size_t>(smem);
  cfg->stream = stream;
  attr->id = cudaLaunchAttributeClusterDimension;
  attr->val.clusterDim.x = 1;
  attr->val.clusterDim.y = 1;
  attr->val.clusterDim.z = 1;
  cfg->attrs = attr;
  cfg->numAttrs = 1;
}

template <class C>
cudaError_t launch_fwd_decode(const FwdLaunch& a) {
  int k_first, k_last;
  key_range(a.s, 0, a.s.Tq, &k_first, &k_last);
  auto kern = fa_fwd_decode_kernel<C>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  CUtensorMap mk, mv;
  const int bhkv = a.s.B * a.s.Hkv;
  if (!encode_tile_map(&mk, a.k, C::BF16, C::D, a.s.Tkv, bhkv, C::SK) ||
      !encode_tile_map(&mv, a.v, C::BF16, C::D, a.s.Tkv, bhkv, C::SK))
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  decode_config(&cfg, attr, C::SMEM_BYTES, a.stream);
  static std::atomic<int> max_active[64][kDecodeMaxSplit + 1] = {};  // shared by host threads
  int split, per;
  decode_split(reinterpret_cast<const void*>(kern), &cfg, attr, max_active,
               static_cast<int64_t>(a.s.B) * a.s.Hq, k_last - k_first, &split, &per);
  allow_early_launch(&cfg, attr);
  return cudaLaunchKernelEx(&cfg, kern, mk, mv, static_cast<const uint16_t*>(a.q),
                            static_cast<uint16_t*>(a.o), a.lse, a.s, split, k_first, k_last, per,
                            a.wc);
}

// dQ of short query blocks, on the call's own (unfolded) shape; reads the
// D-vector the first backward phase wrote.
template <class C>
cudaError_t launch_dq_decode(const BwdLaunch& a, bool overlap_prior) {
  const AttnShape& s = a.s_rows;
  int k_first, k_last;
  key_range(s, 0, s.Tq, &k_first, &k_last);
  auto kern = fa_bwd_dq_decode_kernel<C>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  CUtensorMap mk, mv;
  const int bhkv = s.B * s.Hkv;
  if (!encode_tile_map(&mk, a.k, C::BF16, C::D, s.Tkv, bhkv, C::SK) ||
      !encode_tile_map(&mv, a.v, C::BF16, C::D, s.Tkv, bhkv, C::SK))
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  decode_config(&cfg, attr, C::SMEM_BYTES, a.stream);
  static std::atomic<int> max_active[64][kDecodeMaxSplit + 1] = {};  // shared by host threads
  int split, per;
  decode_split(reinterpret_cast<const void*>(kern), &cfg, attr, max_active,
               static_cast<int64_t>(s.B) * s.Hq, k_last - k_first, &split, &per);
  allow_early_launch(&cfg, attr);
  return cudaLaunchKernelEx(&cfg, kern, mk, mv, static_cast<const uint16_t*>(a.q),
                            static_cast<const uint16_t*>(a.dout), a.lse, a.dvec,
                            static_cast<uint16_t*>(a.dq), a.scale, s, split, k_first, k_last, per,
                            a.wc, overlap_prior ? 1 : 0);
}

template <int D, bool BF16>
cudaError_t run_dq_decode(const BwdLaunch& a, bool overlap_prior) {
  const int tq = a.s_rows.Tq;
  if (tq <= 1) return launch_dq_decode<DecodeDqCfg<D, 1, BF16>>(a, overlap_prior);
  if (tq <= 2) return launch_dq_decode<DecodeDqCfg<D, 2, BF16>>(a, overlap_prior);
  if (tq <= 4) return launch_dq_decode<DecodeDqCfg<D, 4, BF16>>(a, overlap_prior);
  return launch_dq_decode<DecodeDqCfg<D, 8, BF16>>(a, overlap_prior);
}

template <int D, bool BF16>
cudaError_t run_fwd_decode(const FwdLaunch& a) {
  if (a.s.Tq <= 1) return launch_fwd_decode<DecodeFwdCfg<D, 1, BF16>>(a);
  if (a.s.Tq <= 2) return launch_fwd_decode<DecodeFwdCfg<D, 2, BF16>>(a);
  if (a.s.Tq <= 4) return launch_fwd_decode<DecodeFwdCfg<D, 4, BF16>>(a);
  return launch_fwd_decode<DecodeFwdCfg<D, 8, BF16>>(a);
}

}  // namespace fa

// A forward grid of two-tile (256-row) query blocks that would leave SMs
// idle: run one 128-row tile per CTA instead (twice the blocks; with one tile
// a CTA's TMEM has room for two score buffers, so S(j+1) is computed while the
// softmax works on S(j)).
namespace fa {
inline bool fwd_small_grid(const AttnShape& s) {
  return static_cast<int64_t>(s.B) * s.Hq * ((s.Tq + 2 * kBM - 1) / (2 * kBM)) < device_sm_count();
}
}  // namespace fa

// Define launch_fwd_d<D> / launch_bwd_d<D> for one head dim, given the forward
// tile configuration (NQ query tiles per CTA, key tile BN, STAGES of the K/V
// ring). With two query tiles per CTA, small grids take one tile per CTA and a
// K/V ring three deep.
#define FA_DEFINE_HEAD_DIM(D, FNQ, FBN, FST)                                              \
  namespace fa {                                                                          \
  cudaError_t launch_fwd_d##D(const FwdLaunch& a) {                                       \
    if (a.s.Tq <= kDecodeMaxTq)                                                           \
      return a.bf16 ? run_fwd_decode<D, true>(a) : run_fwd_decode<D, false>(a);           \
    if constexpr (FNQ == 2) {                                                             \
      if (fwd_small_grid(a.s))                                                            \
        return a.bf16 ? run_fwd<FwdCfg<D, 1, FBN, 3, true>>(a)                            \
                      : run_fwd<FwdCfg<D, 1, FBN, 3, false>>(a);                          \
    }                                                                                     \
    return a.bf16 ? run_fwd<FwdCfg<D, FNQ, FBN, FST, true>>(a)                            \
                  : run_fwd<FwdCfg<D, FNQ, FBN, FST, false>>(a);                          \
  }                                                                                       \
  cudaError_t launch_bwd_d##D(const BwdLaunch& a, int phases) {                           \
    return a.bf16 ? run_bwd<D, true>(a, phases) : run_bwd<D, false>(a, phases);           \
  }                                                                                       \
  }
