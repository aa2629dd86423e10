// dK/dV for head dim 256 on a pair of CTAs (or two pairs of a four-CTA
// cluster on small grids).
//
// What it computes is backward pass 2 of page "mlx-bun 0.0.4: package/src/
// model/flash-attention.ts" with the KV-row ownership of page "[Metal] Add
// Flash Attention VJP for training", Implementation Notes: one cluster owns
// 128 KV rows of one (batch, KV group) and walks every query tile of every
// query head of the group that sees them, accumulating
//   dV += P^T dO      and      dK += scale * dS^T Q,   dS = P o (dP - D),
// with P = 2^(S log2 e - LSE log2 e) recomputed from the cached LSE.
//
// GB300 design. At this width the two fp32 accumulators (128 rows x 256
// columns each) fill all of one SM's TMEM, so the work is split over the two
// CTAs of a cluster, each with a full TMEM of its own, in a way that gives
// both the same two contractions per tile:
//   rank 0 (P side)   S^T = K Q^T   ->  P^T  ->  dV += P^T dO
//   rank 1 (dS side)  dP^T = V dO^T ->  dS^T = P^T o (dP^T - D)  ->  dK += dS^T Q
// The P side hands P (fp16, 16 KB per tile) to the dS side through
// distributed shared memory: its softmax threads write their rows into a local
// buffer, and one thread copies the buffer into the peer's with a bulk copy
// that counts its bytes on the peer's mbarrier (the dS side announces 16 KB
// per buffer phase); the dS side arrives back, relaxed, once it has read a
// buffer. Two buffers alternate on each side. (Measured on this shape: plain
// peer stores followed by a cluster-scope fence cost 3.5k cycles per tile,
// per-thread asynchronous peer stores 0.9k cycles of the softmax warps' time;
// the tile's MMAs take 1k.)
// The operand every tile of the item multiplies (K on the P side, V on the
// dS side) is kept in TMEM as the A operand of the score MMA (an A operand
// from TMEM runs at the full rate at N = 64, one from shared memory does not),
// which leaves shared memory for two query-tile rings three deep:
//   ring A  the score's B operand (Q on the P side, dO on the dS side),
//           freed by the score MMA
//   ring B  the accumulation's B operand (dO on the P side, Q on the dS
//           side), freed by the accumulating MMA.
// Per 64-row query tile each side issues 16 score MMAs (N = 64, K = 16) and 4
// accumulating MMAs (N = 256); the score of tile j+1 runs while the softmax
// warps work on tile j. Score blocks alternate between two 64-column TMEM
// blocks, so the score of tile j+2 reuses tile j's block after the
// accumulating MMA of tile j has read it (issue order).
// Roles per CTA (384 threads):
//   warp 0  TMA producer of ring A        warp 1  MMA issuer
//   warp 2  TMA producer of ring B; TMEM allocator
//   warp 3  per-tile row statistics (-LSE log2 e on the P side, -D on the
//           dS side) into a double-buffered shared array; on the P side it
//           also sends each tile's P buffer to the peer
//   warps 4-11  two softmax warpgroups, 32 query columns each; they also
//           write the item's K or V rows into TMEM and store the accumulator.
// HALVES = 2 (grids where one causal block's tiles would be the critical
// path): a cluster of four CTAs, two such pairs (ranks 0-1 and 2-3), each
// taking half of the block's query tiles; pair 1 leaves its fp32
// accumulators in its own shared memory (the rings are free once its MMAs
// have completed) and pair 0 adds them, rank r from rank r + 2, through
// distributed shared memory before it stores.
#pragma once

#include <type_traits>

#include "fa_bwd_pipelined.cuh"
#include "fa_common.cuh"

namespace fa {

template <bool BF16_, int HALVES_ = 1>
struct DkvPairCfg {
  static constexpr int D = 256;
  static constexpr bool BF16 = BF16_;
  static constexpr int HALVES = HALVES_;        // pairs sharing a block's query tiles
  static constexpr int CLUSTER = 2 * HALVES;    // CTAs per cluster
  static constexpr int PART_ROW = D * 4;        // a row of fp32 partial sums (pair 1)
  static constexpr int BMQ = 64;              // query rows per tile (N of the score MMAs)
  static constexpr int NWG = 2;               // softmax warpgroups, 32 query columns each
  static constexpr int RST = 3;               // depth of both rings
  static constexpr int KREG = D / 64;         // 64-column blocks of a row
  static constexpr int REGION = BMQ * 128;    // one 64-column block of a query tile
  static constexpr int TILE = KREG * REGION;  // 32 KB
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + RST * TILE;
  static constexpr int PBUF = 128 * BMQ * 2;  // P of one tile: 128 KV rows x 64 fp16
  static constexpr int OFF_PBUF = OFF_B + RST * TILE;  // P buffers (same place on both sides)
  static constexpr int OFF_STATS = OFF_PBUF + 2 * PBUF;  // [2][BMQ] fp32
  static constexpr int OFF_BAR = OFF_STATS + 2 * BMQ * 4;
  // barriers (same indices on both sides; b_pbuf is "P buffer free" on the P
  // side and "P buffer full" on the dS side, each arrived on by the peer)
  static constexpr int B_AFULL = 0, B_AEMPTY = B_AFULL + RST, B_BFULL = B_AEMPTY + RST,
                       B_BEMPTY = B_BFULL + RST, B_STFULL = B_BEMPTY + RST,
                       B_STEMPTY = B_STFULL + 2, B_OPREADY = B_STEMPTY + 2,
                       B_SCFULL = B_OPREADY + 1, B_READY = B_SCFULL + 2, B_PBUF = B_READY + 2,
                       B_STAGED = B_PBUF + 2, B_DONE = B_STAGED + 2, B_DRAIN = B_DONE + 1,
                       NBAR = B_DRAIN + 1;
  // misc: TMEM base address, abort flag, and (dS side) the number of P
  // buffers the peer has sent, stored there by the peer at its exit
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16;  // base must be 1024-aligned (checked)
  static constexpr int THREADS = 128 + 128 * NWG;
  static constexpr int SOFT_WARPS = 4 * NWG;
  // TMEM: the item's K or V (16-bit pairs, D / 2 columns), two score blocks,
  // the accumulator
  static constexpr int OP_COL = 0;
  static constexpr int SC_COL0 = D / 2;
  static constexpr int ACC_COL = 256;
  static constexpr uint32_t sc_col(int b) { return SC_COL0 + BMQ * b; }
  static_assert(SC_COL0 + 2 * BMQ <= ACC_COL && ACC_COL + D <= 512, "TMEM budget");
  static_assert(BMQ == 32 * NWG, "one 32-column chunk per softmax warpgroup");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
  static_assert(HALVES == 1 || (HALVES == 2 && 128 * PART_ROW <= OFF_PBUF), "partial sums");
};

// Launched with a cluster of C::CLUSTER CTAs (cudaLaunchKernelEx).
template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
fa_bwd_dkv_pair_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_do,
                       const void* __restrict__ k_rows, const void* __restrict__ v_rows,
                       const float* __restrict__ lse, const float* __restrict__ dvec,
                       void* __restrict__ dk_out, void* __restrict__ dv_out, float scale,
                       AttnShape s, TileOrder order, WaitCfg wc) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const uint32_t rank = cluster_ctarank();   // even: P side, odd: dS side
  const bool pside = (rank & 1u) == 0;
  const uint32_t peer = rank ^ 1u;            // the other side of this pair
  const int pair = static_cast<int>(rank >> 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  auto bar = [&](int i) { return smem_u32(bars + i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile int* peer_sent = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);
  float* stats = reinterpret_cast<float*>(smem + C::OFF_STATS);
  const uint64_t tmo = wc.timeout_cycles;
  const int reps = s.Hq / s.Hkv;
  const DkvItem t = dkv_item(static_cast<int>(blockIdx.x) / C::CLUSTER, order, s, C::BMQ,
                             C::HALVES, pair);
  const int n = t.n_iter;
  const bool aligned = (sbase & 1023u) == 0;  // the 128-byte swizzle needs it

  if (threadIdx.x == 0) {
    *abort_flag = aligned ? 0 : 1;
    *peer_sent = 0;
    if (!aligned) {
      grid_wait_prior();
      atomicOr(wc.status, kStatusSmemMisaligned);
    }
    for (int i = 0; i < C::NBAR; ++i) {
      uint32_t cnt = 1;
      if (i == C::B_STFULL || i == C::B_STFULL + 1) cnt = 32;  // the staging warp's lanes
      if (i == C::B_STEMPTY || i == C::B_STEMPTY + 1 || i == C::B_OPREADY || i == C::B_READY ||
          i == C::B_READY + 1 || i == C::B_STAGED || i == C::B_STAGED + 1)
        cnt = C::SOFT_WARPS;  // one arrival per softmax warp
      // P buffer free (P side): one arrival per softmax warp of the peer; P
      // buffer full (dS side): its own expect_tx arrival, then the peer's bytes
      if (i == C::B_PBUF || i == C::B_PBUF + 1) cnt = pside ? C::SOFT_WARPS : 1;
      mbar_init(bar(i), cnt);
    }
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  grid_wait_prior();  // the previous grid's outputs are complete and visible
  grid_release_next();
  tc_fence_before();
  __syncthreads();
  // every CTA has initialised its barriers before any arrives on a peer's or
  // writes into its shared memory
  cluster_barrier();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  int seen = 0;  // dS side, warp 4 lane 0: P buffers received so far
  if (warp == 0 || warp == 2) {
    // --------------------------------------------------- producers: rings A, B
    // the whole warp runs the loop; one elected lane issues. Q and dO tiles
    // are read by every KV block of the group: keep them in L2.
    const bool leader = elect_one_sync();
    const bool ring_a = warp == 0;
    const CUtensorMap* map = (ring_a == pside) ? &map_q : &map_do;
    if (leader) tma_prefetch_desc(map);
    const int full = ring_a ? C::B_AFULL : C::B_BFULL, empty = ring_a ? C::B_AEMPTY : C::B_BEMPTY;
    const uint32_t ring = sbase + (ring_a ? C::OFF_A : C::OFF_B);
    const uint64_t pol = l2_policy_evict_last();
    int it = 0;
    bool ok = !*abort_flag;
    for (; ok && it < n; ++it) {
      const int zq = t.b * s.Hq + t.g * reps + (t.it0 + it) / t.n_qt;
      const int i0 = (t.i_lo + (t.it0 + it) % t.n_qt) * C::BMQ;
      const int st = it % C::RST;
      if (it >= C::RST) ok = mbar_wait(bar(empty + st), ((it / C::RST) - 1) & 1, tmo, abort_flag, wc.status);
      if (!ok) break;
      if (leader) mbar_arrive_expect_tx(bar(full + st), C::TILE);
      for (int r = 0; r < C::KREG; ++r)
        if (leader) tma_load_3d_hint(ring + st * C::TILE + r * C::REGION, map, bar(full + st), r * 64, i0, zq, pol);
    }
    if (*abort_flag) drain_ring(bar(full), C::RST, it, wc.drain_cycles, wc.status);
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer
    const bool leader = elect_one_sync();
    constexpr uint32_t ab = C::BF16 ? 1 : 0;
    constexpr uint32_t idesc_sc = make_idesc_f16(kBM, C::BMQ, ab, 0, 0);  // S^T, dP^T
    constexpr uint32_t idesc_acc = make_idesc_f16(kBM, C::D, ab, 0, 1);   // dV, dK
    auto wait = [&](int b, int parity) {
      return mbar_wait_poll(bar(b), parity & 1, tmo, abort_flag, wc.status);
    };
    // score(j) = OP x ringA(j)^T into block j % 2: A (K or V) from TMEM, K = head dim
    auto issue_score = [&](int j) {
      const uint64_t bd = make_sdesc(sbase + C::OFF_A + (j % C::RST) * C::TILE, 16, 1024, 2);
#pragma unroll
      for (int kk = 0; kk < C::D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * C::REGION + (kk & 3) * 32;
        if (leader) mma_ts(tmem + C::sc_col(j & 1), tmem + C::OP_COL + 8 * kk, bd + (off >> 4), idesc_sc, kk > 0);
      }
      if (leader) mma_commit(bar(C::B_SCFULL + (j & 1)));
      if (leader) mma_commit(bar(C::B_AEMPTY + j % C::RST));  // ring A is read by the score only
    };
    // acc += block(j) x ringB(j): A (P^T or dS^T, 16-bit) from TMEM, B MN-major, K = query rows
    auto issue_acc = [&](int j) {
      const uint64_t bd = make_sdesc(sbase + C::OFF_B + (j % C::RST) * C::TILE, C::REGION, 1024, 2);
#pragma unroll
      for (int kk = 0; kk < C::BMQ / 16; ++kk)
        if (leader) mma_ts(tmem + C::ACC_COL, tmem + chunk_operand_col(C::sc_col(j & 1), kk),
                           bd + ((kk * 16 * 128) >> 4), idesc_acc, (j > 0 || kk > 0) ? 1u : 0u);
      if (leader) mma_commit(bar(C::B_BEMPTY + j % C::RST));
    };
    bool ok = !*abort_flag;
    if (ok && n > 0) {
      // the item's K / V rows in TMEM, then the first score
      ok = wait(C::B_OPREADY, 0) && wait(C::B_AFULL, 0);
      if (ok) {
        tc_fence_after();
        issue_score(0);
      }
      for (int j = 0; ok && j < n; ++j) {
        if (j + 1 < n) {
          // score(j+1) into the block acc(j-1) has read (issue order)
          ok = wait(C::B_AFULL + (j + 1) % C::RST, ((j + 1) / C::RST) & 1);
          if (!ok) break;
          tc_fence_after();
          issue_score(j + 1);
        }
        // P^T(j) (P side) or dS^T(j) (dS side) in TMEM, and ring B(j)
        ok = wait(C::B_READY + (j & 1), (j >> 1) & 1) && wait(C::B_BFULL + j % C::RST, (j / C::RST) & 1);
        if (!ok) break;
        tc_fence_after();
        issue_acc(j);
      }
      if (ok && leader) mma_commit(bar(C::B_DONE));  // the accumulator is final
    }
    // every issued MMA completes before the CTA exits
    if (leader) mma_commit(bar(C::B_DRAIN));
    mbar_wait(bar(C::B_DRAIN), 0, wc.drain_cycles, nullptr, wc.status);
  } else if (warp == 3) {
    // ------------------------------------------- per-tile row statistics
    // each lane loads its two rows of the next tile before waiting for the
    // slot, so the global-load latency hides behind the wait
    constexpr int RPL = C::BMQ / 32;
    float v[RPL];
    auto load = [&](int it) {
      const int h = t.g * reps + (t.it0 + it) / t.n_qt;
      const int i0 = (t.i_lo + (t.it0 + it) % t.n_qt) * C::BMQ;
      const int64_t base = static_cast<int64_t>(t.b * s.Hq + h) * s.Tq;
#pragma unroll
      for (int r = 0; r < RPL; ++r) {
        const int i = i0 + lane + 32 * r;
        if (pside) {
          // -LSE log2 e; a row past Tq or with no visible key: P = 0
          const float L = i < s.Tq ? lse[base + i] : -INFINITY;
          v[r] = (L == -INFINITY) ? -INFINITY : -L * kLog2e;
        } else {
          v[r] = i < s.Tq ? -dvec[base + i] : 0.f;
        }
      }
    };
    // P side: copy tile j's P buffer to the peer once the softmax warps have
    // written it (they waited for the peer to free it first)
    const bool leader = elect_one_sync();
    auto send = [&](int j) {
      const int b = j & 1;
      if (!mbar_wait(bar(C::B_STAGED + b), (j >> 1) & 1, tmo, abort_flag, wc.status)) return false;
      const uint32_t buf = sbase + C::OFF_PBUF + b * C::PBUF;
      if (leader) bulk_copy_to_peer(peer_addr(buf, peer), buf, C::PBUF, peer_addr(bar(C::B_PBUF + b), peer));
      __syncwarp();
      return true;
    };
    int sent = 0;
    bool ok = !*abort_flag;
    if (ok && n > 0) load(0);
    for (int it = 0; ok && it < n; ++it) {
      const int slot = it & 1;
      if (it >= 2 && !mbar_wait(bar(C::B_STEMPTY + slot), ((it >> 1) - 1) & 1, tmo, abort_flag, wc.status)) break;
      float* dst = stats + slot * C::BMQ;
#pragma unroll
      for (int r = 0; r < RPL; ++r) dst[lane + 32 * r] = v[r];
      mbar_arrive(bar(C::B_STFULL + slot));
      if (it + 1 < n) load(it + 1);
      if (pside && it >= 1) {
        ok = send(it - 1);
        sent += ok ? 1 : 0;
      }
    }
    if (pside && ok && n > 0) sent += send(n - 1) ? 1 : 0;
    // the peer drains exactly the copies that were issued if it gives up; the
    // count reaches it through the cluster barrier at exit
    if (pside && leader) {
      const uint32_t remote = peer_addr(smem_u32(const_cast<int*>(peer_sent)), peer);
      asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(remote), "r"(sent) : "memory");
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int wg = (warp - 4) >> 2;       // query columns [32 wg, 32 wg + 32) of a tile
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;    // KV row within the block (TMEM lane)
    const int krow = t.k0 + r;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    using T16 = typename std::conditional<C::BF16, __nv_bfloat16, __half>::type;
    bool ok = !*abort_flag;
    // the item's K (P side) or V (dS side) rows in TMEM: this warpgroup's half
    // of the head dim for the thread's row (zeros past Tkv)
    {
      constexpr int COLS = C::D / 2 / C::NWG;  // 32-bit TMEM columns per warpgroup
      const T16* rows = static_cast<const T16*>(pside ? k_rows : v_rows);
      const bool valid = krow < s.Tkv;
      const uint4* src = reinterpret_cast<const uint4*>(
          rows + (static_cast<int64_t>(t.bg) * s.Tkv + (valid ? krow : 0)) * C::D) + wg * (COLS / 4);
#pragma unroll
      for (int c = 0; c < COLS; c += 32) {
        uint32_t w[32];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint4 x = valid ? __ldg(src + c / 4 + e) : make_uint4(0, 0, 0, 0);
          w[4 * e] = x.x; w[4 * e + 1] = x.y; w[4 * e + 2] = x.z; w[4 * e + 3] = x.w;
        }
        tmem_st32(tmem + lane_base + C::OP_COL + wg * COLS + c, w);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::B_OPREADY));
    }
    const uint64_t c2 = f2_pack(s.scale_log2, s.scale_log2);
    // this thread's 64 bytes of a P buffer row: 16-byte chunks 4 wg .. 4 wg + 3,
    // swizzled by the row so that a warp's accesses spread over the banks
    auto pbuf_off = [&](int b, int c) {
      return static_cast<uint32_t>(C::OFF_PBUF + b * C::PBUF + r * 128 + (((4 * wg + c) ^ (r & 7)) << 4));
    };
    // dS side: announce the bytes of the first two P buffers
    const bool poster = !pside && warp == 4 && lane == 0;
    if (poster && ok) {
      mbar_arrive_expect_tx(bar(C::B_PBUF), C::PBUF);
      mbar_arrive_expect_tx(bar(C::B_PBUF + 1), C::PBUF);
    }
    const int i_first = t.i_lo * C::BMQ, i_end = (t.i_lo + t.n_qt) * C::BMQ;
    int i0 = (t.i_lo + t.it0 % max(t.n_qt, 1)) * C::BMQ;  // the pair's first tile
    for (int j = 0; ok && j < n; ++j, i0 = (i0 + C::BMQ == i_end) ? i_first : i0 + C::BMQ) {
      const int b = j & 1, slot = j & 1;
      ok = mbar_wait(bar(C::B_STFULL + slot), (j >> 1) & 1, tmo, abort_flag, wc.status) &&
           mbar_wait(bar(C::B_SCFULL + b), (j >> 1) & 1, tmo, abort_flag, wc.status);
      if (!ok) break;
      tc_fence_after();
      const uint32_t chunk = tmem + lane_base + C::sc_col(b) + wg * 32;
      uint32_t sv[32];
      tmem_ld32(chunk, sv);
      tmem_ld_wait();
      const float* st_row = stats + slot * C::BMQ + wg * 32;
      if (pside) {
        // P^T = 2^(S^T scale log2 e - LSE log2 e), masked entries 0
        if (!block_unmasked(s, i0, i0 + C::BMQ, t.k0, t.k0 + kBM)) {
          int lo, hi;
          visible_queries(s, krow, i0 + wg * 32, &lo, &hi);
#pragma unroll
          for (int q = 0; q < 32; ++q)
            sv[q] = (q >= lo && q < hi) ? sv[q] : __float_as_uint(-INFINITY);
        }
        exp2_scores32(sv, c2, st_row, true, 0);  // sv now holds P (fp32)
        uint32_t pp[16], ph[16];
#pragma unroll
        for (int q = 0; q < 32; q += 2) {
          pp[q / 2] = pack2<C::BF16>(__uint_as_float(sv[q]), __uint_as_float(sv[q + 1]));
          ph[q / 2] = pack2<false>(__uint_as_float(sv[q]), __uint_as_float(sv[q + 1]));
        }
        // P^T over the first 16 columns of this chunk: dV may start
        tmem_st16(chunk, pp);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(C::B_READY + b));
          mbar_arrive(bar(C::B_STEMPTY + slot));
        }
        // P (fp16) into the local buffer b once the peer has read its copy of
        // tile j-2 (which also means that copy has finished reading buffer b);
        // the staging warp then sends it
        if (j >= 2) {
          ok = mbar_wait(bar(C::B_PBUF + b), ((j >> 1) - 1) & 1, tmo, abort_flag, wc.status);
          if (!ok) break;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c)
          *reinterpret_cast<uint4*>(smem + pbuf_off(b, c)) =
              make_uint4(ph[4 * c], ph[4 * c + 1], ph[4 * c + 2], ph[4 * c + 3]);
        fence_proxy_async_smem();  // the copy engine reads what this thread wrote
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_STAGED + b));
      } else {
        // dS^T = P^T o (dP^T - D), with P from the peer's buffer b
        ok = mbar_wait_cluster(bar(C::B_PBUF + b), (j >> 1) & 1, tmo, abort_flag, wc.status);
        if (!ok) break;
        // the buffer's phase for tile j has completed: announce tile j+2's bytes
        // (they cannot arrive before every warp has released the buffer below)
        if (poster) {
          seen = j + 1;
          if (j + 2 < n) mbar_arrive_expect_tx(bar(C::B_PBUF + b), C::PBUF);
        }
        uint32_t ph[16];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 x = *reinterpret_cast<const uint4*>(smem + pbuf_off(b, c));
          ph[4 * c] = x.x; ph[4 * c + 1] = x.y; ph[4 * c + 2] = x.z; ph[4 * c + 3] = x.w;
        }
        uint32_t ds[16];
#pragma unroll
        for (int q = 0; q < 32; q += 4) {
          const ulonglong2 nd = *reinterpret_cast<const ulonglong2*>(st_row + q);
#pragma unroll
          for (int e = 0; e < 4; e += 2) {
            const float2 p = unpack2<false>(ph[(q + e) / 2]);
            const uint64_t d = fadd2(f2_pack(__uint_as_float(sv[q + e]), __uint_as_float(sv[q + e + 1])),
                                     e == 0 ? nd.x : nd.y);
            const float2 d2 = f2_unpack(fmul2(d, f2_pack(p.x, p.y)));
            ds[(q + e) / 2] = pack2<C::BF16>(d2.x, d2.y);
          }
        }
        // dS^T over the first 16 columns of this chunk, for dK
        tmem_st16(chunk, ds);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(C::B_READY + b));
          mbar_arrive(bar(C::B_STEMPTY + slot));
          mbar_arrive_peer_relaxed(peer_addr(bar(C::B_PBUF + b), peer));  // the peer's "P buffer b free"
        }
      }
    }
    // --------------------------------------------------------- epilogue
    // dV (P side) or scale dK (dS side): 64-column blocks of the rows dealt
    // over the warpgroups; a block with no query tile stores zeros
    const bool have = n > 0;
    if (ok && have) {
      ok = mbar_wait(bar(C::B_DONE), 0, tmo, abort_flag, wc.status);
      if (ok) tc_fence_after();
    }
    if (ok && C::HALVES == 2 && pair == 1) {
      // pair 1: its fp32 accumulator rows into its own shared memory (16-byte
      // chunks swizzled by the row), read by pair 0 after the cluster barrier
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        const int col = 128 * wg + 16 * c;
        uint32_t v[16];
        if (have) {
          tmem_ld16(tmem + lane_base + C::ACC_COL + col, v);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = 0u;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<uint4*>(smem + r * C::PART_ROW + (((col / 4 + q) ^ (r & 7)) << 4)) =
              make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      }
    } else if (ok && C::HALVES == 1) {
      const int row0 = t.k0 + quarter * 32;
      const int rows_valid = min(32, s.Tkv - row0);
      const int64_t orow = static_cast<int64_t>(t.bg) * s.Tkv + (rows_valid > 0 ? row0 : 0);
      T16* out = reinterpret_cast<T16*>(pside ? dv_out : dk_out) + orow * C::D;
#pragma unroll 1
      for (int task = wg; task < C::D / 64; task += C::NWG)
        store_acc_block<8, C::BF16>(tmem + lane_base + C::ACC_COL + task * 64, have,
                                    pside ? 1.f : scale, out + task * 64, C::D, rows_valid);
    }
  }

  tc_fence_before();
  __syncthreads();
  // neither CTA leaves while its peer may still arrive on its barriers; after
  // it the dS side knows how many P copies the peer issued
  cluster_barrier();
  // after an abort, the dS side lets every copy the peer issued land (bounded)
  // before it can exit (the peer cannot send a buffer whose bytes were not
  // announced: it waits for the buffer to be freed, which comes after)
  if (!pside && warp == 4 && lane == 0 && *abort_flag)
    for (int j = seen; j < *peer_sent; ++j)
      mbar_wait_cluster(bar(C::B_PBUF + (j & 1)), (j >> 1) & 1, wc.drain_cycles, nullptr, wc.status);
  if constexpr (C::HALVES == 2) {
    // pair 0: its accumulator plus pair 1's partial sums (rank r reads rank
    // r + 2, written before the cluster barrier above), scaled, rounded and
    // stored; 16-column chunks, each warpgroup half of the columns
    if (pair == 0 && warp >= 4 && !*abort_flag) {
      const int wg = (warp - 4) >> 2, quarter = warp & 3;
      const int r = quarter * 32 + lane, krow = t.k0 + r;
      const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
      const bool have = n > 0;
      const float mul = pside ? 1.f : scale;
      using T16 = typename std::conditional<C::BF16, __nv_bfloat16, __half>::type;
      T16* out = reinterpret_cast<T16*>(pside ? dv_out : dk_out) +
                 (static_cast<int64_t>(t.bg) * s.Tkv + krow) * C::D;
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        const int col = 128 * wg + 16 * c;
        uint32_t v[16];
        if (have) {
          tmem_ld16(tmem + lane_base + C::ACC_COL + col, v);
          tmem_ld_wait();
        }
        float x[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) x[e] = have ? __uint_as_float(v[e]) : 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 w;
          const uint32_t remote =
              peer_addr(sbase + r * C::PART_ROW + (((col / 4 + q) ^ (r & 7)) << 4), rank + 2u);
          asm volatile("ld.shared::cluster.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w) : "r"(remote));
          x[4 * q] += __uint_as_float(w.x);
          x[4 * q + 1] += __uint_as_float(w.y);
          x[4 * q + 2] += __uint_as_float(w.z);
          x[4 * q + 3] += __uint_as_float(w.w);
        }
        uint32_t o[8];
#pragma unroll
        for (int e = 0; e < 16; e += 2) o[e / 2] = pack2<C::BF16>(x[e] * mul, x[e + 1] * mul);
        if (krow < s.Tkv) {
          reinterpret_cast<uint4*>(out + col)[0] = make_uint4(o[0], o[1], o[2], o[3]);
          reinterpret_cast<uint4*>(out + col)[1] = make_uint4(o[4], o[5], o[6], o[7]);
        }
      }
    }
    // pair 1 keeps its shared memory until pair 0 has read it
    cluster_barrier();
  }
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace fa
