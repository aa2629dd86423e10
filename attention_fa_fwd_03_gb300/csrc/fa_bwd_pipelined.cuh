// Pipelined dK/dV and dQ kernels for head dims up to 128 (128 x 128 tiles).
//
// Same computation as the kernels in fa_bwd.cuh (page "mlx-bun 0.0.4:
// package/src/model/flash-attention.ts", backward passes 2 and 3; page
// "[Metal] Add Flash Attention VJP for training", Implementation Notes: KV-row
// ownership, log2 domain), scheduled so that the tensor core never waits for
// the softmax warps or for tile loads:
//
// * Both score blocks stay 128 x 128: an M=128 tcgen05.mma costs at least
//   ~44 cycles however narrow N is, and N = 128 runs at the full rate. TMEM
//   (512 columns) then holds one score block S, one dP block and the fp32
//   accumulators.
// * The softmax runs in two steps. As soon as S(i) lands it computes
//   P = 2^(S * scale * log2 e - LSE2) into registers (the exponentials, the
//   expensive part), while the tensor core is still busy with the previous
//   tile's accumulating MMAs and this tile's dP. Only dS = P o (dP - D) waits
//   for dP(i); P and dS (16-bit) are then written over the dP columns.
// * dK/dV: P^T is written over the score columns it came from as soon as
//   the exponentials are done, so dV(i) and the next S^T run while dP^T(i)
//   and dS^T are still in progress; dK(i) follows when dS^T(i) is in TMEM:
//     S^T(i+1) after dV(i),  dK(i) after dS^T(i),  dP^T(i+1) after dK(i)
//   dQ: the score columns are free once the softmax has read them, so S(j+1)
//   is issued then; dP alternates between two TMEM blocks, so dP(j+1) need not
//   wait for dQ(j) to read dS(j):  S(j+1)  dP(j+1)  dQ += dS(j) K(j)
// * The operand the next tile needs first (Q in dK/dV, K in dQ) is
//   prefetched three tiles deep, the other two deep, each slot released by
//   the MMA that last reads it.
// * Persistent CTAs: the grid has one CTA per work item (row block of the
//   TileOrder), but a running CTA does not exit after its item: it takes
//   over the next not-yet-started CTA's item through cluster launch control
//   (ItemQueue), so one CTA per SM serves a dynamically balanced stream of
//   items in launch order. Tiles stream through the rings without a break
//   between items, so the next item's first score block is computed while
//   the softmax warps still finish (and store) the previous one; the operand
//   loaded once per item (K, V in dK/dV; Q, dO in dQ) is reloaded as soon as
//   the item's last MMA that reads it completes. The softmax warps store an
//   item's accumulators (dK, dV or dQ) before they release the next item's
//   first P/dS block, which orders the store before that item's first
//   accumulating MMA.
// NWG softmax warpgroups split the 128 columns of every tile (128 / NWG each).
//
// TMEM layout of the 16-bit operands: the score columns are handled in chunks
// of 32 (one per softmax warpgroup); chunk m writes its 16-bit result packed
// into the first 16 columns of the chunk it was read from. dK/dV: P^T into
// S^T chunk m, dS^T into dP^T chunk m (dP^T is read in two 16-column halves,
// each half's 8 result columns landing in columns already read); dQ: dS into
// chunk m of the dP block it came from. So K-block kk of the next MMA reads
// column base + 32 (kk / 2) + 8 (kk % 2).
#pragma once

#include <type_traits>

#include "fa_common.cuh"

namespace fa {

__host__ __device__ constexpr uint32_t chunk_operand_col(uint32_t dp_col, int kk) {
  return dp_col + 32 * (kk >> 1) + 8 * (kk & 1);
}

// p[k] = 2^(s[k] * c + nl[k]) for 32 scores held as raw fp32 bits (in place).
__device__ __forceinline__ void exp2_scores32(uint32_t (&sv)[32], uint64_t c2, const float* nl,
                                              bool per_column_nl, uint64_t nl_row) {
#pragma unroll
  for (int k = 0; k < 32; k += 4) {
    ulonglong2 nl4;
    if (per_column_nl) nl4 = *reinterpret_cast<const ulonglong2*>(nl + k);
#pragma unroll
    for (int e = 0; e < 4; e += 2) {
      const uint64_t add = per_column_nl ? (e == 0 ? nl4.x : nl4.y) : nl_row;
      const float2 x = f2_unpack(
          ffma2(f2_pack(__uint_as_float(sv[k + e]), __uint_as_float(sv[k + e + 1])), c2, add));
      sv[k + e] = __float_as_uint(ex2(x.x));
      sv[k + e + 1] = __float_as_uint(ex2(x.y));
    }
  }
}

// ---------------------------------------------------------------- dK / dV
// One dK/dV work item: a (batch, KV group) and a block of 128 KV rows; its
// tiles are the query tiles (of every head of the group) that see the block,
// numbered head by head. With the item split over the `split` CTAs of a
// cluster, CTA `part` takes the tiles [it0, it0 + n_iter) of that list.
struct DkvItem {
  int bg, b, g, k0, i_lo, n_qt, it0, n_iter;
};

__device__ __forceinline__ DkvItem dkv_item(int linear, const TileOrder& o, const AttnShape& s,
                                            int bmq, int split = 1, int part = 0) {
  DkvItem t;
  int kvt;
  decode_tile(linear, o, &t.bg, &kvt);
  t.b = t.bg / s.Hkv;
  t.g = t.bg - t.b * s.Hkv;
  t.k0 = kvt * kBM;
  int qf, ql;
  query_range(s, t.k0, min(s.Tkv, t.k0 + kBM), &qf, &ql);
  t.i_lo = qf / bmq;
  t.n_qt = max(0, (ql + bmq - 1) / bmq - t.i_lo);
  const int total = t.n_qt * (s.Hq / s.Hkv);
  const int share = (total + split - 1) / split;
  t.it0 = min(total, part * share);
  t.n_iter = min(total, t.it0 + share) - t.it0;
  return t;
}

// SPLIT = 2: each work item's tiles are split between the two CTAs of a
// cluster (for grids with fewer items than half the SMs). Each CTA leaves in
// its shared memory the fp32 partial sums of the half it does not finish
// (CTA 0 its dK, CTA 1 its dV); after a cluster barrier CTA 0 adds CTA 1's dV
// to its own and stores dV, CTA 1 adds CTA 0's dK and stores dK, each through
// distributed shared memory. One item per cluster (no cluster launch control).
template <int D_, bool BF16_, int NWG_, int SPLIT_ = 1>
struct DkvCfg {
  static constexpr int D = D_;
  static constexpr bool BF16 = BF16_;
  static constexpr int SPLIT = SPLIT_;
  static constexpr int NWG = NWG_;          // softmax warpgroups
  static constexpr int CW = 128 / NWG;      // score columns per warpgroup
  static constexpr int QST = 3;             // Q ring: needed first by the next tile
  static constexpr int DST = 2;             // dO ring
  static constexpr int BMQ = 128;           // query rows per inner tile (N of S^T, dP^T)
  static constexpr int DP = (D + 63) / 64 * 64;
  static constexpr int KREG = DP / 64;
  static constexpr int REGION = 128 * 128;  // one 64-column block of a 128-row tile
  static constexpr int TILE = KREG * REGION;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + TILE;
  static constexpr int OFF_Q = OFF_V + TILE;
  static constexpr int OFF_DO = OFF_Q + QST * TILE;
  static constexpr int OFF_STATS = OFF_DO + DST * TILE;  // [2][-lse2 | -dvec][128] fp32
  static constexpr int OFF_BAR = OFF_STATS + 2 * 2 * BMQ * 4;
  // barriers: k_full, k_empty, v_full, v_empty, q_full[QST], q_empty[QST],
  // do_full[DST], do_empty[DST], stats_full[2], stats_empty[2], s_full,
  // ds_ready, dp_full, p_ready, done, drain
  static constexpr int B_KFULL = 0, B_KEMPTY = 1, B_VFULL = 2, B_VEMPTY = 3, B_QFULL = 4,
                       B_QEMPTY = B_QFULL + QST, B_DOFULL = B_QEMPTY + QST,
                       B_DOEMPTY = B_DOFULL + DST, B_STFULL = B_DOEMPTY + DST,
                       B_STEMPTY = B_STFULL + 2, B_SFULL = B_STEMPTY + 2, B_DSREADY = B_SFULL + 1,
                       B_DPFULL = B_SFULL + 2, B_PREADY = B_SFULL + 3, B_DONE = B_SFULL + 4,
                       B_DRAIN = B_SFULL + 5, B_CLCFULL = B_DRAIN + 1,
                       B_CLCEMPTY = B_CLCFULL + kClcSlots, NBAR = B_CLCEMPTY + kClcSlots;
  static constexpr int OFF_CLC = (OFF_BAR + NBAR * 8 + 15) / 16 * 16;  // item responses
  static constexpr int OFF_MISC = OFF_CLC + 16 * kClcSlots;
  static constexpr int SMEM_BYTES = OFF_MISC + 16;  // base must be 1024-aligned (checked)
  static constexpr int THREADS = 128 + 128 * NWG;
  // Registers per thread after the warpgroup split (0: no split); the launch
  // must hold THREADS x launch registers >= REG_NEEDED (checked on the host).
  // Off here: at 64 per thread the producer / MMA / staging code spills, and
  // that costs more than the softmax spills it would remove (measured).
  static constexpr int REG_CTRL = 0, REG_SOFT = 0;
  static constexpr int REG_NEEDED = REG_SOFT > 0 ? 128 * REG_CTRL + 128 * NWG * REG_SOFT : 0;
  static constexpr int S_COL = 0;     // S^T block, 128 fp32 columns
  static constexpr int DP_COL = 128;  // dP^T block, 128 fp32 columns
  static constexpr int DV_COL = 256;
  static constexpr int DK_COL = 256 + D;
  static constexpr uint32_t pt_col(int kk) { return chunk_operand_col(S_COL, kk); }
  static constexpr uint32_t dst_col(int kk) { return chunk_operand_col(DP_COL, kk); }
  static_assert(NWG == 4, "one 32-column chunk per softmax warpgroup");
  static_assert(D <= 128, "dV and dK accumulators share 256 TMEM columns");
  // the half a CTA hands to its peer: 128 rows x D fp32 over the tile buffers
  // (free once the item's MMAs have completed), 16-byte chunks swizzled by row
  static constexpr int PART_ROW = D * 4;
  static_assert(SPLIT == 1 || (SPLIT == 2 && 128 * PART_ROW <= OFF_STATS &&
                               (PART_ROW / 16) % 8 == 0), "partial sums buffer");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

// Persistent (see ItemQueue): every role walks the same item stream and counts
// tiles across items, so the ring slots and barrier phases run on from one
// item to the next.
template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
fa_bwd_dkv_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                  const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                  const float* __restrict__ lse, const float* __restrict__ dvec,
                  void* __restrict__ dk_out, void* __restrict__ dv_out, float scale, AttnShape s,
                  TileOrder order, WaitCfg wc) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {  // the 128-byte swizzle needs 1024-byte aligned tiles
    grid_wait_prior();
    if (threadIdx.x == 0) atomicOr(wc.status, kStatusSmemMisaligned);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  auto bar = [&](int i) { return smem_u32(bars + i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  float* stats = reinterpret_cast<float*>(smem + C::OFF_STATS);
  const uint64_t tmo = wc.timeout_cycles;
  const int reps = s.Hq / s.Hkv;
  const ItemQueue iq{sbase + C::OFF_CLC, bar(C::B_CLCFULL), bar(C::B_CLCEMPTY)};
  // split items: cluster rank and the item of the cluster; otherwise the
  // CTA's first item, later ones through cluster launch control
  const int part = C::SPLIT > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int first_item = C::SPLIT > 1 ? static_cast<int>(blockIdx.x) / C::SPLIT : static_cast<int>(blockIdx.x);
  auto next_item = [&](int k, int* item) {
    if constexpr (C::SPLIT > 1) return false;
    return clc_next(iq, k, lane, item, tmo, abort_flag, wc.status);
  };
  auto item_of = [&](int item) { return dkv_item(item, order, s, C::BMQ, C::SPLIT, part); };

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < C::NBAR; ++i) {
      uint32_t cnt = 1;
      if (i == C::B_STFULL || i == C::B_STFULL + 1) cnt = 32;  // the staging warp's lanes
      if (i == C::B_STEMPTY || i == C::B_STEMPTY + 1 || i == C::B_DSREADY || i == C::B_PREADY)
        cnt = 4 * C::NWG;  // one arrival per softmax warp
      if (i >= C::B_CLCEMPTY && i < C::B_CLCEMPTY + kClcSlots) cnt = C::THREADS / 32;
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
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
  // producer / MMA / staging warpgroup: registers handed to the softmax
  if constexpr (C::REG_SOFT > 0) regs_release<C::REG_CTRL>();
  if (warp == 0 || warp == 2) {
    // ----------------------------------------------------------- producers
    // warp 0: K of each item, then the item's Q ring tiles (and the item
    // requests); warp 2: V, then the dO ring. A tile pair takes ~1.4 us to
    // land under full load, so each ring is refilled the moment its own slot
    // frees. The whole warp runs the loop (a lone active lane whose siblings
    // wait at the final barrier issues far slower); one elected lane issues.
    // Producers wait with try_wait (the warp sleeps in the barrier instead of
    // taking issue slots from the softmax warps of its SM sub-partition); only
    // the MMA issuer polls.
    const bool leader = elect_one_sync();
    const bool q_ring = warp == 0;
    if (leader) tma_prefetch_desc(q_ring ? &map_q : &map_do);
    const int nst = q_ring ? C::QST : C::DST;
    const int full = q_ring ? C::B_QFULL : C::B_DOFULL, empty = q_ring ? C::B_QEMPTY : C::B_DOEMPTY;
    const int once_full = q_ring ? C::B_KFULL : C::B_VFULL, once_empty = q_ring ? C::B_KEMPTY : C::B_VEMPTY;
    const uint32_t ring = sbase + (q_ring ? C::OFF_Q : C::OFF_DO);
    const uint32_t once = sbase + (q_ring ? C::OFF_K : C::OFF_V);
    const CUtensorMap* map = q_ring ? &map_q : &map_do;
    const CUtensorMap* once_map = q_ring ? &map_k : &map_v;
    // Q / dO tiles are read by every KV block of the group: keep them in L2;
    // each K / V block is read once
    const uint64_t pol_ring = l2_policy_evict_last(), pol_once = l2_policy_evict_first();
    int gt = 0, ln = 0, asked = 0;  // ring tiles issued, items with work, item requests
    bool ok = true;
    for (int k = 0, item = first_item; ok; ++k) {
      if (q_ring && C::SPLIT == 1) {
        ok = clc_request(iq, k, leader, tmo, abort_flag, wc.status);
        if (!ok) break;
        ++asked;
      }
      const DkvItem t = item_of(item);
      if (t.n_iter > 0) {
        // K (or V) of this KV block, once its previous contents were last read
        if (ln > 0) ok = mbar_wait(bar(once_empty), (ln - 1) & 1, tmo, abort_flag, wc.status);
        if (!ok) break;
        if (leader) mbar_arrive_expect_tx(bar(once_full), C::TILE);
        for (int r = 0; r < C::KREG; ++r)
          if (leader) tma_load_3d_hint(once + r * C::REGION, once_map, bar(once_full), r * 64, t.k0, t.bg, pol_once);
        ++ln;
        for (int it = 0; it < t.n_iter; ++it, ++gt) {
          const int zq = t.b * s.Hq + t.g * reps + (t.it0 + it) / t.n_qt;
          const int i0 = (t.i_lo + (t.it0 + it) % t.n_qt) * C::BMQ;
          const int st = gt % nst;
          if (gt >= nst) ok = mbar_wait(bar(empty + st), ((gt / nst) - 1) & 1, tmo, abort_flag, wc.status);
          if (!ok) break;
          if (leader) mbar_arrive_expect_tx(bar(full + st), C::TILE);
          for (int r = 0; r < C::KREG; ++r)
            if (leader) tma_load_3d_hint(ring + st * C::TILE + r * C::REGION, map, bar(full + st), r * 64, i0, zq, pol_ring);
        }
        if (!ok) break;
      }
      if (!next_item(k, &item)) break;
    }
    if (*abort_flag) {
      drain_ring(bar(once_full), 1, ln, wc.drain_cycles, wc.status);
      drain_ring(bar(full), nst, gt, wc.drain_cycles, wc.status);
      if (q_ring) drain_ring(iq.full, kClcSlots, asked, wc.drain_cycles, wc.status);
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer
    // the whole warp runs the loop; one elected lane issues
    const bool leader = elect_one_sync();
    constexpr uint32_t ab = C::BF16 ? 1 : 0;
    constexpr uint32_t idesc_st = make_idesc_f16(kBM, C::BMQ, ab, 0, 0);  // S^T, dP^T
    constexpr uint32_t idesc_acc = make_idesc_f16(kBM, C::D, ab, 0, 1);   // dV, dK
    // S^T = K Q^T (into S_COL) or dP^T = V dO^T (into DP_COL): K-major, K = head dim.
    // Descriptors are built once per operand base; the k-step offsets are
    // added to the start-address field (shared addresses < 256 KB never carry).
    auto issue_score = [&](uint32_t a_base, uint32_t b_base, uint32_t col) {
      const uint64_t ad = make_sdesc(a_base, 16, 1024, 2), bd = make_sdesc(b_base, 16, 1024, 2);
#pragma unroll
      for (int kk = 0; kk < C::D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * C::REGION + (kk & 3) * 32;
        if (leader) mma_ss(tmem + col, ad + (off >> 4), bd + (off >> 4), idesc_st, kk > 0);
      }
    };
    auto wait = [&](int b, int parity) {
      return mbar_wait_poll(bar(b), parity & 1, tmo, abort_flag, wc.status);
    };
    int gt = 0, ln = 0;  // tiles before this item, items with work
    bool ok = true;
    for (int k = 0, item = first_item; ok; ++k) {
      const DkvItem t = item_of(item);
      const int n = t.n_iter;
      if (n > 0) {
        // S^T of the item's first tile: its K block and Q(gt) (the score
        // columns were last read by the previous tile's dV, issued before)
        ok = wait(C::B_KFULL, ln) && wait(C::B_QFULL + gt % C::QST, gt / C::QST);
        if (!ok) break;
        tc_fence_after();
        if (leader) issue_score(sbase + C::OFF_K, sbase + C::OFF_Q + (gt % C::QST) * C::TILE, C::S_COL);
        if (leader) mma_commit(bar(C::B_SFULL));
        if (n == 1 && leader) mma_commit(bar(C::B_KEMPTY));  // K read for the last time
        // dP^T of the first tile (over the dS^T columns of the previous tile,
        // whose dK precedes it in issue order)
        ok = wait(C::B_VFULL, ln) && wait(C::B_DOFULL + gt % C::DST, gt / C::DST);
        if (!ok) break;
        tc_fence_after();
        if (leader) issue_score(sbase + C::OFF_V, sbase + C::OFF_DO + (gt % C::DST) * C::TILE, C::DP_COL);
        if (leader) mma_commit(bar(C::B_DPFULL));
        if (n == 1 && leader) mma_commit(bar(C::B_VEMPTY));
        for (int it = 0; it < n; ++it) {
          const int gi = gt + it;
          const int qs = gi % C::QST, ds = gi % C::DST;
          const bool more = it + 1 < n;
          // dV += P^T dO once P^T(it) is in TMEM (A from TMEM, B MN-major, K =
          // query rows); for the item's first tile this also means the softmax
          // warps have stored the previous item's dK, dV. dO(it) is then free.
          ok = wait(C::B_PREADY, gi);
          if (!ok) break;
          tc_fence_after();
          const uint64_t ddesc = make_sdesc(sbase + C::OFF_DO + ds * C::TILE, C::REGION, 1024, 2);
#pragma unroll
          for (int kk = 0; kk < C::BMQ / 16; ++kk)
            if (leader) mma_ts(tmem + C::DV_COL, tmem + C::pt_col(kk), ddesc + ((kk * 16 * 128) >> 4),
                               idesc_acc, (it > 0 || kk > 0) ? 1u : 0u);
          if (leader) mma_commit(bar(C::B_DOEMPTY + ds));
          if (more) {
            // next S^T over the P^T columns dV has just read (in issue order)
            const int nq = (gi + 1) % C::QST;
            ok = wait(C::B_QFULL + nq, (gi + 1) / C::QST);
            if (!ok) break;
            tc_fence_after();
            if (leader) issue_score(sbase + C::OFF_K, sbase + C::OFF_Q + nq * C::TILE, C::S_COL);
            if (leader) mma_commit(bar(C::B_SFULL));
            if (it + 2 == n && leader) mma_commit(bar(C::B_KEMPTY));
          }
          // dK += dS^T Q once dS^T(it) is in TMEM; Q(it) is then free
          ok = wait(C::B_DSREADY, gi);
          if (!ok) break;
          tc_fence_after();
          const uint64_t qdesc = make_sdesc(sbase + C::OFF_Q + qs * C::TILE, C::REGION, 1024, 2);
#pragma unroll
          for (int kk = 0; kk < C::BMQ / 16; ++kk)
            if (leader) mma_ts(tmem + C::DK_COL, tmem + C::dst_col(kk), qdesc + ((kk * 16 * 128) >> 4),
                               idesc_acc, (it > 0 || kk > 0) ? 1u : 0u);
          if (leader) mma_commit(bar(C::B_QEMPTY + qs));
          if (more) {
            // dP^T(it+1) over the dS^T columns dK has just read (in issue order)
            const int nd = (gi + 1) % C::DST;
            ok = wait(C::B_DOFULL + nd, (gi + 1) / C::DST);
            if (!ok) break;
            tc_fence_after();
            if (leader) issue_score(sbase + C::OFF_V, sbase + C::OFF_DO + nd * C::TILE, C::DP_COL);
            if (leader) mma_commit(bar(C::B_DPFULL));
            if (it + 2 == n && leader) mma_commit(bar(C::B_VEMPTY));
          }
        }
        if (!ok) break;
        if (leader) mma_commit(bar(C::B_DONE));  // the item's dK, dV are final
        gt += n;
        ++ln;
      }
      if (!next_item(k, &item)) break;
    }
    // every issued MMA completes before the CTA exits
    if (leader) mma_commit(bar(C::B_DRAIN));
    mbar_wait(bar(C::B_DRAIN), 0, wc.drain_cycles, nullptr, wc.status);
  } else if (warp == 3) {
    // ------------------------------------------- LSE / D-vector staging
    // a flat stream over the tiles of the CTA's items; each lane loads its
    // four rows of the next tile into registers before waiting for that
    // tile's slot, so the global-load latency hides behind the wait
    int k = 0, item = first_item, it = 0;
    DkvItem t = item_of(item);
    auto advance = [&]() {  // to the next tile with work; false at the end
      while (it >= t.n_iter) {
        if (!next_item(k, &item)) return false;
        ++k;
        t = item_of(item);
        it = 0;
      }
      return true;
    };
    constexpr int RPL = C::BMQ / 32;  // rows per lane
    float L[RPL], Dv[RPL];
    auto load = [&]() {
      const int h = t.g * reps + (t.it0 + it) / t.n_qt;
      const int i0 = (t.i_lo + (t.it0 + it) % t.n_qt) * C::BMQ;
      const int64_t base = static_cast<int64_t>(t.b * s.Hq + h) * s.Tq;
#pragma unroll
      for (int r = 0; r < RPL; ++r) {
        const int i = i0 + lane + 32 * r;
        L[r] = -INFINITY;  // rows past Tq: P = 0
        Dv[r] = 0.f;
        if (i < s.Tq) {
          L[r] = lse[base + i];
          Dv[r] = dvec[base + i];
        }
      }
    };
    bool have = advance();
    if (have) load();
    for (int gt = 0; have; ++gt) {
      const int slot = gt & 1;
      if (gt >= 2 &&
          !mbar_wait(bar(C::B_STEMPTY + slot), ((gt >> 1) - 1) & 1, tmo, abort_flag, wc.status))
        break;
      float* dst = stats + slot * 2 * C::BMQ;
#pragma unroll
      for (int r = 0; r < RPL; ++r) {
        // -LSE * log2(e) (a row with no visible key: P = 0) and -D
        dst[lane + 32 * r] = (L[r] == -INFINITY) ? -INFINITY : -L[r] * kLog2e;
        dst[C::BMQ + lane + 32 * r] = -Dv[r];
      }
      mbar_arrive(bar(C::B_STFULL + slot));
      ++it;
      have = advance();
      if (have) load();
    }
  }
  } else {
    if constexpr (C::REG_SOFT > 0) regs_claim<C::REG_SOFT>();
    // ------------------------------------------- softmax: P^T and dS^T
    const int wg = (warp - 4) >> 2;             // query columns [32 wg, 32 wg + 32)
    const int quarter = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint64_t c2 = f2_pack(s.scale_log2, s.scale_log2);
    const uint32_t col = C::DP_COL + wg * C::CW;  // this warpgroup's dP^T chunk
    using T16 = typename std::conditional<C::BF16, __nv_bfloat16, __half>::type;
    int gt = 0, ln = 0;
    bool ok = true;
    for (int k = 0, item = first_item; ok; ++k) {
      const DkvItem t = item_of(item);
      const int krow = t.k0 + quarter * 32 + lane;  // KV row of this thread (TMEM lane)
      const int i_first = t.i_lo * C::BMQ, i_end = (t.i_lo + t.n_qt) * C::BMQ;
      // query tile of this step: the heads of the group in turn
      int i0 = t.n_qt > 0 ? (t.i_lo + t.it0 % t.n_qt) * C::BMQ : i_first;
      for (int it = 0; it < t.n_iter; ++it, i0 = (i0 + C::BMQ == i_end) ? i_first : i0 + C::BMQ) {
        const int gi = gt + it;
        const int slot = gi & 1;
        ok = mbar_wait(bar(C::B_STFULL + slot), (gi >> 1) & 1, tmo, abort_flag, wc.status) &&
             mbar_wait(bar(C::B_SFULL), gi & 1, tmo, abort_flag, wc.status);
        if (!ok) break;
        tc_fence_after();
        uint32_t sv[32];
        const uint32_t s_chunk = tmem + lane_base + C::S_COL + wg * C::CW;
        tmem_ld32(s_chunk, sv);
        tmem_ld_wait();
        const float* nl_s = stats + slot * 2 * C::BMQ + wg * C::CW;  // -LSE * log2(e)
        const float* nd_s = nl_s + C::BMQ;                           // -D
        if (!block_unmasked(s, i0, i0 + C::BMQ, t.k0, t.k0 + kBM)) {
          int lo, hi;
          visible_queries(s, krow, i0 + wg * C::CW, &lo, &hi);
#pragma unroll
          for (int q = 0; q < 32; ++q)
            sv[q] = (q >= lo && q < hi) ? sv[q] : __float_as_uint(-INFINITY);
        }
        exp2_scores32(sv, c2, nl_s, true, 0);  // sv now holds P (fp32)
        {
          // P^T (16-bit) over this chunk's S^T columns, for dV right away
          uint32_t pp[16];
#pragma unroll
          for (int q = 0; q < 32; q += 2)
            pp[q / 2] = pack2<C::BF16>(__uint_as_float(sv[q]), __uint_as_float(sv[q + 1]));
          tmem_st16(s_chunk, pp);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(C::B_PREADY));
        }
        // dS^T = P^T o (dP^T - D) once dP^T(it) is in TMEM
        ok = mbar_wait(bar(C::B_DPFULL), gi & 1, tmo, abort_flag, wc.status);
        if (!ok) break;
        tc_fence_after();
        // two 16-column halves: load dP^T, then write 8 columns of dS^T into
        // columns already read
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t pv[16], w[8];
          tmem_ld16(tmem + lane_base + col + 16 * h, pv);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 16; k += 4) {
            const ulonglong2 nd = *reinterpret_cast<const ulonglong2*>(nd_s + 16 * h + k);
#pragma unroll
            for (int e = 0; e < 4; e += 2) {
              const int q = 16 * h + k + e;
              const uint64_t p2 = f2_pack(__uint_as_float(sv[q]), __uint_as_float(sv[q + 1]));
              const uint64_t d = fadd2(
                  f2_pack(__uint_as_float(pv[k + e]), __uint_as_float(pv[k + e + 1])),
                  e == 0 ? nd.x : nd.y);
              const float2 d2 = f2_unpack(fmul2(d, p2));
              w[(k + e) / 2] = pack2<C::BF16>(d2.x, d2.y);
            }
          }
          tmem_st8(tmem + lane_base + col + 8 * h, w);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(C::B_DSREADY));
          mbar_arrive(bar(C::B_STEMPTY + slot));
        }
      }
      if (!ok) break;
      // ----------------------------------------------------- item epilogue
      // 16-column chunks of the dV then dK row (dK scaled), dealt round-robin
      // over the softmax warpgroups; one row per thread. The accumulators are
      // free again once every softmax warp has passed here (their next P/dS
      // arrival orders it before the next item's first accumulating MMA).
      const bool have = t.n_iter > 0;
      if (have) {
        ok = mbar_wait(bar(C::B_DONE), ln & 1, tmo, abort_flag, wc.status);
        if (!ok) break;
        tc_fence_after();
      }
      if constexpr (C::SPLIT > 1) {
        // the half the peer finishes (CTA 0: dK, CTA 1: dV) to this CTA's own
        // shared memory (the tile buffers are free: the item's MMAs have
        // completed); the peer adds it after the cluster barrier at the end
        {
          const int row = quarter * 32 + lane;
          const uint32_t half = part == 0 ? C::DK_COL : C::DV_COL;
#pragma unroll 1
          for (int c = wg; c < C::D / 16; c += C::NWG) {  // 16-column chunks
            uint32_t v[16];
            if (have) {
              tmem_ld16(tmem + lane_base + half + 16 * c, v);
              tmem_ld_wait();
            } else {
#pragma unroll
              for (int e = 0; e < 16; ++e) v[e] = 0u;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q)
              *reinterpret_cast<uint4*>(smem + row * C::PART_ROW + (((4 * c + q) ^ (row & 7)) << 4)) =
                  make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
          }
        }
        if (have) {
          tc_fence_before();
          gt += t.n_iter;
          ++ln;
        }
        break;  // one item per cluster
      }
      // blocks of W columns of [dV | dK] dealt round-robin over the warps of
      // this lane quarter
      constexpr int S = (C::D % 64 == 0 && 2 * C::D / 64 >= C::NWG) ? 8 : 4, W = 8 * S;
      const int row0 = t.k0 + quarter * 32;
      const int rows_valid = min(32, s.Tkv - row0);
      const int64_t orow = static_cast<int64_t>(t.bg) * s.Tkv + (rows_valid > 0 ? row0 : 0);
#pragma unroll 1
      for (int task = wg; task < 2 * C::D / W; task += C::NWG) {
        const bool is_dk = task * W >= C::D;
        const int cc = is_dk ? task * W - C::D : task * W;
        T16* dst = reinterpret_cast<T16*>(is_dk ? dk_out : dv_out) + orow * C::D + cc;
        store_acc_block<S, C::BF16>(tmem + lane_base + (is_dk ? C::DK_COL : C::DV_COL) + cc, have,
                                    is_dk ? scale : 1.f, dst, C::D, rows_valid);
      }
      if (have) {
        tc_fence_before();
        gt += t.n_iter;
        ++ln;
      }
      if (!next_item(k, &item)) break;
    }
  }

  if constexpr (C::SPLIT > 1) {
    // every thread of both CTAs: each CTA's half for its peer is in its shared
    // memory
    cluster_barrier();
    if (warp >= 4 && !*abort_flag) {
      // CTA 0: dV, CTA 1: dK (scaled) — its own accumulator plus the peer's
      // partial sums, rounded and stored; 16-column chunks dealt over the
      // softmax warpgroups
      const DkvItem t = item_of(first_item);
      const int wg = (warp - 4) >> 2, quarter = warp & 3;
      const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
      const int row = quarter * 32 + lane, krow = t.k0 + row;
      const bool have = t.n_iter > 0;
      using T16 = typename std::conditional<C::BF16, __nv_bfloat16, __half>::type;
      const bool is_dk = part == 1;
#pragma unroll 1
      for (int c = wg; c < C::D / 16; c += C::NWG) {
        uint32_t v[16];
        if (have) {
          tc_fence_after();
          tmem_ld16(tmem + lane_base + (is_dk ? C::DK_COL : C::DV_COL) + 16 * c, v);
          tmem_ld_wait();
        }
        float x[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 w;
          const uint32_t remote =
              peer_addr(sbase + row * C::PART_ROW + (((4 * c + q) ^ (row & 7)) << 4), part ^ 1);
          asm volatile("ld.shared::cluster.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w) : "r"(remote));
          x[4 * q] = __uint_as_float(w.x);
          x[4 * q + 1] = __uint_as_float(w.y);
          x[4 * q + 2] = __uint_as_float(w.z);
          x[4 * q + 3] = __uint_as_float(w.w);
        }
        const float mul = is_dk ? scale : 1.f;
        uint32_t o[8];
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          const float a = (have ? __uint_as_float(v[e]) : 0.f) + x[e];
          const float b2 = (have ? __uint_as_float(v[e + 1]) : 0.f) + x[e + 1];
          o[e / 2] = pack2<C::BF16>(a * mul, b2 * mul);
        }
        if (krow < s.Tkv) {
          T16* dst = reinterpret_cast<T16*>(is_dk ? dk_out : dv_out) +
                     (static_cast<int64_t>(t.bg) * s.Tkv + krow) * C::D + 16 * c;
          reinterpret_cast<uint4*>(dst)[0] = make_uint4(o[0], o[1], o[2], o[3]);
          reinterpret_cast<uint4*>(dst)[1] = make_uint4(o[4], o[5], o[6], o[7]);
        }
      }
    }
    // each CTA keeps its shared memory until the peer has read it
    cluster_barrier();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// --------------------------------------------------------------------- dQ
// One dQ work item: a (batch, head) and a block of 128 query rows; its tiles
// are the key tiles the block sees.
struct DqItem {
  int bh, b, g, q0, j_lo, n_iter;
};

__device__ __forceinline__ DqItem dq_item(int linear, const TileOrder& o, const AttnShape& s,
                                          int bn) {
  DqItem t;
  int qt;
  decode_tile(linear, o, &t.bh, &qt);
  t.b = t.bh / s.Hq;
  t.g = (t.bh - t.b * s.Hq) / (s.Hq / s.Hkv);
  t.q0 = qt * kBM;
  int kf, kl;
  key_range(s, t.q0, min(s.Tq, t.q0 + kBM), &kf, &kl);
  t.j_lo = kf / bn;
  t.n_iter = max(0, (kl + bn - 1) / bn - t.j_lo);
  return t;
}

// Tile configuration of the dQ kernel. BN key rows per tile (N of S and dP),
// NWG softmax warpgroups of 32 key columns each, K / V rings of KST / VST
// tiles, and where Q sits:
//  * D <= 128: Q and dO in shared memory, 128-key tiles, four warpgroups,
//    rings 3 / 2, two dP blocks in TMEM.
//  * D = 256 (QTM): the dQ accumulator takes 256 TMEM columns and a 128-row
//    Q or dO tile 64 KB of shared memory. Q is kept in TMEM instead, as the A
//    operand of S = Q K^T (the softmax warps write each item's Q rows there),
//    which leaves shared memory for dO and 64-key K / V rings of 3 / 2 tiles.
//    TMEM then holds two 64-column score blocks, Q and dQ (128 + 128 + 256
//    columns): tile j computes S into block j % 2, and dP into the same block
//    once the softmax has read S from it.
template <int D_, bool BF16_, int NWG_, int BN_ = 128, int KST_ = 3, int VST_ = 2,
          bool QTM_ = false>
struct DqCfg {
  static constexpr int D = D_;
  static constexpr bool BF16 = BF16_;
  static constexpr int NWG = NWG_;
  static constexpr int BN = BN_;        // key rows per tile (N of S, dP)
  static constexpr int CW = BN / NWG;   // key columns per softmax warpgroup
  static constexpr int KST = KST_;      // K ring: needed first by the next tile
  static constexpr int VST = VST_;      // V ring
  static constexpr bool QTM = QTM_;     // Q in TMEM (A operand of S from TMEM)
  static constexpr int DP = (D + 63) / 64 * 64;
  static constexpr int KREG = DP / 64;
  static constexpr int Q_REGION = 128 * 128;   // one 64-column block of a 128-row Q / dO tile
  static constexpr int KV_REGION = BN * 128;   // one 64-column block of a K / V tile
  static constexpr int Q_TILE = KREG * Q_REGION;
  static constexpr int KV_TILE = KREG * KV_REGION;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = OFF_Q + (QTM ? 0 : Q_TILE);
  static constexpr int OFF_K = OFF_DO + Q_TILE;
  static constexpr int OFF_V = OFF_K + KST * KV_TILE;
  static constexpr int OFF_BAR = OFF_V + VST * KV_TILE;
  // barriers: q_full, q_empty, do_full, do_empty, k_full[KST], k_empty[KST],
  // v_full[VST], v_empty[VST], s_full[2], s_free, dp_full[2], p_full[2], done,
  // drain.
  // * p_full alternates with the tile's parity: with Q in shared memory, S and
  //   dP of tile j+1 are issued before the MMA waits for dS(j), so one softmax
  //   warp can finish tile j+1 while another still works on tile j; with a
  //   single barrier its second arrival would complete tile j's phase early.
  //   Two tiles ahead is impossible (S(j+2) waits for every warp's s_free of
  //   tile j+1).
  // * s_full[1] is used with Q in TMEM only, where S alternates between two
  //   blocks: S(j+1) may complete before a slow softmax warp has waited for
  //   S(j), so each block has its own barrier (S(j+2) waits for that warp's
  //   dS(j)). s_free then gates dP(j), which goes into S(j)'s block.
  // * With Q in TMEM, q_full counts one arrival per softmax warp (the warps
  //   that write Q there) and q_empty is unused.
  static constexpr int B_QFULL = 0, B_QEMPTY = 1, B_DOFULL = 2, B_DOEMPTY = 3, B_KFULL = 4,
                       B_KEMPTY = B_KFULL + KST, B_VFULL = B_KEMPTY + KST,
                       B_VEMPTY = B_VFULL + VST, B_SFULL = B_VEMPTY + VST,
                       B_SFREE = B_SFULL + 2, B_DPFULL = B_SFULL + 3, B_PFULL = B_SFULL + 5,
                       B_DONE = B_SFULL + 7, B_DRAIN = B_DONE + 1,
                       B_CLCFULL = B_DRAIN + 1, B_CLCEMPTY = B_CLCFULL + kClcSlots,
                       NBAR = B_CLCEMPTY + kClcSlots;
  static constexpr int OFF_CLC = (OFF_BAR + NBAR * 8 + 15) / 16 * 16;  // item responses
  static constexpr int OFF_MISC = OFF_CLC + 16 * kClcSlots;
  static constexpr int SMEM_BYTES = OFF_MISC + 16;  // base must be 1024-aligned (checked)
  static constexpr int THREADS = 128 + 128 * NWG;
  // Registers per thread after the warpgroup split (0: no split); the launch
  // must hold THREADS x launch registers >= REG_NEEDED (checked on the host).
  // Four softmax warpgroups (640 threads) get 104 registers each from the
  // producer / MMA warpgroup's 64; with two (384 threads) every thread has
  // enough at launch.
  static constexpr int REG_CTRL = NWG == 4 ? 64 : 0, REG_SOFT = NWG == 4 ? 104 : 0;
  static constexpr int REG_NEEDED = REG_SOFT > 0 ? 128 * REG_CTRL + 128 * NWG * REG_SOFT : 0;
  // TMEM. Q in shared memory: S at 0, dP blocks at BN and 2 BN (tile j uses
  // dp block j % 2). Q in TMEM: blocks at 0 and BN, tile j uses block j % 2
  // for S and then dP; Q (16-bit pairs, DP / 2 columns) after them.
  static constexpr int QT_COL = 2 * BN;
  static constexpr int DQ_COL = 512 - DP;  // one dQ accumulator
  static constexpr uint32_t s_col(int b) { return QTM ? BN * b : 0; }
  static constexpr uint32_t dp_col(int b) { return QTM ? BN * b : BN + BN * b; }
  static constexpr uint32_t ds_col(int b, int kk) { return chunk_operand_col(dp_col(b), kk); }
  static_assert(CW == 32, "one 32-column chunk per softmax warpgroup");
  static_assert((QTM ? 2 * BN + DP / 2 : 3 * BN) <= DQ_COL,
                "score blocks, Q and dQ in 512 TMEM columns");
  static_assert(!QTM || (DP / 2) % (32 * NWG) == 0, "Q columns split evenly over the warpgroups");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

// Pipelined dQ. dP alternates between two TMEM blocks, so dP(j+1) is computed
// while the softmax still turns dP(j) into dS(j), and the tensor core runs
// S(j+1), dP(j+1), dQ(j) without waiting for dQ(j) to read dS. With Q in TMEM
// the score of tile j+1 shares its block with dP(j+1): S(j+1) goes there after
// dQ(j-1) has read the block (issue order), and dP(j+1) once the softmax has
// read S(j+1). The item's dQ store is ordered before the next item's first dQ
// by the softmax warps' next dS arrival (as in dK/dV). Persistent like the
// dK/dV kernel above.
template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                 const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                 const void* __restrict__ q_rows, const float* __restrict__ lse,
                 const float* __restrict__ dvec, void* __restrict__ dq_out, float scale,
                 AttnShape s, TileOrder order, WaitCfg wc, int overlap_prior) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {  // the 128-byte swizzle needs 1024-byte aligned tiles
    grid_wait_prior();
    if (threadIdx.x == 0) atomicOr(wc.status, kStatusSmemMisaligned);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  auto bar = [&](int i) { return smem_u32(bars + i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const uint64_t tmo = wc.timeout_cycles;
  const ItemQueue iq{sbase + C::OFF_CLC, bar(C::B_CLCFULL), bar(C::B_CLCEMPTY)};

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < C::NBAR; ++i) {
      uint32_t cnt = 1;
      if (i == C::B_PFULL || i == C::B_PFULL + 1 || i == C::B_SFREE)
        cnt = 4 * C::NWG;  // one arrival per softmax warp
      if (C::QTM && i == C::B_QFULL) cnt = 4 * C::NWG;
      if (i >= C::B_CLCEMPTY && i < C::B_CLCEMPTY + kClcSlots) cnt = C::THREADS / 32;
      mbar_init(bar(i), cnt);
    }
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  // overlap_prior: the previous grid is the dK/dV launch of the same backward,
  // which reads nothing this grid writes and writes nothing it reads, and
  // which this grid follows only once every CTA of it has passed its own wait
  // for the D-vector. Then the grid starts at once, filling the SMs dK/dV
  // leaves idle or frees, and waits for it at exit instead, so its completion
  // still implies that of every grid before it.
  if (!overlap_prior) grid_wait_prior();
  grid_release_next();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
  // producer / MMA warpgroup: registers handed to the softmax
  if constexpr (C::REG_SOFT > 0) regs_release<C::REG_CTRL>();
  if (warp == 3) {
    // ------------------------------------------ producer: Q (unless in TMEM), dO
    // once per item, each as soon as the previous item's last MMA reading it
    // (its last S, its last dP) completes; read once, so not kept in L2
    const bool leader = elect_one_sync();
    const uint64_t pol_once = l2_policy_evict_first();
    int ln = 0, nq = 0, ndo = 0;  // items with work; Q, dO loads issued
    bool ok = true;
    for (int k = 0, item = blockIdx.x; ok; ++k) {
      const DqItem t = dq_item(item, order, s, C::BN);
      if (t.n_iter > 0) {
        if constexpr (!C::QTM) {
          if (ln > 0) ok = mbar_wait(bar(C::B_QEMPTY), (ln - 1) & 1, tmo, abort_flag, wc.status);
          if (!ok) break;
          if (leader) mbar_arrive_expect_tx(bar(C::B_QFULL), C::Q_TILE);
          for (int r = 0; r < C::KREG; ++r)
            if (leader) tma_load_3d_hint(sbase + C::OFF_Q + r * C::Q_REGION, &map_q, bar(C::B_QFULL), r * 64, t.q0, t.bh, pol_once);
          ++nq;
        }
        if (ln > 0) ok = mbar_wait(bar(C::B_DOEMPTY), (ln - 1) & 1, tmo, abort_flag, wc.status);
        if (!ok) break;
        if (leader) mbar_arrive_expect_tx(bar(C::B_DOFULL), C::Q_TILE);
        for (int r = 0; r < C::KREG; ++r)
          if (leader) tma_load_3d_hint(sbase + C::OFF_DO + r * C::Q_REGION, &map_do, bar(C::B_DOFULL), r * 64, t.q0, t.bh, pol_once);
        ++ndo;
        ++ln;
      }
      if (!clc_next(iq, k, lane, &item, tmo, abort_flag, wc.status)) break;
    }
    if (*abort_flag) {
      if (!C::QTM) drain_ring(bar(C::B_QFULL), 1, nq, wc.drain_cycles, wc.status);
      drain_ring(bar(C::B_DOFULL), 1, ndo, wc.drain_cycles, wc.status);
    }
  } else if (warp == 0 || warp == 2) {
    // ------------------------------------------- producers: K ring, V ring
    // each refilled the moment its own slot frees (warp 0 also requests the
    // items); the whole warp runs the loop, one elected lane issues
    const bool leader = elect_one_sync();
    const bool k_ring = warp == 0;
    if (leader) tma_prefetch_desc(k_ring ? &map_k : &map_v);
    const int nst = k_ring ? C::KST : C::VST;
    const int full = k_ring ? C::B_KFULL : C::B_VFULL, empty = k_ring ? C::B_KEMPTY : C::B_VEMPTY;
    const uint32_t ring = sbase + (k_ring ? C::OFF_K : C::OFF_V);
    const CUtensorMap* map = k_ring ? &map_k : &map_v;
    // K / V tiles are read by every query block of the group's heads: keep
    // them in L2
    const uint64_t pol_ring = l2_policy_evict_last();
    int gt = 0, asked = 0;
    bool ok = true;
    for (int k = 0, item = blockIdx.x; ok; ++k) {
      if (k_ring) {
        ok = clc_request(iq, k, leader, tmo, abort_flag, wc.status);
        if (!ok) break;
        ++asked;
      }
      const DqItem t = dq_item(item, order, s, C::BN);
      const int zkv = t.b * s.Hkv + t.g;
      for (int it = 0; it < t.n_iter; ++it, ++gt) {
        const int kr = (t.j_lo + it) * C::BN;
        const int st = gt % nst;
        if (gt >= nst) ok = mbar_wait(bar(empty + st), ((gt / nst) - 1) & 1, tmo, abort_flag, wc.status);
        if (!ok) break;
        if (leader) mbar_arrive_expect_tx(bar(full + st), C::KV_TILE);
        for (int r = 0; r < C::KREG; ++r)
          if (leader) tma_load_3d_hint(ring + st * C::KV_TILE + r * C::KV_REGION, map, bar(full + st), r * 64, kr, zkv, pol_ring);
      }
      if (!ok) break;
      if (!clc_next(iq, k, lane, &item, tmo, abort_flag, wc.status)) break;
    }
    if (*abort_flag) {
      drain_ring(bar(full), nst, gt, wc.drain_cycles, wc.status);
      if (k_ring) drain_ring(iq.full, kClcSlots, asked, wc.drain_cycles, wc.status);
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer
    const bool leader = elect_one_sync();
    constexpr uint32_t ab = C::BF16 ? 1 : 0;
    constexpr uint32_t idesc_s = make_idesc_f16(kBM, C::BN, ab, 0, 0);
    constexpr uint32_t idesc_q = make_idesc_f16(kBM, C::D, ab, 0, 1);
    // score block = A B^T, K = head dim: A (Q or dO) K-major from shared memory
    auto issue_score = [&](uint32_t a_base, uint32_t b_base, uint32_t col) {
      const uint64_t ad = make_sdesc(a_base, 16, 1024, 2), bd = make_sdesc(b_base, 16, 1024, 2);
#pragma unroll
      for (int kk = 0; kk < C::D / 16; ++kk) {
        const uint32_t off_a = (kk >> 2) * C::Q_REGION + (kk & 3) * 32;
        const uint32_t off_b = (kk >> 2) * C::KV_REGION + (kk & 3) * 32;
        if (leader) mma_ss(tmem + col, ad + (off_a >> 4), bd + (off_b >> 4), idesc_s, kk > 0);
      }
    };
    // S(gi) = Q K^T into its block, with Q from TMEM (QTM) or shared memory
    auto issue_s = [&](int gi) {
      const uint32_t k_base = sbase + C::OFF_K + (gi % C::KST) * C::KV_TILE;
      if constexpr (C::QTM) {
        const uint64_t bd = make_sdesc(k_base, 16, 1024, 2);
#pragma unroll
        for (int kk = 0; kk < C::D / 16; ++kk) {
          const uint32_t off_b = (kk >> 2) * C::KV_REGION + (kk & 3) * 32;
          if (leader) mma_ts(tmem + C::s_col(gi & 1), tmem + C::QT_COL + 8 * kk, bd + (off_b >> 4), idesc_s, kk > 0);
        }
      } else {
        issue_score(sbase + C::OFF_Q, k_base, C::s_col(gi & 1));
      }
    };
    auto wait = [&](int b, int parity) {
      return mbar_wait_poll(bar(b), parity & 1, tmo, abort_flag, wc.status);
    };
    // dQ += dS K   (dS from TMEM, K as MN-major B, K = key rows)
    auto issue_dq = [&](int gi, int it) {
      const uint64_t kdesc = make_sdesc(sbase + C::OFF_K + (gi % C::KST) * C::KV_TILE, C::KV_REGION, 1024, 2);
#pragma unroll
      for (int kk = 0; kk < C::BN / 16; ++kk)
        if (leader) mma_ts(tmem + C::DQ_COL, tmem + C::ds_col(gi & 1, kk), kdesc + ((kk * 16 * 128) >> 4), idesc_q,
                           (it > 0 || kk > 0) ? 1u : 0u);
      if (leader) mma_commit(bar(C::B_KEMPTY + gi % C::KST));
    };
    // dP(gi) into its block; V is read by dP only
    auto issue_dp = [&](int gi) {
      issue_score(sbase + C::OFF_DO, sbase + C::OFF_V + (gi % C::VST) * C::KV_TILE, C::dp_col(gi & 1));
      if (leader) mma_commit(bar(C::B_DPFULL + (gi & 1)));
      if (leader) mma_commit(bar(C::B_VEMPTY + gi % C::VST));
    };
    int gt = 0, ln = 0;
    bool ok = true;
    for (int k = 0, item = blockIdx.x; ok; ++k) {
      const DqItem t = dq_item(item, order, s, C::BN);
      const int n = t.n_iter;
      if (n > 0) {
        // S of the item's first tile: its Q, K(gt), and (Q in shared memory)
        // the softmax done reading the previous S
        ok = wait(C::B_QFULL, ln) && wait(C::B_KFULL + gt % C::KST, gt / C::KST) &&
             (C::QTM || gt == 0 || wait(C::B_SFREE, gt - 1));
        if (!ok) break;
        tc_fence_after();
        issue_s(gt);
        if (leader) mma_commit(bar(C::B_SFULL + (C::QTM ? (gt & 1) : 0)));
        if (!C::QTM && n == 1 && leader) mma_commit(bar(C::B_QEMPTY));  // Q read for the last time
        // dP of the first tile (its block's dS of the previous item was read
        // by a dQ issued before; with Q in TMEM, once S(gt) was read from it)
        ok = wait(C::B_DOFULL, ln) && wait(C::B_VFULL + gt % C::VST, gt / C::VST) &&
             (!C::QTM || wait(C::B_SFREE, gt));
        if (!ok) break;
        tc_fence_after();
        issue_dp(gt);
        if (n == 1 && leader) mma_commit(bar(C::B_DOEMPTY));
        for (int it = 0; it < n; ++it) {
          const int gi = gt + it;
          const bool more = it + 1 < n;
          if (more) {
            // S(it+1): with Q in shared memory over the S block the softmax has
            // read; with Q in TMEM into the block dQ(it-1) has read (issue order)
            const int nk = (gi + 1) % C::KST;
            ok = wait(C::B_KFULL + nk, (gi + 1) / C::KST) && (C::QTM || wait(C::B_SFREE, gi));
            if (!ok) break;
            tc_fence_after();
            issue_s(gi + 1);
            if (leader) mma_commit(bar(C::B_SFULL + (C::QTM ? ((gi + 1) & 1) : 0)));
            if (!C::QTM && it + 2 == n && leader) mma_commit(bar(C::B_QEMPTY));
            if constexpr (!C::QTM) {
              // dP(it+1) into the other block (its dS(it-1) was read by dQ(it-1))
              const int nv = (gi + 1) % C::VST;
              ok = wait(C::B_VFULL + nv, (gi + 1) / C::VST);
              if (!ok) break;
              tc_fence_after();
              issue_dp(gi + 1);
              if (it + 2 == n && leader) mma_commit(bar(C::B_DOEMPTY));
            }
          }
          // dS(it) in TMEM; for the item's first tile this also means the
          // softmax warps have stored the previous item's dQ
          ok = wait(C::B_PFULL + (gi & 1), gi >> 1);
          if (!ok) break;
          tc_fence_after();
          issue_dq(gi, it);
          if (C::QTM && more) {
            // dP(it+1) into S(it+1)'s block once the softmax has read S(it+1)
            // (it does while dQ(it) runs); the issuing thread blocks while the
            // tensor core works through a batch, so dQ(it) goes first
            const int nv = (gi + 1) % C::VST;
            ok = wait(C::B_VFULL + nv, (gi + 1) / C::VST) && wait(C::B_SFREE, gi + 1);
            if (!ok) break;
            tc_fence_after();
            issue_dp(gi + 1);
            if (it + 2 == n && leader) mma_commit(bar(C::B_DOEMPTY));
          }
        }
        if (!ok) break;
        if (leader) mma_commit(bar(C::B_DONE));  // this item's dQ is final
        gt += n;
        ++ln;
      }
      if (!clc_next(iq, k, lane, &item, tmo, abort_flag, wc.status)) break;
    }
    // every issued MMA completes before the CTA exits
    if (leader) mma_commit(bar(C::B_DRAIN));
    mbar_wait(bar(C::B_DRAIN), 0, wc.drain_cycles, nullptr, wc.status);
  }
  } else {
    if constexpr (C::REG_SOFT > 0) regs_claim<C::REG_SOFT>();
    const int wg = (warp - 4) >> 2;  // key columns [32 wg, 32 wg + 32)
    const int quarter = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint64_t c2 = f2_pack(s.scale_log2, s.scale_log2);
    using T16 = typename std::conditional<C::BF16, __nv_bfloat16, __half>::type;
    // LSE and D of this thread's row of an item (loaded one item ahead)
    auto row_stats = [&](const DqItem& u, float* L, float* dv) {
      *L = -INFINITY;
      *dv = 0.f;
      const int r = u.q0 + quarter * 32 + lane;
      if (u.n_iter > 0 && r < s.Tq) {
        const int64_t idx = static_cast<int64_t>(u.bh) * s.Tq + r;
        *L = lse[idx];
        *dv = dvec[idx];
      }
    };
    // Q in TMEM: this warpgroup writes its share of the item's Q columns for
    // its thread's row (zeros past Tq), then tells the MMA warp. Called once
    // the previous item's last S has completed (the warps waited for it).
    auto load_q_rows = [&](const DqItem& u) {
      if constexpr (C::QTM) {
        if (u.n_iter == 0) return;
        constexpr int COLS = C::DP / 2 / C::NWG;   // 32-bit TMEM columns per warpgroup
        const int r = u.q0 + quarter * 32 + lane;
        const uint4* src = reinterpret_cast<const uint4*>(
            static_cast<const T16*>(q_rows) + (static_cast<int64_t>(u.bh) * s.Tq + (r < s.Tq ? r : 0)) * C::D) +
            wg * (COLS / 4);
#pragma unroll
        for (int c = 0; c < COLS; c += 32) {
          uint32_t w[32];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const uint4 x = r < s.Tq ? __ldg(src + c / 4 + e) : make_uint4(0, 0, 0, 0);
            w[4 * e] = x.x; w[4 * e + 1] = x.y; w[4 * e + 2] = x.z; w[4 * e + 3] = x.w;
          }
          tmem_st32(tmem + lane_base + C::QT_COL + wg * COLS + c, w);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_QFULL));
      }
    };
    DqItem t = dq_item(blockIdx.x, order, s, C::BN);
    float L, dv;
    row_stats(t, &L, &dv);
    load_q_rows(t);
    int gt = 0, ln = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int row = t.q0 + quarter * 32 + lane;
      // -LSE * log2(e) and -D of this row; no visible key (or past Tq): P = 0
      const float nl2 = (L == -INFINITY) ? -INFINITY : -L * kLog2e;
      const uint64_t nl2x2 = f2_pack(nl2, nl2), ndx2 = f2_pack(-dv, -dv);
      for (int it = 0; it < t.n_iter; ++it) {
        const int gi = gt + it;
        const int kb = (t.j_lo + it) * C::BN + wg * C::CW;
        // with Q in TMEM, S alternates between two blocks (and s_full barriers)
        const int sb = C::QTM ? (gi & 1) : 0;
        ok = mbar_wait(bar(C::B_SFULL + sb), (C::QTM ? (gi >> 1) : gi) & 1, tmo, abort_flag, wc.status);
        if (!ok) break;
        tc_fence_after();
        uint32_t sv[32];
        tmem_ld32(tmem + lane_base + C::s_col(gi & 1) + wg * C::CW, sv);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_SFREE));  // the next S may overwrite them
        if (!block_unmasked(s, t.q0, t.q0 + kBM, kb, kb + C::CW)) {
          int lo, hi;
          visible_keys(s, row, kb, &lo, &hi);
#pragma unroll
          for (int q = 0; q < 32; ++q)
            sv[q] = (q >= lo && q < hi) ? sv[q] : __float_as_uint(-INFINITY);
        }
        exp2_scores32(sv, c2, nullptr, false, nl2x2);  // sv now holds P (fp32)
        ok = mbar_wait(bar(C::B_DPFULL + (gi & 1)), (gi >> 1) & 1, tmo, abort_flag, wc.status);
        if (!ok) break;
        tc_fence_after();
        const uint32_t col = C::dp_col(gi & 1) + wg * C::CW;
        uint32_t pv[32];
        tmem_ld32(tmem + lane_base + col, pv);
        tmem_ld_wait();
        uint32_t dsv[16];
#pragma unroll
        for (int q = 0; q < 32; q += 2) {
          // ds = p * (dp - D)
          const uint64_t d =
              fadd2(f2_pack(__uint_as_float(pv[q]), __uint_as_float(pv[q + 1])), ndx2);
          const float2 d2 = f2_unpack(
              fmul2(d, f2_pack(__uint_as_float(sv[q]), __uint_as_float(sv[q + 1]))));
          dsv[q / 2] = pack2_rna<C::BF16>(d2.x, d2.y);
        }
        tmem_st16(tmem + lane_base + col, dsv);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_PFULL + (gi & 1)));
      }
      if (!ok) break;
      // the next item and its row statistics, loaded while this one is stored
      int next = 0;
      const bool more = clc_next(iq, k, lane, &next, tmo, abort_flag, wc.status);
      DqItem tn = t;
      float Ln = -INFINITY, dvn = 0.f;
      if (more) {
        tn = dq_item(next, order, s, C::BN);
        row_stats(tn, &Ln, &dvn);
        // this item's last S has completed (waited for above), so its Q
        // columns are free for the next item's rows
        load_q_rows(tn);
      }
      // ----------------------------------------------------- item epilogue
      // 32-column blocks of the dQ rows dealt round-robin over the warps of
      // this lane quarter; then the accumulator is free for the next item
      const bool have = t.n_iter > 0;
      if (have) {
        ok = mbar_wait(bar(C::B_DONE), ln & 1, tmo, abort_flag, wc.status);
        if (!ok) break;
        tc_fence_after();
      }
      const int row0 = t.q0 + quarter * 32;
      const int rows_valid = min(32, s.Tq - row0);
      T16* dst_blk = reinterpret_cast<T16*>(dq_out) +
                     (static_cast<int64_t>(t.bh) * s.Tq + (rows_valid > 0 ? row0 : 0)) * C::D;
#pragma unroll 1
      for (int task = wg; task < C::D / 32; task += C::NWG)
        store_acc_block<4, C::BF16>(tmem + lane_base + C::DQ_COL + task * 32, have, scale,
                                    dst_blk + task * 32, C::D, rows_valid);
      if (have) {
        tc_fence_before();  // the next item's first dQ follows these reads
        gt += t.n_iter;
        ++ln;
      }
      if (!more) break;
      t = tn;
      L = Ln;
      dv = dvn;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (overlap_prior) grid_wait_prior();
}

}  // namespace fa
