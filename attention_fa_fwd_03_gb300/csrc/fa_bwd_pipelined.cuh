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
// * The score columns are free once the softmax has read them, so S(i+1) is
//   issued then. Per tile the tensor core runs, back to back:
//     dK/dV:  S^T(i+1)  dK,dV += (dS^T, P^T)(i) . (Q, dO)(i)  dP^T(i+1)
//     dQ:     S(j+1)    dQ += dS(j) K(j)                        dP(j+1)
// * The operand the next tile needs first (Q in dK/dV, K in dQ) is
//   prefetched three tiles deep, the other two deep, each slot released by
//   the MMA that last reads it.
// NWG softmax warpgroups split the 128 columns of every tile (128 / NWG each).
//
// TMEM layout of the 16-bit operands: the score columns are handled in chunks
// of 32; chunk m (loaded from dP columns DP_COL + 32m ..) writes its outputs
// back to DP_COL + 32m: P^T to [+0, +16) and dS^T to [+16, +32) in dK/dV, dS
// to [+0, +16) in dQ. So the 16-row K-block kk of the next MMA reads column
// DP_COL + 32 (kk / 2) + 8 (kk % 2).
#pragma once

#include <type_traits>

#include "fa_common.cuh"

namespace fa {

__host__ __device__ constexpr uint32_t chunk_operand_col(uint32_t dp_col, int kk) {
  return dp_col + 32 * (kk >> 1) + 8 * (kk & 1);
}

// Store one 16-column chunk of an fp32 TMEM accumulator row, scaled, as
// 16-bit values (32 bytes of the output row).
template <bool BF16, class T16>
__device__ __forceinline__ void store_acc_chunk16(uint32_t taddr, bool have_data, float mul,
                                                  bool valid, T16* dst) {
  uint32_t v[16];
  if (have_data) {
    tmem_ld16(taddr, v);
    tmem_ld_wait();
  }
  uint32_t w[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float a = have_data ? __uint_as_float(v[2 * k]) * mul : 0.f;
    const float b = have_data ? __uint_as_float(v[2 * k + 1]) * mul : 0.f;
    w[k] = pack2<BF16>(a, b);
  }
  if (valid) {
    uint4* d = reinterpret_cast<uint4*>(dst);
    d[0] = make_uint4(w[0], w[1], w[2], w[3]);
    d[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
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
template <int D_, bool BF16_, int NWG_>
struct DkvCfg {
  static constexpr int D = D_;
  static constexpr bool BF16 = BF16_;
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
  // barriers: kv_full, q_full[QST], q_empty[QST], do_full[DST], do_empty[DST],
  // stats_full[2], stats_empty[2], s_full, s_free, dp_full, p_full, done
  static constexpr int B_KVFULL = 0, B_QFULL = 1, B_QEMPTY = B_QFULL + QST,
                       B_DOFULL = B_QEMPTY + QST, B_DOEMPTY = B_DOFULL + DST,
                       B_STFULL = B_DOEMPTY + DST, B_STEMPTY = B_STFULL + 2,
                       B_SFULL = B_STEMPTY + 2, B_SFREE = B_SFULL + 1, B_DPFULL = B_SFULL + 2,
                       B_PFULL = B_SFULL + 3, B_DONE = B_SFULL + 4, NBAR = B_DONE + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16;  // base must be 1024-aligned (checked)
  static constexpr int THREADS = 128 + 128 * NWG;
  static constexpr int S_COL = 0;     // S^T block, 128 fp32 columns
  static constexpr int DP_COL = 128;  // dP^T block, 128 fp32 columns
  static constexpr int DV_COL = 256;
  static constexpr int DK_COL = 256 + D;
  static constexpr uint32_t pt_col(int kk) { return chunk_operand_col(DP_COL, kk); }
  static constexpr uint32_t dst_col(int kk) { return chunk_operand_col(DP_COL, kk) + 16; }
  static_assert(NWG == 4, "one 32-column chunk per softmax warpgroup");
  static_assert(D <= 128, "dV and dK accumulators share 256 TMEM columns");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

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

  int bg, kvt;  // (b * Hkv + g, block of 128 KV rows)
  decode_tile(blockIdx.x, order, &bg, &kvt);
  const int b = bg / s.Hkv, g = bg % s.Hkv;
  const int reps = s.Hq / s.Hkv;
  const int k0 = kvt * kBM;
  int qf, ql;
  query_range(s, k0, min(s.Tkv, k0 + kBM), &qf, &ql);
  const int i_lo = qf / C::BMQ;
  const int n_qt = max(0, (ql + C::BMQ - 1) / C::BMQ - i_lo);
  const int n_iter = n_qt * reps;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < C::NBAR; ++i) {
      uint32_t cnt = 1;
      if (i == C::B_STFULL || i == C::B_STFULL + 1) cnt = 32;  // the staging warp's lanes
      if (i == C::B_STEMPTY || i == C::B_STEMPTY + 1 || i == C::B_SFREE || i == C::B_PFULL)
        cnt = 4 * C::NWG;  // one arrival per softmax warp
      mbar_init(bar(i), cnt);
    }
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 || warp == 2) {
    // ----------------------------------------------------------- producers
    // warp 0: K, V once, then the Q ring; warp 2: the dO ring. A tile pair
    // takes ~1.4 us to land under full load, so each ring is refilled the
    // moment its own slot frees, independently of the other.
    if (n_iter > 0) {
      // the whole warp runs the loop (a lone active lane whose siblings wait at
      // the final barrier issues far slower); one elected lane issues
      const bool leader = elect_one_sync();
      const bool q_ring = warp == 0;
      if (q_ring) {
        if (leader) tma_prefetch_desc(&map_q);
        if (leader) mbar_arrive_expect_tx(bar(C::B_KVFULL), 2 * C::TILE);
        for (int r = 0; r < C::KREG; ++r) {
          if (leader) tma_load_3d(sbase + C::OFF_K + r * C::REGION, &map_k, bar(C::B_KVFULL), r * 64, k0, bg);
          if (leader) tma_load_3d(sbase + C::OFF_V + r * C::REGION, &map_v, bar(C::B_KVFULL), r * 64, k0, bg);
        }
      } else if (leader) {
        tma_prefetch_desc(&map_do);
      }
      const int nst = q_ring ? C::QST : C::DST;
      const int full = q_ring ? C::B_QFULL : C::B_DOFULL, empty = q_ring ? C::B_QEMPTY : C::B_DOEMPTY;
      const uint32_t ring = sbase + (q_ring ? C::OFF_Q : C::OFF_DO);
      const CUtensorMap* map = q_ring ? &map_q : &map_do;
      for (int it = 0; it < n_iter; ++it) {
        const int zq = b * s.Hq + g * reps + it / n_qt;
        const int i0 = (i_lo + it % n_qt) * C::BMQ;
        const int st = it % nst;
        if (it >= nst)
          mbar_wait_poll(bar(empty + st), ((it / nst) - 1) & 1, tmo, abort_flag, wc.status);
        if (leader) mbar_arrive_expect_tx(bar(full + st), C::TILE);
        for (int r = 0; r < C::KREG; ++r)
          if (leader) tma_load_3d(ring + st * C::TILE + r * C::REGION, map, bar(full + st), r * 64, i0, zq);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer
    if (n_iter > 0) {
      // the whole warp runs the loop (a lone active lane whose siblings wait at
      // the final barrier issues far slower); one elected lane issues
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
      mbar_wait_poll(bar(C::B_KVFULL), 0, tmo, abort_flag, wc.status);
      mbar_wait_poll(bar(C::B_QFULL + 0), 0, tmo, abort_flag, wc.status);
      tc_fence_after();
      if (leader) issue_score(sbase + C::OFF_K, sbase + C::OFF_Q, C::S_COL);
      if (leader) mma_commit(bar(C::B_SFULL));
      mbar_wait_poll(bar(C::B_DOFULL + 0), 0, tmo, abort_flag, wc.status);
      tc_fence_after();
      if (leader) issue_score(sbase + C::OFF_V, sbase + C::OFF_DO, C::DP_COL);
      if (leader) mma_commit(bar(C::B_DPFULL));
      for (int it = 0; it < n_iter; ++it) {
        const int qs = it % C::QST, ds = it % C::DST;
        const bool more = it + 1 < n_iter;
        if (more) {
          // next S^T as soon as the softmax has read this tile's S^T
          const int nq = (it + 1) % C::QST;
          mbar_wait_poll(bar(C::B_QFULL + nq), ((it + 1) / C::QST) & 1, tmo, abort_flag, wc.status);
          mbar_wait_poll(bar(C::B_SFREE), it & 1, tmo, abort_flag, wc.status);
          tc_fence_after();
          if (leader) issue_score(sbase + C::OFF_K, sbase + C::OFF_Q + nq * C::TILE, C::S_COL);
          if (leader) mma_commit(bar(C::B_SFULL));
        }
        mbar_wait_poll(bar(C::B_PFULL), it & 1, tmo, abort_flag, wc.status);
        tc_fence_after();
        // dK += dS^T Q, then dV += P^T dO  (A from TMEM, B MN-major, K = query rows);
        // each ring slot is released by the last MMA that reads it
        const uint64_t qdesc = make_sdesc(sbase + C::OFF_Q + qs * C::TILE, C::REGION, 1024, 2);
        const uint64_t ddesc = make_sdesc(sbase + C::OFF_DO + ds * C::TILE, C::REGION, 1024, 2);
#pragma unroll
        for (int kk = 0; kk < C::BMQ / 16; ++kk)
          if (leader) mma_ts(tmem + C::DK_COL, tmem + C::dst_col(kk), qdesc + ((kk * 16 * 128) >> 4),
                 idesc_acc, (it > 0 || kk > 0) ? 1u : 0u);
        if (leader) mma_commit(bar(C::B_QEMPTY + qs));
#pragma unroll
        for (int kk = 0; kk < C::BMQ / 16; ++kk)
          if (leader) mma_ts(tmem + C::DV_COL, tmem + C::pt_col(kk), ddesc + ((kk * 16 * 128) >> 4),
                 idesc_acc, (it > 0 || kk > 0) ? 1u : 0u);
        if (leader) mma_commit(bar(C::B_DOEMPTY + ds));
        if (more) {
          // dP^T(it+1) overwrites the P^T / dS^T columns the MMAs above read
          // (tcgen05 MMAs of one thread execute in order)
          const int nd = (it + 1) % C::DST;
          mbar_wait_poll(bar(C::B_DOFULL + nd), ((it + 1) / C::DST) & 1, tmo, abort_flag, wc.status);
          tc_fence_after();
          if (leader) issue_score(sbase + C::OFF_V, sbase + C::OFF_DO + nd * C::TILE, C::DP_COL);
          if (leader) mma_commit(bar(C::B_DPFULL));
        }
      }
      if (leader) mma_commit(bar(C::B_DONE));
      mbar_wait_poll(bar(C::B_DONE), 0, tmo, nullptr, wc.status);
    }
  } else if (warp == 3) {
    // ------------------------------------------- LSE / D-vector staging
    for (int it = 0; it < n_iter; ++it) {
      const int slot = it & 1;
      const int h = g * reps + it / n_qt;
      const int i0 = (i_lo + it % n_qt) * C::BMQ;
      if (it >= 2)
        mbar_wait(bar(C::B_STEMPTY + slot), ((it >> 1) - 1) & 1, tmo, abort_flag, wc.status);
      float* dst = stats + slot * 2 * C::BMQ;
      const int64_t base = static_cast<int64_t>(b * s.Hq + h) * s.Tq;
      for (int t = lane; t < C::BMQ; t += 32) {
        const int i = i0 + t;
        float nl2 = -INFINITY, nd = 0.f;  // rows past Tq: P = 0
        if (i < s.Tq) {
          const float L = lse[base + i];
          nl2 = (L == -INFINITY) ? -INFINITY : -L * kLog2e;  // row with no visible key: P = 0
          nd = -dvec[base + i];
        }
        dst[t] = nl2;
        dst[C::BMQ + t] = nd;
      }
      mbar_arrive(bar(C::B_STFULL + slot));
    }
  } else if (warp >= 4) {
    // ------------------------------------------- softmax: P^T and dS^T
    const int wg = (warp - 4) >> 2;             // query columns [32 wg, 32 wg + 32)
    const int quarter = warp & 3;
    const int krow = k0 + quarter * 32 + lane;  // KV row of this thread (TMEM lane)
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint64_t c2 = f2_pack(s.scale_log2, s.scale_log2);
    const uint32_t col = C::DP_COL + wg * C::CW;  // this warpgroup's dP^T chunk
    for (int it = 0; it < n_iter; ++it) {
      const int slot = it & 1;
      const int i0 = (i_lo + it % n_qt) * C::BMQ;
      mbar_wait(bar(C::B_STFULL + slot), (it >> 1) & 1, tmo, abort_flag, wc.status);
      mbar_wait(bar(C::B_SFULL), it & 1, tmo, abort_flag, wc.status);
      tc_fence_after();
      uint32_t sv[32];
      tmem_ld32(tmem + lane_base + C::S_COL + wg * C::CW, sv);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::B_SFREE));  // the next S^T may overwrite them
      const float* nl_s = stats + slot * 2 * C::BMQ + wg * C::CW;  // -LSE * log2(e)
      const float* nd_s = nl_s + C::BMQ;                           // -D
      if (!block_unmasked(s, i0, i0 + C::BMQ, k0, k0 + kBM)) {
#pragma unroll
        for (int q = 0; q < 32; ++q)
          if (!key_visible(i0 + wg * C::CW + q, krow, s.causal, s.window))
            sv[q] = __float_as_uint(-INFINITY);
      }
      exp2_scores32(sv, c2, nl_s, true, 0);  // sv now holds P (fp32)
      // dS^T = P^T o (dP^T - D) once dP^T(it) is in TMEM
      mbar_wait(bar(C::B_DPFULL), it & 1, tmo, abort_flag, wc.status);
      tc_fence_after();
      uint32_t pv[32];
      tmem_ld32(tmem + lane_base + col, pv);
      tmem_ld_wait();
      uint32_t pp[16], dsv[16];
#pragma unroll
      for (int k = 0; k < 32; k += 4) {
        const ulonglong2 nd = *reinterpret_cast<const ulonglong2*>(nd_s + k);
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
          const uint64_t p2 = f2_pack(__uint_as_float(sv[k + e]), __uint_as_float(sv[k + e + 1]));
          const uint64_t t = fadd2(
              f2_pack(__uint_as_float(pv[k + e]), __uint_as_float(pv[k + e + 1])),
              e == 0 ? nd.x : nd.y);
          const float2 d2 = f2_unpack(fmul2(t, p2));
          pp[(k + e) / 2] = pack2<C::BF16>(__uint_as_float(sv[k + e]), __uint_as_float(sv[k + e + 1]));
          dsv[(k + e) / 2] = pack2<C::BF16>(d2.x, d2.y);
        }
      }
      tmem_st16(tmem + lane_base + col, pp);
      tmem_st16(tmem + lane_base + col + 16, dsv);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(C::B_PFULL));
        mbar_arrive(bar(C::B_STEMPTY + slot));
      }
    }
    // ------------------------------------------------------- epilogue
    // 16-column chunks of the dV then dK row (dK scaled), dealt round-robin
    // over the softmax warpgroups; one row per thread
    if (n_iter > 0) {
      mbar_wait(bar(C::B_DONE), 0, tmo, abort_flag, wc.status);
      tc_fence_after();
    }
    using T16 = typename std::conditional<C::BF16, __nv_bfloat16, __half>::type;
    const bool valid = krow < s.Tkv;
    const int64_t orow = (static_cast<int64_t>(bg) * s.Tkv + (valid ? krow : 0)) * C::D;
#pragma unroll 1
    for (int chunk = wg; chunk < 2 * C::D / 16; chunk += C::NWG) {
      const bool is_dk = chunk >= C::D / 16;
      const int cc = (is_dk ? chunk - C::D / 16 : chunk) * 16;
      T16* dst = reinterpret_cast<T16*>(is_dk ? dk_out : dv_out) + orow + cc;
      store_acc_chunk16<C::BF16>(tmem + lane_base + (is_dk ? C::DK_COL : C::DV_COL) + cc,
                                 n_iter > 0, is_dk ? scale : 1.f, valid, dst);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// --------------------------------------------------------------------- dQ
template <int D_, bool BF16_, int NWG_>
struct DqCfg {
  static constexpr int D = D_;
  static constexpr bool BF16 = BF16_;
  static constexpr int NWG = NWG_;
  static constexpr int CW = 128 / NWG;  // key columns per softmax warpgroup
  static constexpr int KST = 3;         // K ring: needed first by the next tile
  static constexpr int VST = 2;         // V ring
  static constexpr int BN = 128;        // key rows per tile (N of S, dP)
  static constexpr int DP = (D + 63) / 64 * 64;
  static constexpr int KREG = DP / 64;
  static constexpr int REGION = 128 * 128;
  static constexpr int TILE = KREG * REGION;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = OFF_Q + TILE;
  static constexpr int OFF_K = OFF_DO + TILE;
  static constexpr int OFF_V = OFF_K + KST * TILE;
  static constexpr int OFF_BAR = OFF_V + VST * TILE;
  // barriers: q_full, k_full[KST], k_empty[KST], v_full[VST], v_empty[VST],
  // s_full, s_free, dp_full, p_full, done
  static constexpr int B_QFULL = 0, B_KFULL = 1, B_KEMPTY = B_KFULL + KST,
                       B_VFULL = B_KEMPTY + KST, B_VEMPTY = B_VFULL + VST,
                       B_SFULL = B_VEMPTY + VST, B_SFREE = B_SFULL + 1, B_DPFULL = B_SFULL + 2,
                       B_PFULL = B_SFULL + 3, B_DONE = B_SFULL + 4, NBAR = B_DONE + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16;  // base must be 1024-aligned (checked)
  static constexpr int THREADS = 128 + 128 * NWG;
  static constexpr int S_COL = 0;
  static constexpr int DP_COL = 128;
  static constexpr int DQ_COL = 256;
  static constexpr uint32_t ds_col(int kk) { return chunk_operand_col(DP_COL, kk); }
  static_assert(NWG == 4, "one 32-column chunk per softmax warpgroup");
  static_assert(D <= 128, "dQ accumulator in TMEM columns 256-383");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                 const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                 const float* __restrict__ lse, const float* __restrict__ dvec,
                 void* __restrict__ dq_out, float scale, AttnShape s, TileOrder order,
                 WaitCfg wc) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {  // the 128-byte swizzle needs 1024-byte aligned tiles
    if (threadIdx.x == 0) atomicOr(wc.status, kStatusSmemMisaligned);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  auto bar = [&](int i) { return smem_u32(bars + i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const uint64_t tmo = wc.timeout_cycles;

  int bh, qt;  // (b * Hq + h, block of 128 query rows)
  decode_tile(blockIdx.x, order, &bh, &qt);
  const int b = bh / s.Hq, h = bh % s.Hq;
  const int g = h / (s.Hq / s.Hkv);
  const int q0 = qt * kBM;
  int kf, kl;
  key_range(s, q0, min(s.Tq, q0 + kBM), &kf, &kl);
  const int j_lo = kf / C::BN;
  const int n_iter = max(0, (kl + C::BN - 1) / C::BN - j_lo);

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < C::NBAR; ++i)  // one arrival per softmax warp on p_full / s_free
      mbar_init(bar(i), (i == C::B_PFULL || i == C::B_SFREE) ? 4u * C::NWG : 1u);
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 || warp == 2) {
    // producers: warp 0 loads Q, dO once, then the K ring; warp 2 the V ring,
    // each refilled the moment its own slot frees
    if (n_iter > 0) {
      // the whole warp runs the loop (a lone active lane whose siblings wait at
      // the final barrier issues far slower); one elected lane issues
      const bool leader = elect_one_sync();
      const bool k_ring = warp == 0;
      if (k_ring) {
        if (leader) tma_prefetch_desc(&map_k);
        if (leader) mbar_arrive_expect_tx(bar(C::B_QFULL), 2 * C::TILE);
        for (int r = 0; r < C::KREG; ++r) {
          if (leader) tma_load_3d(sbase + C::OFF_Q + r * C::REGION, &map_q, bar(C::B_QFULL), r * 64, q0, bh);
          if (leader) tma_load_3d(sbase + C::OFF_DO + r * C::REGION, &map_do, bar(C::B_QFULL), r * 64, q0, bh);
        }
      } else if (leader) {
        tma_prefetch_desc(&map_v);
      }
      const int zkv = b * s.Hkv + g;
      const int nst = k_ring ? C::KST : C::VST;
      const int full = k_ring ? C::B_KFULL : C::B_VFULL, empty = k_ring ? C::B_KEMPTY : C::B_VEMPTY;
      const uint32_t ring = sbase + (k_ring ? C::OFF_K : C::OFF_V);
      const CUtensorMap* map = k_ring ? &map_k : &map_v;
      for (int it = 0; it < n_iter; ++it) {
        const int kr = (j_lo + it) * C::BN;
        const int st = it % nst;
        if (it >= nst)
          mbar_wait_poll(bar(empty + st), ((it / nst) - 1) & 1, tmo, abort_flag, wc.status);
        if (leader) mbar_arrive_expect_tx(bar(full + st), C::TILE);
        for (int r = 0; r < C::KREG; ++r)
          if (leader) tma_load_3d(ring + st * C::TILE + r * C::REGION, map, bar(full + st), r * 64, kr, zkv);
      }
    }
  } else if (warp == 1) {
    if (n_iter > 0) {
      // the whole warp runs the loop (a lone active lane whose siblings wait at
      // the final barrier issues far slower); one elected lane issues
      const bool leader = elect_one_sync();
      constexpr uint32_t ab = C::BF16 ? 1 : 0;
      constexpr uint32_t idesc_s = make_idesc_f16(kBM, C::BN, ab, 0, 0);
      constexpr uint32_t idesc_q = make_idesc_f16(kBM, C::D, ab, 0, 1);
      auto issue_score = [&](uint32_t a_base, uint32_t b_base, uint32_t col) {
        const uint64_t ad = make_sdesc(a_base, 16, 1024, 2), bd = make_sdesc(b_base, 16, 1024, 2);
#pragma unroll
        for (int kk = 0; kk < C::D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::REGION + (kk & 3) * 32;
          if (leader) mma_ss(tmem + col, ad + (off >> 4), bd + (off >> 4), idesc_s, kk > 0);
        }
      };
      mbar_wait_poll(bar(C::B_QFULL), 0, tmo, abort_flag, wc.status);
      mbar_wait_poll(bar(C::B_KFULL + 0), 0, tmo, abort_flag, wc.status);
      tc_fence_after();
      if (leader) issue_score(sbase + C::OFF_Q, sbase + C::OFF_K, C::S_COL);
      if (leader) mma_commit(bar(C::B_SFULL));
      mbar_wait_poll(bar(C::B_VFULL + 0), 0, tmo, abort_flag, wc.status);
      tc_fence_after();
      if (leader) issue_score(sbase + C::OFF_DO, sbase + C::OFF_V, C::DP_COL);
      if (leader) mma_commit(bar(C::B_DPFULL));
      if (leader) mma_commit(bar(C::B_VEMPTY + 0));
      for (int it = 0; it < n_iter; ++it) {
        const int ks = it % C::KST;
        const bool more = it + 1 < n_iter;
        if (more) {
          const int nk = (it + 1) % C::KST;
          mbar_wait_poll(bar(C::B_KFULL + nk), ((it + 1) / C::KST) & 1, tmo, abort_flag, wc.status);
          mbar_wait_poll(bar(C::B_SFREE), it & 1, tmo, abort_flag, wc.status);
          tc_fence_after();
          if (leader) issue_score(sbase + C::OFF_Q, sbase + C::OFF_K + nk * C::TILE, C::S_COL);
          if (leader) mma_commit(bar(C::B_SFULL));
        }
        mbar_wait_poll(bar(C::B_PFULL), it & 1, tmo, abort_flag, wc.status);
        tc_fence_after();
        // dQ += dS K   (dS from TMEM, K as MN-major B, K = key rows)
        const uint64_t kdesc = make_sdesc(sbase + C::OFF_K + ks * C::TILE, C::REGION, 1024, 2);
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk)
          if (leader) mma_ts(tmem + C::DQ_COL, tmem + C::ds_col(kk), kdesc + ((kk * 16 * 128) >> 4), idesc_q,
                 (it > 0 || kk > 0) ? 1u : 0u);
        if (leader) mma_commit(bar(C::B_KEMPTY + ks));
        if (more) {
          // dP(it+1) overwrites the dS columns the MMAs above read (in order)
          const int nv = (it + 1) % C::VST;
          mbar_wait_poll(bar(C::B_VFULL + nv), ((it + 1) / C::VST) & 1, tmo, abort_flag, wc.status);
          tc_fence_after();
          if (leader) issue_score(sbase + C::OFF_DO, sbase + C::OFF_V + nv * C::TILE, C::DP_COL);
          if (leader) mma_commit(bar(C::B_DPFULL));
          if (leader) mma_commit(bar(C::B_VEMPTY + nv));  // V is read by dP only
        }
      }
      if (leader) mma_commit(bar(C::B_DONE));
      mbar_wait_poll(bar(C::B_DONE), 0, tmo, nullptr, wc.status);
    }
  } else if (warp >= 4) {
    const int wg = (warp - 4) >> 2;  // key columns [32 wg, 32 wg + 32)
    const int quarter = warp & 3;
    const int row = q0 + quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    float nl2 = -INFINITY, nd = 0.f;  // -LSE * log2(e) and -D of this row
    if (row < s.Tq) {
      const int64_t idx = static_cast<int64_t>(bh) * s.Tq + row;
      const float L = lse[idx];
      nl2 = (L == -INFINITY) ? -INFINITY : -L * kLog2e;  // no visible key: P = 0
      nd = -dvec[idx];
    }
    const uint64_t c2 = f2_pack(s.scale_log2, s.scale_log2), nl2x2 = f2_pack(nl2, nl2),
                   ndx2 = f2_pack(nd, nd);
    const uint32_t col = C::DP_COL + wg * C::CW;
    for (int it = 0; it < n_iter; ++it) {
      const int kb = (j_lo + it) * C::BN + wg * C::CW;
      mbar_wait(bar(C::B_SFULL), it & 1, tmo, abort_flag, wc.status);
      tc_fence_after();
      uint32_t sv[32];
      tmem_ld32(tmem + lane_base + C::S_COL + wg * C::CW, sv);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::B_SFREE));  // the next S may overwrite them
      if (!block_unmasked(s, q0, q0 + kBM, kb, kb + C::CW)) {
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const int j = kb + k;
          if (j >= s.Tkv || !key_visible(row, j, s.causal, s.window))
            sv[k] = __float_as_uint(-INFINITY);
        }
      }
      exp2_scores32(sv, c2, nullptr, false, nl2x2);  // sv now holds P (fp32)
      mbar_wait(bar(C::B_DPFULL), it & 1, tmo, abort_flag, wc.status);
      tc_fence_after();
      uint32_t pv[32];
      tmem_ld32(tmem + lane_base + col, pv);
      tmem_ld_wait();
      uint32_t dsv[16];
#pragma unroll
      for (int k = 0; k < 32; k += 2) {
        // ds = p * (dp - D)
        const uint64_t t =
            fadd2(f2_pack(__uint_as_float(pv[k]), __uint_as_float(pv[k + 1])), ndx2);
        const float2 d2 = f2_unpack(
            fmul2(t, f2_pack(__uint_as_float(sv[k]), __uint_as_float(sv[k + 1]))));
        dsv[k / 2] = pack2<C::BF16>(d2.x, d2.y);
      }
      tmem_st16(tmem + lane_base + col, dsv);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::B_PFULL));
    }
    // epilogue: 16-column chunks of the dQ row dealt round-robin over the
    // softmax warpgroups
    if (n_iter > 0) {
      mbar_wait(bar(C::B_DONE), 0, tmo, abort_flag, wc.status);
      tc_fence_after();
    }
    using T16 = typename std::conditional<C::BF16, __nv_bfloat16, __half>::type;
    const bool valid = row < s.Tq;
    T16* dst_row = reinterpret_cast<T16*>(dq_out) +
                   (static_cast<int64_t>(bh) * s.Tq + (valid ? row : 0)) * C::D;
#pragma unroll 1
    for (int chunk = wg; chunk < C::D / 16; chunk += C::NWG)
      store_acc_chunk16<C::BF16>(tmem + lane_base + C::DQ_COL + chunk * 16, n_iter > 0, scale,
                                 valid, dst_row + chunk * 16);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace fa
