// Pipelined dK/dV and dQ kernels for head dims up to 128 (128 x 128 tiles).
//
// Same computation as the kernels in fa_bwd.cuh (page "mlx-bun 0.0.4:
// package/src/model/flash-attention.ts", backward passes 2 and 3; page
// "[Metal] Add Flash Attention VJP for training", Implementation Notes: KV-row
// ownership, log2 domain), scheduled so that the tensor core keeps working
// while the softmax warps turn scores into P and dS:
//
// An M=128 tcgen05.mma costs at least ~44 cycles however narrow N is, so both
// score blocks stay 128 x 128 (N = 128 runs at the full rate). TMEM (512
// columns) then holds exactly one score block, one dP block and the fp32
// accumulators; there is no room for a second score buffer. Instead, the
// softmax warps load the score and dP blocks into registers, and write the
// 16-bit operands they produce (P and dS, 64 packed columns each) into the dP
// block's columns. The score columns are free as soon as the loads are done,
// so the next tile's score MMA runs while the softmax is still computing:
//   dK/dV:  S^T(i+1) || softmax(i)  ->  dV += P^T dO, dK += dS^T Q  ->  dP^T(i+1)
//   dQ:     S(j+1)   || softmax(j)  ->  dQ += dS K                  ->  dP(j+1)
// Two softmax warpgroups split the 128 columns of every tile.
#pragma once

#include <type_traits>

#include "fa_common.cuh"

namespace fa {

// ---------------------------------------------------------------- dK / dV
template <int D_, int STAGES_, bool BF16_>
struct DkvCfg {
  static constexpr int D = D_;
  static constexpr int STAGES = STAGES_;
  static constexpr bool BF16 = BF16_;
  static constexpr int BMQ = 128;  // query rows per inner tile (N of S^T, dP^T)
  static constexpr int DP = (D + 63) / 64 * 64;
  static constexpr int KREG = DP / 64;
  static constexpr int REGION = 128 * 128;  // one 64-column block of a 128-row tile
  static constexpr int TILE = KREG * REGION;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + TILE;
  static constexpr int OFF_Q = OFF_V + TILE;
  static constexpr int OFF_DO = OFF_Q + STAGES * TILE;
  static constexpr int OFF_STATS = OFF_DO + STAGES * TILE;  // [STAGES][lse2 | dvec][128] fp32
  static constexpr int OFF_BAR = OFF_STATS + STAGES * 2 * BMQ * 4;
  // barriers: kv_full, q_full[S], q_empty[S], stats_full[S], s_full, s_free, p_full, done
  static constexpr int NBAR = 1 + 3 * STAGES + 4;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int THREADS = 384;
  static constexpr int S_COL = 0;     // S^T block, 128 fp32 columns
  static constexpr int DP_COL = 128;  // dP^T block, 128 fp32 columns
  static constexpr int DV_COL = 256;
  static constexpr int DK_COL = 256 + D;
  // P^T and dS^T (16-bit, two per column) are written over the dP^T columns
  // by the warpgroup that loaded them: query rows 32c..32c+31 of warpgroup w
  // (its chunk c) land in dP^T columns 64w + 32c + [0, 16) (P^T) and
  // 64w + 32c + [16, 32) (dS^T). Query block kk (16 rows) of the tile:
  static constexpr uint32_t pt_col(int kk) {
    return DP_COL + 64 * (kk >> 2) + 32 * ((kk >> 1) & 1) + 8 * (kk & 1);
  }
  static constexpr uint32_t dst_col(int kk) { return pt_col(kk) + 16; }
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
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  auto bar = [&](int i) { return smem_u32(bars + i); };
  const int B_KVFULL = 0, B_QFULL = 1, B_QEMPTY = 1 + C::STAGES, B_STATS = 1 + 2 * C::STAGES,
            B_SFULL = 1 + 3 * C::STAGES, B_SFREE = B_SFULL + 1, B_PFULL = B_SFULL + 2,
            B_DONE = B_SFULL + 3;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  float* stats = reinterpret_cast<float*>(smem + C::OFF_STATS);

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
      if (i >= B_STATS && i < B_STATS + C::STAGES) cnt = 32;
      if (i == B_PFULL || i == B_SFREE) cnt = 8;  // one arrival per softmax warp
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_iter > 0) {
      tma_prefetch_desc(&map_q);
      tma_prefetch_desc(&map_do);
      mbar_arrive_expect_tx(bar(B_KVFULL), 2 * C::TILE);
      for (int r = 0; r < C::KREG; ++r) {
        tma_load_3d(sbase + C::OFF_K + r * C::REGION, &map_k, bar(B_KVFULL), r * 64, k0, bg);
        tma_load_3d(sbase + C::OFF_V + r * C::REGION, &map_v, bar(B_KVFULL), r * 64, k0, bg);
      }
      for (int it = 0; it < n_iter; ++it) {
        const int st = it % C::STAGES;
        const int h = g * reps + it / n_qt;
        const int i0 = (i_lo + it % n_qt) * C::BMQ;
        if (it >= C::STAGES)
          mbar_wait(bar(B_QEMPTY + st), ((it / C::STAGES) - 1) & 1, wc.timeout_ns, abort_flag,
                    wc.status);
        mbar_arrive_expect_tx(bar(B_QFULL + st), 2 * C::TILE);
        const int zq = b * s.Hq + h;
        for (int r = 0; r < C::KREG; ++r) {
          tma_load_3d(sbase + C::OFF_Q + st * C::TILE + r * C::REGION, &map_q, bar(B_QFULL + st),
                      r * 64, i0, zq);
          tma_load_3d(sbase + C::OFF_DO + st * C::TILE + r * C::REGION, &map_do,
                      bar(B_QFULL + st), r * 64, i0, zq);
        }
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0 && n_iter > 0) {
      constexpr uint32_t ab = C::BF16 ? 1 : 0;
      constexpr uint32_t idesc_st = make_idesc_f16(kBM, C::BMQ, ab, 0, 0);  // S^T, dP^T
      constexpr uint32_t idesc_acc = make_idesc_f16(kBM, C::D, ab, 0, 1);   // dV, dK
      // S^T = K Q^T (into S_COL) or dP^T = V dO^T (into DP_COL): K-major, K = head dim
      // descriptors are built once per operand base; the k-step offsets are
      // added to the start-address field (shared addresses < 256 KB never carry)
      auto issue_score = [&](uint32_t a_base, uint32_t b_base, uint32_t col) {
        const uint64_t ad = make_sdesc(a_base, 16, 1024, 2), bd = make_sdesc(b_base, 16, 1024, 2);
#pragma unroll
        for (int kk = 0; kk < C::D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::REGION + (kk & 3) * 32;
          mma_ss(tmem + col, ad + (off >> 4), bd + (off >> 4), idesc_st, kk > 0);
        }
      };
      mbar_wait(bar(B_KVFULL), 0, wc.timeout_ns, abort_flag, wc.status);
      mbar_wait(bar(B_QFULL + 0), 0, wc.timeout_ns, abort_flag, wc.status);
      tc_fence_after();
      issue_score(sbase + C::OFF_K, sbase + C::OFF_Q, C::S_COL);
      issue_score(sbase + C::OFF_V, sbase + C::OFF_DO, C::DP_COL);
      mma_commit(bar(B_SFULL));
      for (int it = 0; it < n_iter; ++it) {
        const int st = it % C::STAGES;
        const int nst = (it + 1) % C::STAGES;
        const bool more = it + 1 < n_iter;
        if (more) {
          // next S^T as soon as the softmax has read this tile's S^T and dP^T
          mbar_wait(bar(B_QFULL + nst), ((it + 1) / C::STAGES) & 1, wc.timeout_ns, abort_flag,
                    wc.status);
          mbar_wait(bar(B_SFREE), it & 1, wc.timeout_ns, abort_flag, wc.status);
          tc_fence_after();
          issue_score(sbase + C::OFF_K, sbase + C::OFF_Q + nst * C::TILE, C::S_COL);
        }
        mbar_wait(bar(B_PFULL), it & 1, wc.timeout_ns, abort_flag, wc.status);
        tc_fence_after();
        // dV += P^T dO,  dK += dS^T Q   (A from TMEM, B MN-major, K = query rows)
        const uint64_t qdesc = make_sdesc(sbase + C::OFF_Q + st * C::TILE, C::REGION, 1024, 2);
        const uint64_t ddesc = make_sdesc(sbase + C::OFF_DO + st * C::TILE, C::REGION, 1024, 2);
#pragma unroll
        for (int kk = 0; kk < C::BMQ / 16; ++kk) {
          const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
          mma_ts(tmem + C::DV_COL, tmem + C::pt_col(kk),
                 ddesc + ((kk * 16 * 128) >> 4), idesc_acc, acc);
          mma_ts(tmem + C::DK_COL, tmem + C::dst_col(kk),
                 qdesc + ((kk * 16 * 128) >> 4), idesc_acc, acc);
        }
        mma_commit(bar(B_QEMPTY + st));
        if (more) {
          // dP^T(it+1) overwrites the P^T / dS^T columns the MMAs above read
          // (tcgen05 MMAs of one thread execute in order)
          issue_score(sbase + C::OFF_V, sbase + C::OFF_DO + nst * C::TILE, C::DP_COL);
          mma_commit(bar(B_SFULL));
        }
      }
      mma_commit(bar(B_DONE));
      mbar_wait(bar(B_DONE), 0, wc.timeout_ns, nullptr, wc.status);
    }
  } else if (warp == 3) {
    // ------------------------------------------- LSE / D-vector staging
    for (int it = 0; it < n_iter; ++it) {
      const int st = it % C::STAGES;
      const int h = g * reps + it / n_qt;
      const int i0 = (i_lo + it % n_qt) * C::BMQ;
      if (it >= C::STAGES)
        mbar_wait(bar(B_QEMPTY + st), ((it / C::STAGES) - 1) & 1, wc.timeout_ns, abort_flag,
                  wc.status);
      float* dst = stats + st * 2 * C::BMQ;
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
      mbar_arrive(bar(B_STATS + st));
    }
  } else if (warp >= 4) {
    // ------------------------------------------- softmax: P^T and dS^T
    const int wg = (warp - 4) >> 2;             // 0: query columns 0-63, 1: 64-127
    const int quarter = warp & 3;
    const int krow = k0 + quarter * 32 + lane;  // KV row of this thread (TMEM lane)
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const float c = s.scale_log2;
    for (int it = 0; it < n_iter; ++it) {
      const int st = it % C::STAGES;
      const int i0 = (i_lo + it % n_qt) * C::BMQ;
      mbar_wait(bar(B_STATS + st), (it / C::STAGES) & 1, wc.timeout_ns, abort_flag, wc.status);
      mbar_wait(bar(B_SFULL), it & 1, wc.timeout_ns, abort_flag, wc.status);
      tc_fence_after();
      // this warpgroup's 64 S^T columns; once every softmax thread holds its
      // share, the next S^T may overwrite them
      uint32_t sv[64];
      tmem_ld32(tmem + lane_base + C::S_COL + wg * 64, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
      tmem_ld32(tmem + lane_base + C::S_COL + wg * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_SFREE));
      // staged per query row: -LSE * log2(e) and -D
      const float* nl_s = stats + st * 2 * C::BMQ + wg * 64;
      const float* nd_s = nl_s + C::BMQ;
      const bool need_mask = !block_unmasked(s, i0, i0 + C::BMQ, k0, k0 + kBM);
      if (need_mask) {
#pragma unroll
        for (int q = 0; q < 64; ++q)
          if (!key_visible(i0 + wg * 64 + q, krow, s.causal, s.window))
            sv[q] = __float_as_uint(-INFINITY);
      }
      const uint64_t c2 = f2_pack(c, c);
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        // dP^T chunk (32 columns); its P^T / dS^T go back over the same columns
        const uint32_t col = C::DP_COL + wg * 64 + ch * 32;
        uint32_t pv[32];
        tmem_ld32(tmem + lane_base + col, pv);
        tmem_ld_wait();
        uint32_t pp[16], ds[16];
#pragma unroll
        for (int k = 0; k < 32; k += 4) {
          const int q = ch * 32 + k;  // column within this warpgroup's 64
          const ulonglong2 nl = *reinterpret_cast<const ulonglong2*>(nl_s + q);
          const ulonglong2 nd = *reinterpret_cast<const ulonglong2*>(nd_s + q);
#pragma unroll
          for (int e = 0; e < 4; e += 2) {
            // x = s * scale * log2(e) - LSE2;  p = 2^x;  ds = p * (dp - D)
            const uint64_t x = ffma2(f2_pack(__uint_as_float(sv[q + e]), __uint_as_float(sv[q + e + 1])),
                                     c2, e == 0 ? nl.x : nl.y);
            const float2 xf = f2_unpack(x);
            const float p0 = ex2(xf.x), p1 = ex2(xf.y);
            const uint64_t t = fadd2(f2_pack(__uint_as_float(pv[k + e]), __uint_as_float(pv[k + e + 1])),
                                     e == 0 ? nd.x : nd.y);
            const float2 d2 = f2_unpack(fmul2(t, f2_pack(p0, p1)));
            pp[(k + e) / 2] = pack2<C::BF16>(p0, p1);
            ds[(k + e) / 2] = pack2<C::BF16>(d2.x, d2.y);
          }
        }
        tmem_st16(tmem + lane_base + col, pp);
        tmem_st16(tmem + lane_base + col + 16, ds);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_PFULL));
    }
    // ------------------------------------------------------- epilogue
    // warpgroup 0 writes dV, warpgroup 1 writes dK (scaled), one row per thread
    if (n_iter > 0) {
      mbar_wait(bar(B_DONE), 0, wc.timeout_ns, abort_flag, wc.status);
      tc_fence_after();
    }
    using T16 = typename std::conditional<C::BF16, __nv_bfloat16, __half>::type;
    const bool valid = krow < s.Tkv;
    const uint32_t col = wg == 0 ? C::DV_COL : C::DK_COL;
    const float mul = wg == 0 ? 1.f : scale;
    T16* dst_row = reinterpret_cast<T16*>(wg == 0 ? dv_out : dk_out) +
                   (static_cast<int64_t>(bg) * s.Tkv + (valid ? krow : 0)) * C::D;
#pragma unroll 1
    for (int cc = 0; cc < C::D; cc += 32) {
      uint32_t v[32];
      if (n_iter > 0) {
        tmem_ld32(tmem + lane_base + col + cc, v);
        tmem_ld_wait();
      }
      uint32_t w[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float a = n_iter > 0 ? __uint_as_float(v[2 * k]) * mul : 0.f;
        const float bb = n_iter > 0 ? __uint_as_float(v[2 * k + 1]) * mul : 0.f;
        w[k] = pack2<C::BF16>(a, bb);
      }
      if (valid) {
        uint4* dst = reinterpret_cast<uint4*>(dst_row + cc);
#pragma unroll
        for (int k = 0; k < 4; ++k) dst[k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
      }
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
template <int D_, int STAGES_, bool BF16_>
struct DqCfg {
  static constexpr int D = D_;
  static constexpr int STAGES = STAGES_;
  static constexpr bool BF16 = BF16_;
  static constexpr int BN = 128;  // key rows per tile (N of S, dP)
  static constexpr int DP = (D + 63) / 64 * 64;
  static constexpr int KREG = DP / 64;
  static constexpr int REGION = 128 * 128;
  static constexpr int TILE = KREG * REGION;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = OFF_Q + TILE;
  static constexpr int OFF_K = OFF_DO + TILE;
  static constexpr int OFF_V = OFF_K + STAGES * TILE;
  static constexpr int OFF_BAR = OFF_V + STAGES * TILE;
  // barriers: q_full, kv_full[S], kv_empty[S], s_full, s_free, p_full, done
  static constexpr int NBAR = 1 + 2 * STAGES + 4;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int THREADS = 384;
  static constexpr int S_COL = 0;
  static constexpr int DP_COL = 128;
  static constexpr int DQ_COL = 256;
  // dS (16-bit, two per column) goes over the dP columns of the warpgroup that
  // loaded them: key rows 64w..64w+63 land in dP columns 64w + [0, 32).
  // Key block kk (16 rows) of the tile:
  static constexpr uint32_t ds_col(int kk) { return DP_COL + 64 * (kk >> 2) + 8 * (kk & 3); }
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
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  auto bar = [&](int i) { return smem_u32(bars + i); };
  const int B_QFULL = 0, B_KVFULL = 1, B_KVEMPTY = 1 + C::STAGES, B_SFULL = 1 + 2 * C::STAGES,
            B_SFREE = B_SFULL + 1, B_PFULL = B_SFULL + 2, B_DONE = B_SFULL + 3;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

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
      mbar_init(bar(i), (i == B_PFULL || i == B_SFREE) ? 8u : 1u);
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

  if (warp == 0) {
    if (lane == 0 && n_iter > 0) {
      tma_prefetch_desc(&map_k);
      tma_prefetch_desc(&map_v);
      mbar_arrive_expect_tx(bar(B_QFULL), 2 * C::TILE);
      for (int r = 0; r < C::KREG; ++r) {
        tma_load_3d(sbase + C::OFF_Q + r * C::REGION, &map_q, bar(B_QFULL), r * 64, q0, bh);
        tma_load_3d(sbase + C::OFF_DO + r * C::REGION, &map_do, bar(B_QFULL), r * 64, q0, bh);
      }
      const int zkv = b * s.Hkv + g;
      for (int it = 0; it < n_iter; ++it) {
        const int st = it % C::STAGES;
        if (it >= C::STAGES)
          mbar_wait(bar(B_KVEMPTY + st), ((it / C::STAGES) - 1) & 1, wc.timeout_ns, abort_flag,
                    wc.status);
        const int kr = (j_lo + it) * C::BN;
        mbar_arrive_expect_tx(bar(B_KVFULL + st), 2 * C::TILE);
        for (int r = 0; r < C::KREG; ++r) {
          tma_load_3d(sbase + C::OFF_K + st * C::TILE + r * C::REGION, &map_k,
                      bar(B_KVFULL + st), r * 64, kr, zkv);
          tma_load_3d(sbase + C::OFF_V + st * C::TILE + r * C::REGION, &map_v,
                      bar(B_KVFULL + st), r * 64, kr, zkv);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && n_iter > 0) {
      constexpr uint32_t ab = C::BF16 ? 1 : 0;
      constexpr uint32_t idesc_s = make_idesc_f16(kBM, C::BN, ab, 0, 0);
      constexpr uint32_t idesc_q = make_idesc_f16(kBM, C::D, ab, 0, 1);
      // descriptors are built once per operand base; the k-step offsets are
      // added to the start-address field (shared addresses < 256 KB never carry)
      auto issue_score = [&](uint32_t a_base, uint32_t b_base, uint32_t col) {
        const uint64_t ad = make_sdesc(a_base, 16, 1024, 2), bd = make_sdesc(b_base, 16, 1024, 2);
#pragma unroll
        for (int kk = 0; kk < C::D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::REGION + (kk & 3) * 32;
          mma_ss(tmem + col, ad + (off >> 4), bd + (off >> 4), idesc_s, kk > 0);
        }
      };
      mbar_wait(bar(B_QFULL), 0, wc.timeout_ns, abort_flag, wc.status);
      mbar_wait(bar(B_KVFULL + 0), 0, wc.timeout_ns, abort_flag, wc.status);
      tc_fence_after();
      issue_score(sbase + C::OFF_Q, sbase + C::OFF_K, C::S_COL);
      issue_score(sbase + C::OFF_DO, sbase + C::OFF_V, C::DP_COL);
      mma_commit(bar(B_SFULL));
      for (int it = 0; it < n_iter; ++it) {
        const int st = it % C::STAGES;
        const int nst = (it + 1) % C::STAGES;
        const bool more = it + 1 < n_iter;
        if (more) {
          mbar_wait(bar(B_KVFULL + nst), ((it + 1) / C::STAGES) & 1, wc.timeout_ns, abort_flag,
                    wc.status);
          mbar_wait(bar(B_SFREE), it & 1, wc.timeout_ns, abort_flag, wc.status);
          tc_fence_after();
          issue_score(sbase + C::OFF_Q, sbase + C::OFF_K + nst * C::TILE, C::S_COL);
        }
        mbar_wait(bar(B_PFULL), it & 1, wc.timeout_ns, abort_flag, wc.status);
        tc_fence_after();
        // dQ += dS K   (dS from TMEM, K as MN-major B, K = key rows)
        const uint64_t kdesc = make_sdesc(sbase + C::OFF_K + st * C::TILE, C::REGION, 1024, 2);
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk)
          mma_ts(tmem + C::DQ_COL, tmem + C::ds_col(kk),
                 kdesc + ((kk * 16 * 128) >> 4), idesc_q,
                 (it > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar(B_KVEMPTY + st));
        if (more) {
          issue_score(sbase + C::OFF_DO, sbase + C::OFF_V + nst * C::TILE, C::DP_COL);
          mma_commit(bar(B_SFULL));
        }
      }
      mma_commit(bar(B_DONE));
      mbar_wait(bar(B_DONE), 0, wc.timeout_ns, nullptr, wc.status);
    }
  } else if (warp >= 4) {
    const int wg = (warp - 4) >> 2;          // 0: key columns 0-63, 1: 64-127
    const int quarter = warp & 3;
    const int row = q0 + quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const float c = s.scale_log2;
    float nl2 = -INFINITY, nd = 0.f;  // -LSE * log2(e) and -D of this row
    if (row < s.Tq) {
      const int64_t idx = static_cast<int64_t>(bh) * s.Tq + row;
      const float L = lse[idx];
      nl2 = (L == -INFINITY) ? -INFINITY : -L * kLog2e;  // no visible key: P = 0
      nd = -dvec[idx];
    }
    const uint64_t c2 = f2_pack(c, c), nl2x2 = f2_pack(nl2, nl2), ndx2 = f2_pack(nd, nd);
    for (int it = 0; it < n_iter; ++it) {
      const int kb = (j_lo + it) * C::BN + wg * 64;
      mbar_wait(bar(B_SFULL), it & 1, wc.timeout_ns, abort_flag, wc.status);
      tc_fence_after();
      uint32_t sv[64], pv[64];
      tmem_ld32(tmem + lane_base + C::S_COL + wg * 64, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
      tmem_ld32(tmem + lane_base + C::S_COL + wg * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
      tmem_ld32(tmem + lane_base + C::DP_COL + wg * 64, *reinterpret_cast<uint32_t(*)[32]>(&pv[0]));
      tmem_ld32(tmem + lane_base + C::DP_COL + wg * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&pv[32]));
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_SFREE));  // this warp's S and dP columns are in registers
      if (!block_unmasked(s, q0, q0 + kBM, kb, kb + 64)) {
#pragma unroll
        for (int k = 0; k < 64; ++k) {
          const int j = kb + k;
          if (j >= s.Tkv || !key_visible(row, j, s.causal, s.window))
            sv[k] = __float_as_uint(-INFINITY);
        }
      }
      uint32_t ds[32];
#pragma unroll
      for (int k = 0; k < 64; k += 2) {
        // p = 2^(s * scale * log2(e) - LSE2);  ds = p * (dp - D)
        const float2 xf = f2_unpack(
            ffma2(f2_pack(__uint_as_float(sv[k]), __uint_as_float(sv[k + 1])), c2, nl2x2));
        const float p0 = ex2(xf.x), p1 = ex2(xf.y);
        const uint64_t t =
            fadd2(f2_pack(__uint_as_float(pv[k]), __uint_as_float(pv[k + 1])), ndx2);
        const float2 d2 = f2_unpack(fmul2(t, f2_pack(p0, p1)));
        ds[k / 2] = pack2<C::BF16>(d2.x, d2.y);
      }
      tmem_st32(tmem + lane_base + C::DP_COL + wg * 64, ds);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_PFULL));
    }
    // epilogue: warpgroup wg writes head-dim columns [wg * D/2, (wg + 1) * D/2)
    if (n_iter > 0) {
      mbar_wait(bar(B_DONE), 0, wc.timeout_ns, abort_flag, wc.status);
      tc_fence_after();
    }
    using T16 = typename std::conditional<C::BF16, __nv_bfloat16, __half>::type;
    const bool valid = row < s.Tq;
    T16* dst_row = reinterpret_cast<T16*>(dq_out) +
                   (static_cast<int64_t>(bh) * s.Tq + (valid ? row : 0)) * C::D;
    constexpr int HALF = C::D / 2;  // 32, 48 or 64 columns
#pragma unroll 1
    for (int cc = wg * HALF; cc < (wg + 1) * HALF; cc += 16) {
      uint32_t v[16];
      if (n_iter > 0) {
        tmem_ld16(tmem + lane_base + C::DQ_COL + cc, v);
        tmem_ld_wait();
      }
      uint32_t w[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float a = n_iter > 0 ? __uint_as_float(v[2 * k]) * scale : 0.f;
        const float bb = n_iter > 0 ? __uint_as_float(v[2 * k + 1]) * scale : 0.f;
        w[k] = pack2<C::BF16>(a, bb);
      }
      if (valid) {
        uint4* dst = reinterpret_cast<uint4*>(dst_row + cc);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace fa
