// Backward (VJP) attention kernels for sm_103a.
//
// What they compute follows page "mlx-bun 0.0.4: package/src/model/
// flash-attention.ts", backward passes 1-3:
//   pass 1  D_i = rowsum(dO_i o O_i) from the stored O           (fa_bwd_dvec_kernel)
//   pass 2  per KV row block, over every query head of its group and every
//           query tile: p = exp(s - L), dp = dO.v, ds = p (dp - D),
//           dV += p dO, dK += ds q scale                        (fa_bwd_dkv_split2_kernel)
//   pass 3  per query row block, over key tiles: dQ += ds k scale (fa_bwd_dq_serial_kernel)
// and page "[Metal] Add Flash Attention VJP for training", Implementation
// Notes: two kernels instead of atomics, with the dK/dV kernel owning its KV
// rows so the query heads of a GQA group are summed without races; the exp2
// domain for the recomputed probabilities.
//
// GB300 design: the four contractions per tile pair are tcgen05 MMAs. In the
// dK/dV kernel the CTA computes the transposed blocks S^T = K Q^T and
// dP^T = V dO^T (KV rows on the TMEM lanes, one softmax thread per KV row), so
// P^T and dS^T land in TMEM in exactly the layout the next MMAs take as their
// A operand: dV += P^T dO and dK += dS^T Q read them from TMEM, with dO and Q
// as MN-major B operands from the same shared-memory tiles that fed S^T/dP^T.
// The dQ kernel mirrors this with S = Q K^T, dP = dO V^T and dQ += dS K.
#pragma once

#include <type_traits>

#include "fa_common.cuh"

namespace fa {

// ------------------------------------------------------------ pass 1: D-vector
// One group of TPR threads per row; each thread reads 16 bytes of O and dO per
// step (fully coalesced), fp32 accumulation, shuffle reduction in the group.
// The loop bound is uniform over the block, so every lane of a warp reaches
// every shuffle (a row past the end loads zeros and stores nothing).
template <int D, bool BF16>
__global__ void __launch_bounds__(256)
fa_bwd_dvec_kernel(const uint4* __restrict__ o, const uint4* __restrict__ dout,
                   float* __restrict__ dvec, int64_t nrows) {
  constexpr int CHUNKS = D / 8;  // 16-byte chunks per row
  constexpr int TPR = CHUNKS <= 8 ? 8 : (CHUNKS <= 16 ? 16 : 32);
  constexpr int ROWS_PER_BLOCK = 256 / TPR;
  const int sub = threadIdx.x % TPR;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * ROWS_PER_BLOCK;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * ROWS_PER_BLOCK; base < nrows;
       base += stride) {
    const int64_t row = base + threadIdx.x / TPR;
    const bool valid = row < nrows;
    float acc = 0.f;
    for (int ch = sub; ch < CHUNKS; ch += TPR) {
      if (!valid) break;
      const uint4 a = __ldg(o + row * CHUNKS + ch);
      const uint4 b = __ldg(dout + row * CHUNKS + ch);
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
      const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 x = unpack2<BF16>(aw[k]);
        const float2 y = unpack2<BF16>(bw[k]);
        acc = fmaf(x.x, y.x, acc);
        acc = fmaf(x.y, y.y, acc);
      }
    }
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (sub == 0 && valid) dvec[row] = acc;
  }
}

// ------------------------------------------------------------ pass 2: dK / dV
enum : int { kModeDV = 1, kModeDK = 2 };

template <int D_, int BMQ_, int STAGES_, bool BF16_, int MODE_>
struct DkvSplitCfg {
  static constexpr int D = D_;
  static constexpr int BMQ = BMQ_;   // query rows per inner tile (N of S^T)
  static constexpr int STAGES = STAGES_;
  static constexpr bool BF16 = BF16_;
  static constexpr int MODE = MODE_;
  static constexpr bool DO_DV = (MODE & kModeDV) != 0;
  static constexpr bool DO_DK = (MODE & kModeDK) != 0;
  static constexpr int DP = (D + 63) / 64 * 64;
  static constexpr int KREG = DP / 64;
  static constexpr int KV_REGION = kBM * 128;      // KV block: 128 rows
  static constexpr int Q_REGION = BMQ * 128;
  static constexpr int KV_TILE = KREG * KV_REGION;
  static constexpr int Q_TILE = KREG * Q_REGION;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KV_TILE;
  static constexpr int OFF_Q = OFF_V + (DO_DK ? KV_TILE : 0);
  static constexpr int OFF_DO = OFF_Q + STAGES * Q_TILE;
  static constexpr int OFF_STATS = OFF_DO + STAGES * Q_TILE;  // [2][2][BMQ] floats
  static constexpr int OFF_BAR = OFF_STATS + 2 * 2 * BMQ * 4;
  // barriers: kv_full, q_full[S], q_empty[S], s_full, p_full, done
  static constexpr int NBAR = 1 + 2 * STAGES + 3;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int THREADS = 256;
  static constexpr int S_COL = 0;
  static constexpr int DP_COL = 128;
  static constexpr int DV_COL = 256;
  static constexpr int DK_COL = DO_DV ? 256 + D : 256;
  static_assert(!DO_DV || !DO_DK || 2 * D <= 256, "TMEM budget for dV and dK together");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
  static_assert(BMQ == 64 || BMQ == 128, "query tile");
};

// One CTA of a pass over KV block `linear` of the grid order (the tensor maps
// are the kernel's own parameters).
template <class C>
__device__ __forceinline__ void dkv_split_body(const CUtensorMap& map_q, const CUtensorMap& map_k,
                                               const CUtensorMap& map_v, const CUtensorMap& map_do,
                                               const float* __restrict__ lse,
                                               const float* __restrict__ dvec,
                                               void* __restrict__ dk_out, void* __restrict__ dv_out,
                                               float scale, const AttnShape& s,
                                               const TileOrder& order, const WaitCfg& wc,
                                               int linear) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  auto bar = [&](int i) { return smem_u32(bars + i); };
  const int B_KVFULL = 0, B_QFULL = 1, B_QEMPTY = 1 + C::STAGES, B_SFULL = 1 + 2 * C::STAGES,
            B_PFULL = B_SFULL + 1, B_DONE = B_PFULL + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  float* stats = reinterpret_cast<float*>(smem + C::OFF_STATS);  // [buf][lse2|dvec][BMQ]

  int bg, kvt;  // (b * Hkv + g, block of 128 KV rows)
  decode_tile(linear, order, &bg, &kvt);
  const int b = bg / s.Hkv, g = bg % s.Hkv;
  const int reps = s.Hq / s.Hkv;
  const int k0 = kvt * kBM;
  int qf, ql;
  query_range(s, k0, min(s.Tkv, k0 + kBM), &qf, &ql);
  const int i_lo = qf / C::BMQ;
  const int i_hi = (ql + C::BMQ - 1) / C::BMQ;
  const int n_qt = max(0, i_hi - i_lo);
  const int n_iter = n_qt * reps;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < C::NBAR; ++i) mbar_init(bar(i), i == B_PFULL ? 128u : 1u);
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
    if (n_iter > 0) {
      // the whole warp runs the loop (a lone active lane whose siblings wait at
      // the final barrier issues far slower); one elected lane issues
      const bool leader = elect_one_sync();
      if (leader) tma_prefetch_desc(&map_q);
      if (leader) tma_prefetch_desc(&map_do);
      if (leader) mbar_arrive_expect_tx(bar(B_KVFULL), (C::DO_DK ? 2 : 1) * C::KV_TILE);
      for (int r = 0; r < C::KREG; ++r) {
        if (leader) tma_load_3d(sbase + C::OFF_K + r * C::KV_REGION, &map_k, bar(B_KVFULL), r * 64, k0, bg);
        if (C::DO_DK)
          if (leader) tma_load_3d(sbase + C::OFF_V + r * C::KV_REGION, &map_v, bar(B_KVFULL), r * 64, k0, bg);
      }
      for (int it = 0; it < n_iter; ++it) {
        const int st = it % C::STAGES;
        const int h = g * reps + it / n_qt;
        const int i0 = (i_lo + it % n_qt) * C::BMQ;
        if (it >= C::STAGES)
          mbar_wait(bar(B_QEMPTY + st), ((it / C::STAGES) - 1) & 1, wc.timeout_cycles, abort_flag,
                    wc.status);
        if (leader) mbar_arrive_expect_tx(bar(B_QFULL + st), 2 * C::Q_TILE);
        const int zq = b * s.Hq + h;
        for (int r = 0; r < C::KREG; ++r) {
          if (leader) tma_load_3d(sbase + C::OFF_Q + st * C::Q_TILE + r * C::Q_REGION, &map_q,
                      bar(B_QFULL + st), r * 64, i0, zq);
          if (leader) tma_load_3d(sbase + C::OFF_DO + st * C::Q_TILE + r * C::Q_REGION, &map_do,
                      bar(B_QFULL + st), r * 64, i0, zq);
        }
      }
    }
  } else if (warp == 1) {
    if (n_iter > 0) {
      // the whole warp runs the loop (a lone active lane whose siblings wait at
      // the final barrier issues far slower); one elected lane issues
      const bool leader = elect_one_sync();
      constexpr uint32_t ab = C::BF16 ? 1 : 0;
      constexpr uint32_t idesc_st = make_idesc_f16(kBM, C::BMQ, ab, 0, 0);  // S^T, dP^T
      constexpr uint32_t idesc_acc = make_idesc_f16(kBM, C::D, ab, 0, 1);   // dV, dK
      mbar_wait(bar(B_KVFULL), 0, wc.timeout_cycles, abort_flag, wc.status);
      for (int it = 0; it < n_iter; ++it) {
        const int st = it % C::STAGES;
        mbar_wait(bar(B_QFULL + st), (it / C::STAGES) & 1, wc.timeout_cycles, abort_flag, wc.status);
        tc_fence_after();
        const uint32_t qa = sbase + C::OFF_Q + st * C::Q_TILE;
        const uint32_t da = sbase + C::OFF_DO + st * C::Q_TILE;
        // S^T = K Q^T  and  dP^T = V dO^T   (K-major operands, K = head dim)
#pragma unroll
        for (int kk = 0; kk < C::D / 16; ++kk) {
          const uint32_t off = (kk & 3) * 32;
          const uint64_t bq = make_sdesc(qa + (kk >> 2) * C::Q_REGION + off, 16, 1024, 2);
          const uint64_t ak = make_sdesc(sbase + C::OFF_K + (kk >> 2) * C::KV_REGION + off, 16, 1024, 2);
          if (leader) mma_ss(tmem + C::S_COL, ak, bq, idesc_st, kk > 0);
          if (C::DO_DK) {
            const uint64_t bd = make_sdesc(da + (kk >> 2) * C::Q_REGION + off, 16, 1024, 2);
            const uint64_t av = make_sdesc(sbase + C::OFF_V + (kk >> 2) * C::KV_REGION + off, 16, 1024, 2);
            if (leader) mma_ss(tmem + C::DP_COL, av, bd, idesc_st, kk > 0);
          }
        }
        if (leader) mma_commit(bar(B_SFULL));
        mbar_wait(bar(B_PFULL), it & 1, wc.timeout_cycles, abort_flag, wc.status);
        tc_fence_after();
        // dV += P^T dO  and  dK += dS^T Q   (A from TMEM, B MN-major, K = query rows)
#pragma unroll
        for (int kk = 0; kk < C::BMQ / 16; ++kk) {
          const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
          if (C::DO_DV) {
            const uint64_t bd = make_sdesc(da + kk * 16 * 128, C::Q_REGION, 1024, 2);
            if (leader) mma_ts(tmem + C::DV_COL, tmem + C::S_COL + kk * 8, bd, idesc_acc, acc);
          }
          if (C::DO_DK) {
            const uint64_t bq = make_sdesc(qa + kk * 16 * 128, C::Q_REGION, 1024, 2);
            if (leader) mma_ts(tmem + C::DK_COL, tmem + C::DP_COL + kk * 8, bq, idesc_acc, acc);
          }
        }
        if (leader) mma_commit(bar(B_QEMPTY + st));
      }
      if (leader) mma_commit(bar(B_DONE));
      mbar_wait(bar(B_DONE), 0, wc.timeout_cycles, nullptr, wc.status);
    }
  } else if (warp >= 4) {
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;        // KV row within the block (TMEM lane)
    const int krow = k0 + r;
    const int tid = threadIdx.x - 128;        // 0..127
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const float c = s.scale_log2;
    for (int it = 0; it < n_iter; ++it) {
      const int h = g * reps + it / n_qt;
      const int i0 = (i_lo + it % n_qt) * C::BMQ;
      float* lse_s = stats + (it & 1) * 2 * C::BMQ;
      float* dv_s = lse_s + C::BMQ;
      if (tid < C::BMQ) {
        const int i = i0 + tid;
        float l2 = INFINITY, dd = 0.f;  // rows past Tq: P = 0
        if (i < s.Tq) {
          const int64_t idx = static_cast<int64_t>(b * s.Hq + h) * s.Tq + i;
          const float L = lse[idx];
          l2 = (L == -INFINITY) ? INFINITY : L * kLog2e;  // row with no visible key: P = 0
          dd = dvec[idx];
        }
        lse_s[tid] = l2;
        dv_s[tid] = dd;
      }
      named_bar_sync(1, 128);
      mbar_wait(bar(B_SFULL), it & 1, wc.timeout_cycles, abort_flag, wc.status);
      tc_fence_after();
      const bool need_mask = !block_unmasked(s, i0, i0 + C::BMQ, k0, k0 + kBM);
      int mlo, mhi;  // query columns of this tile that see this thread's key
      visible_queries(s, krow, i0, &mlo, &mhi);
#pragma unroll
      for (int cc = 0; cc < C::BMQ; cc += 32) {
        uint32_t sv[32], pv[32];
        tmem_ld32(tmem + lane_base + C::S_COL + cc, sv);
        if (C::DO_DK) tmem_ld32(tmem + lane_base + C::DP_COL + cc, pv);
        tmem_ld_wait();
        uint32_t pp[16], ds[16];
#pragma unroll
        for (int k = 0; k < 32; k += 2) {
          float p[2], d2[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int q = cc + k + e;
            float sc = __uint_as_float(sv[k + e]);
            if (need_mask && !(q >= mlo && q < mhi)) sc = -INFINITY;
            p[e] = ex2(fmaf(sc, c, -lse_s[q]));
            d2[e] = C::DO_DK ? p[e] * (__uint_as_float(pv[k + e]) - dv_s[q]) : 0.f;
          }
          pp[k / 2] = pack2<C::BF16>(p[0], p[1]);
          ds[k / 2] = pack2<C::BF16>(d2[0], d2[1]);
        }
        if (C::DO_DV) tmem_st16(tmem + lane_base + C::S_COL + cc / 2, pp);
        if (C::DO_DK) tmem_st16(tmem + lane_base + C::DP_COL + cc / 2, ds);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(B_PFULL));
    }
    // ---------------------------------------------------------- epilogue
    if (n_iter > 0) {
      // the last q_empty commit covers every MMA: wait for it through B_DONE's
      // producer-side twin, the final q_empty phase of the last stage
      const int last = n_iter - 1;
      mbar_wait(bar(B_QEMPTY + last % C::STAGES), (last / C::STAGES) & 1, wc.timeout_cycles,
                abort_flag, wc.status);
      tc_fence_after();
    }
    using T16 = typename std::conditional<C::BF16, __nv_bfloat16, __half>::type;
    const bool valid = krow < s.Tkv;
    const int64_t orow = (static_cast<int64_t>(bg) * s.Tkv + (valid ? krow : 0)) * C::D;
#pragma unroll 1
    for (int which = 0; which < 2; ++which) {
      if (which == 0 && !C::DO_DV) continue;
      if (which == 1 && !C::DO_DK) continue;
      const uint32_t col = which == 0 ? C::DV_COL : C::DK_COL;
      const float mul = which == 0 ? 1.f : scale;
      T16* dst_row = reinterpret_cast<T16*>(which == 0 ? dv_out : dk_out) + orow;
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
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Both passes in one grid: CTA 2u runs the dV pass and CTA 2u + 1 the dK pass
// of KV block u, so the two passes of a block run side by side (twice the CTAs
// in flight of two back-to-back launches, and their Q / dO reads share L2).
template <class CV, class CK>
__global__ void __launch_bounds__(CV::THREADS, 1)
fa_bwd_dkv_split2_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                         const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                         const float* __restrict__ lse, const float* __restrict__ dvec,
                         void* __restrict__ dk_out, void* __restrict__ dv_out, float scale,
                         AttnShape s, TileOrder order, WaitCfg wc) {
  static_assert(CV::THREADS == CK::THREADS && CV::BMQ == CK::BMQ, "one launch shape");
  if ((blockIdx.x & 1) == 0)
    dkv_split_body<CV>(map_q, map_k, map_v, map_do, lse, dvec, dk_out, dv_out, scale, s, order,
                       wc, blockIdx.x >> 1);
  else
    dkv_split_body<CK>(map_q, map_k, map_v, map_do, lse, dvec, dk_out, dv_out, scale, s, order,
                       wc, blockIdx.x >> 1);
}

// ------------------------------------------------------------------ pass 3: dQ
template <int D_, int BN_, int STAGES_, bool BF16_>
struct DqSerialCfg {
  static constexpr int D = D_;
  static constexpr int BN = BN_;
  static constexpr int STAGES = STAGES_;
  static constexpr bool BF16 = BF16_;
  static constexpr int DP = (D + 63) / 64 * 64;
  static constexpr int KREG = DP / 64;
  static constexpr int Q_REGION = kBM * 128;
  static constexpr int KV_REGION = BN * 128;
  static constexpr int Q_TILE = KREG * Q_REGION;
  static constexpr int KV_TILE = KREG * KV_REGION;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = OFF_Q + Q_TILE;
  static constexpr int OFF_K = OFF_DO + Q_TILE;
  static constexpr int OFF_V = OFF_K + STAGES * KV_TILE;
  static constexpr int OFF_BAR = OFF_V + STAGES * KV_TILE;
  // barriers: q_full, kv_full[S], kv_empty[S], s_full, p_full, done
  static constexpr int NBAR = 1 + 2 * STAGES + 3;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int THREADS = 256;
  static constexpr int S_COL = 0;
  static constexpr int DP_COL = 128;
  static constexpr int DQ_COL = 256;
  static_assert(BN % 32 == 0 && BN <= 128, "key tile");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
fa_bwd_dq_serial_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
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
            B_PFULL = B_SFULL + 1, B_DONE = B_PFULL + 1;
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
  const int j_hi = (kl + C::BN - 1) / C::BN;
  const int n_iter = max(0, j_hi - j_lo);

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < C::NBAR; ++i) mbar_init(bar(i), i == B_PFULL ? 128u : 1u);
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
    if (n_iter > 0) {
      // the whole warp runs the loop (a lone active lane whose siblings wait at
      // the final barrier issues far slower); one elected lane issues
      const bool leader = elect_one_sync();
      if (leader) tma_prefetch_desc(&map_k);
      if (leader) tma_prefetch_desc(&map_v);
      if (leader) mbar_arrive_expect_tx(bar(B_QFULL), 2 * C::Q_TILE);
      for (int r = 0; r < C::KREG; ++r) {
        if (leader) tma_load_3d(sbase + C::OFF_Q + r * C::Q_REGION, &map_q, bar(B_QFULL), r * 64, q0, bh);
        if (leader) tma_load_3d(sbase + C::OFF_DO + r * C::Q_REGION, &map_do, bar(B_QFULL), r * 64, q0, bh);
      }
      const int zkv = b * s.Hkv + g;
      for (int it = 0; it < n_iter; ++it) {
        const int st = it % C::STAGES;
        if (it >= C::STAGES)
          mbar_wait(bar(B_KVEMPTY + st), ((it / C::STAGES) - 1) & 1, wc.timeout_cycles, abort_flag,
                    wc.status);
        const int kr = (j_lo + it) * C::BN;
        if (leader) mbar_arrive_expect_tx(bar(B_KVFULL + st), 2 * C::KV_TILE);
        for (int r = 0; r < C::KREG; ++r) {
          if (leader) tma_load_3d(sbase + C::OFF_K + st * C::KV_TILE + r * C::KV_REGION, &map_k,
                      bar(B_KVFULL + st), r * 64, kr, zkv);
          if (leader) tma_load_3d(sbase + C::OFF_V + st * C::KV_TILE + r * C::KV_REGION, &map_v,
                      bar(B_KVFULL + st), r * 64, kr, zkv);
        }
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
      mbar_wait(bar(B_QFULL), 0, wc.timeout_cycles, abort_flag, wc.status);
      for (int it = 0; it < n_iter; ++it) {
        const int st = it % C::STAGES;
        mbar_wait(bar(B_KVFULL + st), (it / C::STAGES) & 1, wc.timeout_cycles, abort_flag, wc.status);
        tc_fence_after();
        const uint32_t ka = sbase + C::OFF_K + st * C::KV_TILE;
        const uint32_t va = sbase + C::OFF_V + st * C::KV_TILE;
        // S = Q K^T and dP = dO V^T
#pragma unroll
        for (int kk = 0; kk < C::D / 16; ++kk) {
          const uint32_t off = (kk & 3) * 32;
          const uint64_t aq = make_sdesc(sbase + C::OFF_Q + (kk >> 2) * C::Q_REGION + off, 16, 1024, 2);
          const uint64_t bk = make_sdesc(ka + (kk >> 2) * C::KV_REGION + off, 16, 1024, 2);
          if (leader) mma_ss(tmem + C::S_COL, aq, bk, idesc_s, kk > 0);
          const uint64_t ad = make_sdesc(sbase + C::OFF_DO + (kk >> 2) * C::Q_REGION + off, 16, 1024, 2);
          const uint64_t bv = make_sdesc(va + (kk >> 2) * C::KV_REGION + off, 16, 1024, 2);
          if (leader) mma_ss(tmem + C::DP_COL, ad, bv, idesc_s, kk > 0);
        }
        if (leader) mma_commit(bar(B_SFULL));
        mbar_wait(bar(B_PFULL), it & 1, wc.timeout_cycles, abort_flag, wc.status);
        tc_fence_after();
        // dQ += dS K   (dS from TMEM, K as MN-major B)
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk) {
          const uint64_t bk = make_sdesc(ka + kk * 16 * 128, C::KV_REGION, 1024, 2);
          if (leader) mma_ts(tmem + C::DQ_COL, tmem + C::S_COL + kk * 8, bk, idesc_q, (it > 0 || kk > 0) ? 1u : 0u);
        }
        if (leader) mma_commit(bar(B_KVEMPTY + st));
      }
      if (leader) mma_commit(bar(B_DONE));
      mbar_wait(bar(B_DONE), 0, wc.timeout_cycles, nullptr, wc.status);
    }
  } else if (warp >= 4) {
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int row = q0 + r;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const float c = s.scale_log2;
    float l2 = INFINITY, dd = 0.f;
    if (row < s.Tq) {
      const int64_t idx = static_cast<int64_t>(bh) * s.Tq + row;
      const float L = lse[idx];
      l2 = (L == -INFINITY) ? INFINITY : L * kLog2e;
      dd = dvec[idx];
    }
    for (int it = 0; it < n_iter; ++it) {
      const int kb = (j_lo + it) * C::BN;
      mbar_wait(bar(B_SFULL), it & 1, wc.timeout_cycles, abort_flag, wc.status);
      tc_fence_after();
      const bool need_mask = !block_unmasked(s, q0, q0 + kBM, kb, kb + C::BN);
      int mlo, mhi;  // key columns of this tile this thread's query sees
      visible_keys(s, row, kb, &mlo, &mhi);
#pragma unroll
      for (int cc = 0; cc < C::BN; cc += 32) {
        uint32_t sv[32], pv[32];
        tmem_ld32(tmem + lane_base + C::S_COL + cc, sv);
        tmem_ld32(tmem + lane_base + C::DP_COL + cc, pv);
        tmem_ld_wait();
        uint32_t ds[16];
#pragma unroll
        for (int k = 0; k < 32; k += 2) {
          float d2[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int j = cc + k + e;
            float sc = __uint_as_float(sv[k + e]);
            if (need_mask && !(j >= mlo && j < mhi)) sc = -INFINITY;
            const float p = ex2(fmaf(sc, c, -l2));
            d2[e] = p * (__uint_as_float(pv[k + e]) - dd);
          }
          ds[k / 2] = pack2<C::BF16>(d2[0], d2[1]);
        }
        tmem_st16(tmem + lane_base + C::S_COL + cc / 2, ds);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(B_PFULL));
    }
    if (n_iter > 0) {
      const int last = n_iter - 1;
      mbar_wait(bar(B_KVEMPTY + last % C::STAGES), (last / C::STAGES) & 1, wc.timeout_cycles,
                abort_flag, wc.status);
      tc_fence_after();
    }
    using T16 = typename std::conditional<C::BF16, __nv_bfloat16, __half>::type;
    const bool valid = row < s.Tq;
    T16* dst_row = reinterpret_cast<T16*>(dq_out) +
                   (static_cast<int64_t>(bh) * s.Tq + (valid ? row : 0)) * C::D;
#pragma unroll 1
    for (int cc = 0; cc < C::D; cc += 32) {
      uint32_t v[32];
      if (n_iter > 0) {
        tmem_ld32(tmem + lane_base + C::DQ_COL + cc, v);
        tmem_ld_wait();
      }
      uint32_t w[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float a = n_iter > 0 ? __uint_as_float(v[2 * k]) * scale : 0.f;
        const float bb = n_iter > 0 ? __uint_as_float(v[2 * k + 1]) * scale : 0.f;
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

}  // namespace fa
