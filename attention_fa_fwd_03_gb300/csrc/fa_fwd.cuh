// Forward attention kernel for sm_103a: tcgen05 MMAs with TMEM accumulators,
// TMA-fed K/V ring, warp-specialised roles, exp2-domain online softmax.
//
// What it computes follows page "mlx-bun 0.0.4: package/src/model/
// flash-attention.ts", forward shader: per query row an online softmax over
// key tiles (running max m, running sum l, rescaled accumulator o), result
// O = o / l and LSE = m + ln(l); a key tile hidden from the whole query tile is
// skipped, and a tile with no visible key for a row changes nothing for it.
// The exp2 domain (scores pre-multiplied by log2 e) follows page "[Metal] Add
// Flash Attention VJP for training", Implementation Notes.
//
// GB300 design (not the pages'): one CTA owns NQ query tiles of 128 rows of
// one (batch, head). Roles per CTA:
//   warp 0       TMA producer: Q tiles once, then K_j / V_j into a STAGES ring
//   warp 1       MMA issuer (one thread): S_t = Q_t K_j^T into TMEM, then
//                O_t += P_t V_j with P_t read straight from TMEM
//   warp 2       TMEM allocator
//   warpgroup 1+t  softmax of query tile t: one thread per row (TMEM lane),
//                writes P_t (16-bit) over its own S_t columns, rescales O_t
//                in TMEM when the running max grows by more than 2^8, and
//                finally normalises O_t and writes O and LSE.
// With NQ = 2 the two softmax warpgroups ping-pong: while one computes its
// softmax the tensor core works on the other tile's MMAs.
#pragma once

#include "fa_common.cuh"

namespace fa {

// Lazy-rescale threshold in the log2 domain: the running max used for the
// exponentials is only raised when the true max exceeds it by more than this,
// so unnormalised P stays below 2^8. The final O = o / l and LSE = m + log2 l
// use the same max, so the result is exact.
constexpr float kRescaleThreshold = 8.0f;

template <int D_, int NQ_, int BN_, int STAGES_, bool BF16_>
struct FwdCfg {
  static constexpr int D = D_;
  static constexpr int NQ = NQ_;
  static constexpr int BN = BN_;
  static constexpr int STAGES = STAGES_;
  static constexpr bool BF16 = BF16_;
  static constexpr int DP = (D + 63) / 64 * 64;  // D padded to whole 128-byte rows
  static constexpr int KREG = DP / 64;           // 64-element column blocks of a tile
  static constexpr int Q_REGION = kBM * 128;     // bytes of one column block of a Q tile
  static constexpr int KV_REGION = BN * 128;
  static constexpr int Q_TILE = KREG * Q_REGION;
  static constexpr int KV_TILE = KREG * KV_REGION;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + NQ * Q_TILE;
  static constexpr int OFF_V = OFF_K + STAGES * KV_TILE;
  static constexpr int OFF_BAR = OFF_V + STAGES * KV_TILE;
  // barriers: q_full, k_full[S], v_full[S], kv_empty[S], s_full[NQ], p_full[NQ],
  // o_ready[NQ], drain
  static constexpr int NBAR = 1 + 3 * STAGES + 3 * NQ + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack
  static constexpr int THREADS = 128 + NQ * 128;
  static constexpr int S_COL(int t) { return t * 128; }
  static constexpr int O_COL(int t) { return 256 + t * 128; }
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(BN % 32 == 0 && BN <= 128, "key tile");
  static_assert(NQ * 128 <= 256 && (NQ == 1 || D <= 128), "TMEM budget");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
fa_fwd_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
              const __grid_constant__ CUtensorMap map_v, void* __restrict__ o_out,
              float* __restrict__ lse_out, AttnShape s, TileOrder order, WaitCfg wc) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  auto bar = [&](int i) { return smem_u32(bars + i); };
  const int B_QFULL = 0, B_KFULL = 1, B_VFULL = 1 + C::STAGES, B_KVEMPTY = 1 + 2 * C::STAGES,
            B_SFULL = 1 + 3 * C::STAGES, B_PFULL = B_SFULL + C::NQ, B_OREADY = B_PFULL + C::NQ,
            B_DRAIN = B_OREADY + C::NQ;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  // ---- work item: a (batch, head) and a block of NQ*128 query rows
  int bh, qblk;
  decode_tile(blockIdx.x, order, &bh, &qblk);
  const int b = bh / s.Hq, h = bh % s.Hq;
  const int g = h / (s.Hq / s.Hkv);
  const int q0 = qblk * (C::NQ * kBM);
  int k_first, k_last;
  key_range(s, q0, min(s.Tq, q0 + C::NQ * kBM), &k_first, &k_last);
  const int j_lo = k_first / C::BN;
  const int j_hi = (k_last + C::BN - 1) / C::BN;
  const int n_iter = max(0, j_hi - j_lo);

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < C::NBAR; ++i)
      mbar_init(bar(i), (i >= B_PFULL && i < B_PFULL + C::NQ) ? 128u : 1u);
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (n_iter > 0) {
      // the whole warp runs the loop (a lone active lane whose siblings wait at
      // the final barrier issues far slower); one elected lane issues
      const bool leader = elect_one_sync();
      if (leader) tma_prefetch_desc(&map_q);
      if (leader) tma_prefetch_desc(&map_k);
      if (leader) tma_prefetch_desc(&map_v);
      if (leader) mbar_arrive_expect_tx(bar(B_QFULL), C::NQ * C::Q_TILE);
      for (int t = 0; t < C::NQ; ++t)
        for (int r = 0; r < C::KREG; ++r)
          if (leader) tma_load_3d(sbase + C::OFF_Q + t * C::Q_TILE + r * C::Q_REGION, &map_q, bar(B_QFULL),
                      r * 64, q0 + t * kBM, bh);
      const int zkv = b * s.Hkv + g;
      for (int it = 0; it < n_iter; ++it) {
        const int st = it % C::STAGES;
        if (it >= C::STAGES)
          mbar_wait(bar(B_KVEMPTY + st), ((it / C::STAGES) - 1) & 1, wc.timeout_cycles, abort_flag,
                    wc.status);
        const int krow = (j_lo + it) * C::BN;
        if (leader) mbar_arrive_expect_tx(bar(B_KFULL + st), C::KV_TILE);
        for (int r = 0; r < C::KREG; ++r)
          if (leader) tma_load_3d(sbase + C::OFF_K + st * C::KV_TILE + r * C::KV_REGION, &map_k,
                      bar(B_KFULL + st), r * 64, krow, zkv);
        if (leader) mbar_arrive_expect_tx(bar(B_VFULL + st), C::KV_TILE);
        for (int r = 0; r < C::KREG; ++r)
          if (leader) tma_load_3d(sbase + C::OFF_V + st * C::KV_TILE + r * C::KV_REGION, &map_v,
                      bar(B_VFULL + st), r * 64, krow, zkv);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer
    if (n_iter > 0) {
      // the whole warp runs the loop (a lone active lane whose siblings wait at
      // the final barrier issues far slower); one elected lane issues
      const bool leader = elect_one_sync();
      constexpr uint32_t idesc_s = make_idesc_f16(kBM, C::BN, C::BF16 ? 1 : 0, 0, 0);
      constexpr uint32_t idesc_o = make_idesc_f16(kBM, C::D, C::BF16 ? 1 : 0, 0, 1);
      auto issue_s = [&](int t, int st) {
        const uint32_t qa = sbase + C::OFF_Q + t * C::Q_TILE;
        const uint32_t ka = sbase + C::OFF_K + st * C::KV_TILE;
#pragma unroll
        for (int kk = 0; kk < C::D / 16; ++kk) {
          const uint32_t off = (kk & 3) * 32;  // 16 elements = 32 bytes along K
          const uint64_t ad = make_sdesc(qa + (kk >> 2) * C::Q_REGION + off, 16, 1024, 2);
          const uint64_t bd = make_sdesc(ka + (kk >> 2) * C::KV_REGION + off, 16, 1024, 2);
          if (leader) mma_ss(tmem + C::S_COL(t), ad, bd, idesc_s, kk > 0);
        }
      };
      auto issue_pv = [&](int t, int st, bool acc) {
        const uint32_t va = sbase + C::OFF_V + st * C::KV_TILE;
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk) {
          const uint64_t bd = make_sdesc(va + kk * 16 * 128, C::KV_REGION, 1024, 2);
          if (leader) mma_ts(tmem + C::O_COL(t), tmem + C::S_COL(t) + kk * 8, bd, idesc_o,
                 (acc || kk > 0) ? 1u : 0u);
        }
      };
      mbar_wait(bar(B_QFULL), 0, wc.timeout_cycles, abort_flag, wc.status);
      mbar_wait(bar(B_KFULL + 0), 0, wc.timeout_cycles, abort_flag, wc.status);
      tc_fence_after();
      for (int t = 0; t < C::NQ; ++t) {
        if (leader) issue_s(t, 0);
        if (leader) mma_commit(bar(B_SFULL + t));
      }
      for (int it = 0; it < n_iter; ++it) {
        const int st = it % C::STAGES;
        const int nst = (it + 1) % C::STAGES;
        mbar_wait(bar(B_VFULL + st), (it / C::STAGES) & 1, wc.timeout_cycles, abort_flag, wc.status);
        for (int t = 0; t < C::NQ; ++t) {
          mbar_wait(bar(B_PFULL + t), it & 1, wc.timeout_cycles, abort_flag, wc.status);
          tc_fence_after();
          if (leader) issue_pv(t, st, it > 0);
          if (leader) mma_commit(bar(B_OREADY + t));
          if (it + 1 < n_iter) {
            if (t == 0) {
              mbar_wait(bar(B_KFULL + nst), ((it + 1) / C::STAGES) & 1, wc.timeout_cycles, abort_flag,
                        wc.status);
              tc_fence_after();
            }
            if (leader) issue_s(t, nst);
            if (leader) mma_commit(bar(B_SFULL + t));
          }
        }
        if (leader) mma_commit(bar(B_KVEMPTY + st));
      }
      // make sure nothing is in flight before TMEM is released
      if (leader) mma_commit(bar(B_DRAIN));
      mbar_wait(bar(B_DRAIN), 0, wc.timeout_cycles, nullptr, wc.status);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------- softmax
    const int t = (warp - 4) >> 2;              // query tile of this warpgroup
    const int quarter = warp & 3;               // TMEM lane quarter of this warp
    const int r = quarter * 32 + lane;          // row within the tile
    const int row = q0 + t * kBM + r;
    const int tq_lo = q0 + t * kBM;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t s_addr = tmem + lane_base + C::S_COL(t);
    const uint32_t o_addr = tmem + lane_base + C::O_COL(t);
    const float c = s.scale_log2;

    float m_used = -INFINITY;  // max used for the exponentials (log2 domain)
    float l = 0.f;
    for (int it = 0; it < n_iter; ++it) {
      const int k0 = (j_lo + it) * C::BN;
      mbar_wait(bar(B_SFULL + t), it & 1, wc.timeout_cycles, abort_flag, wc.status);
      tc_fence_after();
      uint32_t sr[C::BN];
#pragma unroll
      for (int cc = 0; cc < C::BN; cc += 32)
        tmem_ld32(s_addr + cc, *reinterpret_cast<uint32_t(*)[32]>(&sr[cc]));
      tmem_ld_wait();
      float sv[C::BN];
#pragma unroll
      for (int k = 0; k < C::BN; ++k) sv[k] = __uint_as_float(sr[k]);
      if (!block_unmasked(s, tq_lo, tq_lo + kBM, k0, k0 + C::BN)) {
#pragma unroll
        for (int k = 0; k < C::BN; ++k)
          if (k0 + k >= s.Tkv || !key_visible(row, k0 + k, s.causal, s.window)) sv[k] = -INFINITY;
      }
      // row max over 8 independent chains (a single chain is 128 dependent
      // instructions long)
      float m8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) m8[e] = -INFINITY;
#pragma unroll
      for (int k = 0; k < C::BN; ++k) m8[k & 7] = fmaxf(m8[k & 7], sv[k]);
      float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                       fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      mx *= c;
      float alpha = 1.f;
      const bool grow = mx > m_used + kRescaleThreshold || (m_used == -INFINITY && mx > -INFINITY);
      if (grow) {
        alpha = ex2(m_used - mx);  // 0 when m_used = -inf
        m_used = mx;
      }
      const float mexp = (m_used == -INFINITY) ? 0.f : m_used;
      // p = 2^(s c - m): arguments two at a time (f32x2), the row sum in four
      // independent two-lane accumulators
      const uint64_t c2 = f2_pack(c, c), nm2 = f2_pack(-mexp, -mexp);
      uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
      for (int cc = 0; cc < C::BN; cc += 32) {
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 32; k += 2) {
          const float2 x = f2_unpack(ffma2(f2_pack(sv[cc + k], sv[cc + k + 1]), c2, nm2));
          const float p0 = ex2(x.x), p1 = ex2(x.y);
          acc[(k / 2) & 3] = fadd2(acc[(k / 2) & 3], f2_pack(p0, p1));
          pk[k / 2] = pack2<C::BF16>(p0, p1);
        }
        // P overwrites the (already loaded) S columns: 2 values per column
        tmem_st16(s_addr + cc / 2, pk);
      }
      const float2 a01 = f2_unpack(fadd2(acc[0], acc[1])), a23 = f2_unpack(fadd2(acc[2], acc[3]));
      const float rs = (a01.x + a01.y) + (a23.x + a23.y);
      l = l * alpha + rs;
      if (it > 0 && __any_sync(0xffffffffu, grow)) {
        // O_t holds the sum of the previous tiles: wait for the last of them.
        mbar_wait(bar(B_OREADY + t), (it - 1) & 1, wc.timeout_cycles, abort_flag, wc.status);
        tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < C::D; cc += 32) {
          uint32_t ov[32];
          tmem_ld32(o_addr + cc, ov);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 32; ++k) ov[k] = __float_as_uint(__uint_as_float(ov[k]) * alpha);
          tmem_st32(o_addr + cc, ov);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(B_PFULL + t));
    }

    // ------------------------------------------------------------ epilogue
    if (n_iter > 0) {
      mbar_wait(bar(B_OREADY + t), (n_iter - 1) & 1, wc.timeout_cycles, abort_flag, wc.status);
      tc_fence_after();
    }
    const bool valid = row < s.Tq;
    const float inv_l = l > 0.f ? 1.f / l : 0.f;
    using T16 = typename std::conditional<C::BF16, __nv_bfloat16, __half>::type;
    T16* orow = reinterpret_cast<T16*>(o_out) +
                ((static_cast<int64_t>(bh) * s.Tq + (valid ? row : 0)) * C::D);
#pragma unroll 1
    for (int cc = 0; cc < C::D; cc += 32) {
      uint32_t ov[32];
      if (n_iter > 0) {
        tmem_ld32(o_addr + cc, ov);
        tmem_ld_wait();
      }
      uint32_t w[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float a = n_iter > 0 ? __uint_as_float(ov[2 * k]) * inv_l : 0.f;
        const float bb = n_iter > 0 ? __uint_as_float(ov[2 * k + 1]) * inv_l : 0.f;
        w[k] = pack2<C::BF16>(a, bb);
      }
      if (valid) {
        uint4* dst = reinterpret_cast<uint4*>(orow + cc);
#pragma unroll
        for (int k = 0; k < 4; ++k) dst[k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
      }
    }
    if (valid)
      lse_out[static_cast<int64_t>(bh) * s.Tq + row] =
          l > 0.f ? (m_used + __log2f(l)) * kLn2 : -INFINITY;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace fa
