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
//   warps 0, 3   TMA producers: Q tiles once per block and the K ring
//                (warp 0), the V ring (warp 3); a K slot frees when the last
//                score MMA reading it completes, a V slot after the last PV
//   warp 1       MMA issuer (one thread): S_t = Q_t K_j^T into TMEM, then
//                O_t += P_t V_j with P_t read straight from TMEM
//   warp 2       TMEM allocator
//   warpgroup 1+t  softmax of query tile t: one thread per row (TMEM lane),
//                writes P_t (16-bit) over its own S_t columns, rescales O_t
//                in TMEM when the running max grows by more than 2^8, and
//                finally normalises O_t and writes O and LSE.
// With NQ = 2 the two softmax warpgroups run side by side: while one computes
// its softmax the tensor core works on the other tile's MMAs. Where TMEM has
// room (one query tile with 64-key tiles, as at D = 256), each query tile has
// two score buffers: S(j+1) is computed while the softmax turns S(j) into P(j),
// so the softmax of consecutive tiles is not serialised behind PV(j) and the
// next S (a single buffer, which P aliases, must wait for PV(j) to read P).
// Persistent: a CTA that finishes its block takes over the next
// not-yet-started CTA's block through cluster launch control (ItemQueue), so
// one CTA per SM walks a balanced stream of blocks in launch order. The K/V
// ring runs on across blocks, the next block's first scores are computed
// while the softmax warpgroups store the previous block, and Q is reloaded
// once the block's last score MMA has read it.
#pragma once

#include "fa_common.cuh"

namespace fa {

// Lazy-rescale threshold in the log2 domain: the running max used for the
// exponentials is only raised when the true max exceeds it by more than this,
// so unnormalised P stays below 2^8. The final O = o / l and LSE = m + log2 l
// use the same max, so the result is exact.
constexpr float kRescaleThreshold = 8.0f;

// One forward work item: a (batch, head) and a block of NQ * 128 query rows;
// its tiles are the key tiles the block sees.
struct FwdItem {
  int bh, b, g, q0, j_lo, n_iter;
};

__device__ __forceinline__ FwdItem fwd_item(int linear, const TileOrder& o, const AttnShape& s,
                                            int rows, int bn) {
  FwdItem t;
  int qblk;
  decode_tile(linear, o, &t.bh, &qblk);
  t.b = t.bh / s.Hq;
  t.g = (t.bh - t.b * s.Hq) / (s.Hq / s.Hkv);
  t.q0 = qblk * rows;
  int k_first, k_last;
  key_range(s, t.q0, min(s.Tq, t.q0 + rows), &k_first, &k_last);
  t.j_lo = k_first / bn;
  t.n_iter = max(0, (k_last + bn - 1) / bn - t.j_lo);
  return t;
}

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
  // Score buffers per query tile: two when they fit in TMEM next to the O
  // accumulators. With two, S(j+1) is computed while the softmax works on
  // S(j) (P(j) is written over S(j) and read by PV(j); S(j+2) reuses the
  // buffer after PV(j) in issue order), so the softmax never waits for the
  // tensor core to finish PV before its next scores exist.
  static constexpr int SBUF = NQ * (2 * BN + DP) <= 512 ? 2 : 1;
  // barriers: q_full, q_empty, k_full[S], v_full[S], k_empty[S], v_empty[S],
  // s_full[NQ][SBUF], p_full[NQ][SBUF], o_ready[NQ][2], drain, item responses
  // full / empty. p_full has one barrier per score buffer: with two buffers a
  // softmax warp can finish tile j+1 while a sibling still works on tile j,
  // and its arrival must not count towards tile j. o_ready has one barrier per
  // key-tile parity (PV(j) completes phase j / 2 of o_ready[j % 2]), so each
  // advances once every two tiles and a waiter is never two phases off.
  static constexpr int B_QFULL = 0, B_QEMPTY = 1, B_KFULL = 2, B_VFULL = B_KFULL + STAGES,
                       B_KEMPTY = B_VFULL + STAGES, B_VEMPTY = B_KEMPTY + STAGES,
                       B_SFULL = B_VEMPTY + STAGES, B_PFULL = B_SFULL + NQ * SBUF,
                       B_OREADY = B_PFULL + NQ * SBUF, B_DRAIN = B_OREADY + 2 * NQ,
                       B_CLCFULL = B_DRAIN + 1, B_CLCEMPTY = B_CLCFULL + kClcSlots,
                       NBAR = B_CLCEMPTY + kClcSlots;
  static constexpr int sfull(int t, int b) { return B_SFULL + t * SBUF + b; }
  static constexpr int pfull(int t, int b) { return B_PFULL + t * SBUF + b; }
  static constexpr int oready(int t, int j) { return B_OREADY + 2 * t + (j & 1); }
  static constexpr int OFF_CLC = (OFF_BAR + NBAR * 8 + 15) / 16 * 16;
  static constexpr int OFF_MISC = OFF_CLC + 16 * kClcSlots;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack
  static constexpr int THREADS = 128 + NQ * 128;
  static constexpr int ITEM_WARPS = 3 + 4 * NQ;  // warps that walk the items: 0, 1, 3, softmax
  // Registers per thread after the split (0: no split): the producer / MMA
  // warpgroup hands registers to the softmax warpgroups, whose 128-score rows
  // would otherwise spill. The launch must hold THREADS x launch registers >=
  // REG_NEEDED (checked on the host against the compiled kernel).
  // (One score buffer: 128 x 104 + 256 x 200 = 384 x 168, the launch total.)
  static constexpr int REG_CTRL = NQ == 2 ? (SBUF == 2 ? 112 : 104) : 0,
                       REG_SOFT = NQ == 2 ? (SBUF == 2 ? 168 : 200) : 0;
  static constexpr int REG_NEEDED = 128 * REG_CTRL + 128 * NQ * REG_SOFT;
  // TMEM: score buffers of tile t at t * SBUF * BN + b * BN, O_t after all of them
  static constexpr int S_COL(int t, int b) { return (t * SBUF + b) * BN; }
  static constexpr int O_COL(int t) { return NQ * SBUF * BN + t * DP; }
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(BN % 32 == 0 && BN <= 128, "key tile");
  static_assert(NQ * (SBUF * BN + DP) <= 512, "TMEM budget");
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
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const uint64_t tmo = wc.timeout_cycles;
  const ItemQueue iq{sbase + C::OFF_CLC, bar(C::B_CLCFULL), bar(C::B_CLCEMPTY)};
  constexpr int ROWS = C::NQ * kBM;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < C::NBAR; ++i) {
      uint32_t cnt = 1;
      if (i >= C::B_PFULL && i < C::B_PFULL + C::NQ * C::SBUF) cnt = 4;  // one per softmax warp
      if (i >= C::B_CLCEMPTY && i < C::B_CLCEMPTY + kClcSlots) cnt = C::ITEM_WARPS;
      mbar_init(bar(i), cnt);
    }
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  grid_wait_prior();  // the previous grid's outputs are complete and visible
  grid_release_next();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
  if constexpr (C::REG_CTRL > 0) regs_release<C::REG_CTRL>();
  if (warp == 0 || warp == 3) {
    // ----------------------------------------------------------- producers
    // warp 0: Q of each block (once its previous contents were last read),
    // then the block's K ring tiles, and the item requests; warp 3: the V
    // ring. The whole warp runs the loop (a lone active lane whose siblings
    // wait at the final barrier issues far slower); one elected lane issues.
    const bool leader = elect_one_sync();
    const bool k_ring = warp == 0;
    if (leader) tma_prefetch_desc(k_ring ? &map_k : &map_v);
    if (leader && k_ring) tma_prefetch_desc(&map_q);
    // K / V tiles are read by every query block of the group's heads: keep
    // them in L2; each Q block is read once
    const uint64_t pol_kv = l2_policy_evict_last(), pol_q = l2_policy_evict_first();
    const int full = k_ring ? C::B_KFULL : C::B_VFULL, empty = k_ring ? C::B_KEMPTY : C::B_VEMPTY;
    const uint32_t ring = sbase + (k_ring ? C::OFF_K : C::OFF_V);
    const CUtensorMap* map = k_ring ? &map_k : &map_v;
    int gk = 0, ln = 0, asked = 0;  // ring tiles issued, Q loads, requests
    bool ok = true;
    for (int k = 0, item = blockIdx.x; ok; ++k) {
      if (k_ring) {
        ok = clc_request(iq, k, leader, tmo, abort_flag, wc.status);
        if (!ok) break;
        ++asked;
      }
      const FwdItem t = fwd_item(item, order, s, ROWS, C::BN);
      if (t.n_iter > 0) {
        if (k_ring) {
          if (ln > 0) ok = mbar_wait(bar(C::B_QEMPTY), (ln - 1) & 1, tmo, abort_flag, wc.status);
          if (!ok) break;
          if (leader) mbar_arrive_expect_tx(bar(C::B_QFULL), C::NQ * C::Q_TILE);
          for (int tq = 0; tq < C::NQ; ++tq)
            for (int r = 0; r < C::KREG; ++r)
              if (leader)
                tma_load_3d_hint(sbase + C::OFF_Q + tq * C::Q_TILE + r * C::Q_REGION, &map_q,
                                 bar(C::B_QFULL), r * 64, t.q0 + tq * kBM, t.bh, pol_q);
          ++ln;
        }
        const int zkv = t.b * s.Hkv + t.g;
        for (int it = 0; it < t.n_iter; ++it, ++gk) {
          const int st = gk % C::STAGES;
          if (gk >= C::STAGES)
            ok = mbar_wait(bar(empty + st), ((gk / C::STAGES) - 1) & 1, tmo, abort_flag, wc.status);
          if (!ok) break;
          if (leader) mbar_arrive_expect_tx(bar(full + st), C::KV_TILE);
          for (int r = 0; r < C::KREG; ++r)
            if (leader)
              tma_load_3d_hint(ring + st * C::KV_TILE + r * C::KV_REGION, map, bar(full + st), r * 64,
                               (t.j_lo + it) * C::BN, zkv, pol_kv);
        }
        if (!ok) break;
      }
      if (!clc_next(iq, k, lane, &item, tmo, abort_flag, wc.status)) break;
    }
    if (*abort_flag) {
      drain_ring(bar(full), C::STAGES, gk, wc.drain_cycles, wc.status);
      if (k_ring) {
        drain_ring(bar(C::B_QFULL), 1, ln, wc.drain_cycles, wc.status);
        drain_ring(iq.full, kClcSlots, asked, wc.drain_cycles, wc.status);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer
    // the whole warp runs the loop; one elected lane issues
    const bool leader = elect_one_sync();
    constexpr uint32_t idesc_s = make_idesc_f16(kBM, C::BN, C::BF16 ? 1 : 0, 0, 0);
    constexpr uint32_t idesc_o = make_idesc_f16(kBM, C::D, C::BF16 ? 1 : 0, 0, 1);
    // S of query tile tq against the K tile in ring slot st, into score buffer b
    auto issue_s = [&](int tq, int st, int b) {
      const uint32_t qa = sbase + C::OFF_Q + tq * C::Q_TILE;
      const uint32_t ka = sbase + C::OFF_K + st * C::KV_TILE;
#pragma unroll
      for (int kk = 0; kk < C::D / 16; ++kk) {
        const uint32_t off = (kk & 3) * 32;  // 16 elements = 32 bytes along K
        const uint64_t ad = make_sdesc(qa + (kk >> 2) * C::Q_REGION + off, 16, 1024, 2);
        const uint64_t bd = make_sdesc(ka + (kk >> 2) * C::KV_REGION + off, 16, 1024, 2);
        if (leader) mma_ss(tmem + C::S_COL(tq, b), ad, bd, idesc_s, kk > 0);
      }
    };
    // O_tq += P V with P read from score buffer b
    auto issue_pv = [&](int tq, int st, int b, bool acc) {
      const uint32_t va = sbase + C::OFF_V + st * C::KV_TILE;
#pragma unroll
      for (int kk = 0; kk < C::BN / 16; ++kk) {
        const uint64_t bd = make_sdesc(va + kk * 16 * 128, C::KV_REGION, 1024, 2);
        if (leader)
          mma_ts(tmem + C::O_COL(tq), tmem + C::S_COL(tq, b) + kk * 8, bd, idesc_o,
                 (acc || kk > 0) ? 1u : 0u);
      }
    };
    // the issuer polls (test_wait), so it issues the moment a barrier completes
    auto wait = [&](int b, int parity) {
      return mbar_wait_poll(bar(b), parity & 1, tmo, abort_flag, wc.status);
    };
    int gk = 0, ln = 0;
    bool ok = true;
    for (int k = 0, item = blockIdx.x; ok; ++k) {
      const FwdItem t = fwd_item(item, order, s, ROWS, C::BN);
      const int n = t.n_iter;
      if (n > 0) {
        // scores of the block's first SBUF key tiles (over score buffers whose
        // PV MMAs of the previous block precede them in issue order)
        ok = wait(C::B_QFULL, ln);
        const int npro = n < C::SBUF ? n : C::SBUF;
        for (int p = 0; p < npro && ok; ++p) {
          const int gp = gk + p;
          ok = wait(C::B_KFULL + gp % C::STAGES, gp / C::STAGES);
          if (!ok) break;
          tc_fence_after();
          for (int tq = 0; tq < C::NQ; ++tq) {
            if (leader) issue_s(tq, gp % C::STAGES, gp % C::SBUF);
            if (leader) mma_commit(bar(C::sfull(tq, gp % C::SBUF)));
          }
          if (leader) mma_commit(bar(C::B_KEMPTY + gp % C::STAGES));  // K read for the last time
          if (p == n - 1 && leader) mma_commit(bar(C::B_QEMPTY));    // Q read for the last time
        }
        if (!ok) break;
        for (int it = 0; it < n; ++it) {
          const int gi = gk + it;
          const int st = gi % C::STAGES, b = gi % C::SBUF;
          const int gn = gi + C::SBUF, nst = gn % C::STAGES;  // the tile whose S reuses buffer b
          const bool next = it + C::SBUF < n;
          // V(gi) and K of the next score are checked before the P waits (they
          // land long before), so once P arrives only PV and S are issued
          ok = wait(C::B_VFULL + st, gi / C::STAGES) && (!next || wait(C::B_KFULL + nst, gn / C::STAGES));
          if (!ok) break;
          tc_fence_after();
          for (int tq = 0; tq < C::NQ; ++tq) {
            // P_t in TMEM; for the block's first tile this also means the
            // softmax warpgroup has stored the previous block's O_t
            ok = wait(C::pfull(tq, b), gi / C::SBUF);
            if (!ok) break;
            tc_fence_after();
            if (leader) issue_pv(tq, st, b, it > 0);
            if (leader) mma_commit(bar(C::oready(tq, gi)));
            if (next) {
              if (leader) issue_s(tq, nst, b);  // after PV(gi) read P from buffer b
              if (leader) mma_commit(bar(C::sfull(tq, b)));
            }
          }
          if (!ok) break;
          if (next && it + C::SBUF == n - 1 && leader) mma_commit(bar(C::B_QEMPTY));
          if (next && leader) mma_commit(bar(C::B_KEMPTY + nst));  // K(gn) read by its last S
          if (leader) mma_commit(bar(C::B_VEMPTY + st));          // V(gi) read by its last PV
        }
        if (!ok) break;
        gk += n;
        ++ln;
      }
      if (!clc_next(iq, k, lane, &item, tmo, abort_flag, wc.status)) break;
    }
    // make sure nothing is in flight before TMEM is released
    if (leader) mma_commit(bar(C::B_DRAIN));
    mbar_wait(bar(C::B_DRAIN), 0, wc.drain_cycles, nullptr, wc.status);
  }
  } else {
    if constexpr (C::REG_SOFT > 0) regs_claim<C::REG_SOFT>();
    // ------------------------------------------------------------- softmax
    const int tq = (warp - 4) >> 2;             // query tile of this warpgroup
    const int quarter = warp & 3;               // TMEM lane quarter of this warp
    const int r = quarter * 32 + lane;          // row within the tile
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t o_addr = tmem + lane_base + C::O_COL(tq);
    const float c = s.scale_log2;
    using T16 = typename std::conditional<C::BF16, __nv_bfloat16, __half>::type;
    int gk = 0;
    bool ok = true;
    for (int k = 0, item = blockIdx.x; ok; ++k) {
      const FwdItem t = fwd_item(item, order, s, ROWS, C::BN);
      const int tq_lo = t.q0 + tq * kBM;
      const int row = tq_lo + r;
      float m_used = -INFINITY;  // max used for the exponentials (log2 domain)
      float l = 0.f;
      for (int it = 0; it < t.n_iter; ++it) {
        const int gi = gk + it;
        const int k0 = (t.j_lo + it) * C::BN;
        const int b = gi % C::SBUF;  // score buffer of this tile
        const uint32_t s_addr = tmem + lane_base + C::S_COL(tq, b);
        ok = mbar_wait(bar(C::sfull(tq, b)), (gi / C::SBUF) & 1, tmo, abort_flag, wc.status);
        if (!ok) break;
        tc_fence_after();
        // one TMEM round trip for the whole row (a load issued while the tensor
        // core streams through TMEM takes long; a second pass would double it)
        uint32_t sv[C::BN];
#pragma unroll
        for (int cc = 0; cc < C::BN; cc += 32)
          tmem_ld32(s_addr + cc, *reinterpret_cast<uint32_t(*)[32]>(&sv[cc]));
        tmem_ld_wait();
        if (!block_unmasked(s, tq_lo, tq_lo + kBM, k0, k0 + C::BN)) {
          int lo, hi;
          visible_keys(s, row, k0, &lo, &hi);
#pragma unroll
          for (int kx = 0; kx < C::BN; ++kx)
            sv[kx] = (kx >= lo && kx < hi) ? sv[kx] : __float_as_uint(-INFINITY);
        }
        // row max over 8 independent chains (a single chain is 128 dependent
        // instructions long)
        float m8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) m8[e] = -INFINITY;
#pragma unroll
        for (int kx = 0; kx < C::BN; ++kx) m8[kx & 7] = fmaxf(m8[kx & 7], __uint_as_float(sv[kx]));
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
          for (int kx = 0; kx < 32; kx += 2) {
            const float2 x = f2_unpack(ffma2(
                f2_pack(__uint_as_float(sv[cc + kx]), __uint_as_float(sv[cc + kx + 1])), c2, nm2));
            const float p0 = ex2(x.x), p1 = ex2(x.y);
            acc[(kx / 2) & 3] = fadd2(acc[(kx / 2) & 3], f2_pack(p0, p1));
            pk[kx / 2] = pack2<C::BF16>(p0, p1);
          }
          // P overwrites the (already loaded) S columns: 2 values per column
          tmem_st16(s_addr + cc / 2, pk);
        }
        const float2 a01 = f2_unpack(fadd2(acc[0], acc[1])), a23 = f2_unpack(fadd2(acc[2], acc[3]));
        const float rs = (a01.x + a01.y) + (a23.x + a23.y);
        l = l * alpha + rs;
        if (it > 0 && __any_sync(0xffffffffu, grow)) {
          // O_t holds the sum of the previous tiles: wait for the last of them,
          // PV(gi-1). Its barrier's previous phase, PV(gi-3), has completed
          // (S(gi), just read, was issued after PV(gi-2)), and its next, PV(gi+1),
          // waits for this warp's P: at most one phase off.
          ok = mbar_wait(bar(C::oready(tq, gi - 1)), ((gi - 1) >> 1) & 1, tmo, abort_flag,
                         wc.status);
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int cc = 0; cc < C::D; cc += 32) {
            uint32_t ov[32];
            tmem_ld32(o_addr + cc, ov);
            tmem_ld_wait();
#pragma unroll
            for (int kx = 0; kx < 32; ++kx) ov[kx] = __float_as_uint(__uint_as_float(ov[kx]) * alpha);
            tmem_st32(o_addr + cc, ov);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::pfull(tq, b)));
      }
      if (!ok) break;

      // ------------------------------------------------------- block epilogue
      // O = o / l in blocks of 8S columns per warp (rows exchanged across lanes
      // for whole-segment stores), LSE = (m + log2 l) ln 2 per row. The next
      // block's first PV (which overwrites O_t) waits for this warpgroup's next
      // P, which comes after these reads.
      const bool have = t.n_iter > 0;
      if (have) {
        // O_t is final once the block's last PV completed (its commit also
        // covers every MMA issued before it). A parity wait is sound only while
        // the barrier is at most one phase off, which holds by construction:
        // PV(last) shares its barrier with PV(last-2), complete since S(last)
        // was issued after it, and PV(last+2), which needs this warp's next P.
        // (A single barrier for all PVs, waited for PV(last-1) and then
        // PV(last), could be two phases past the first wait when this warp ran
        // late, and that wait then never ended.)
        const int last = gk + t.n_iter - 1;
        ok = mbar_wait(bar(C::oready(tq, last)), (last >> 1) & 1, tmo, abort_flag, wc.status);
        if (!ok) break;
        tc_fence_after();
      }
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      constexpr int S = (C::D % 64 == 0) ? 8 : 4, W = 8 * S;
      const int row0 = tq_lo + quarter * 32;
      const int rows_valid = min(32, s.Tq - row0);
      T16* blk = reinterpret_cast<T16*>(o_out) +
                 (static_cast<int64_t>(t.bh) * s.Tq + (rows_valid > 0 ? row0 : 0)) * C::D;
#pragma unroll 1
      for (int cc = 0; cc < C::D; cc += W)
        store_acc_block<S, C::BF16>(o_addr + cc, have, inv_l, blk + cc, C::D, rows_valid);
      if (row < s.Tq)
        lse_out[static_cast<int64_t>(t.bh) * s.Tq + row] =
            l > 0.f ? (m_used + __log2f(l)) * kLn2 : -INFINITY;
      if (have) {
        tc_fence_before();
        gk += t.n_iter;
      }
      if (!clc_next(iq, k, lane, &item, tmo, abort_flag, wc.status)) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace fa
