// Forward for short query blocks (at most 8 query rows per head): split over
// the keys, on CUDA cores, one cluster of CTAs per (batch, query head).
//
// What it computes is the forward of page "mlx-bun 0.0.4: package/src/model/
// flash-attention.ts" (forward shader): O = softmax(s Q K^T + mask) V with the
// running max / running sum recurrence and the natural-log LSE per row, the
// exp2 domain of page "[Metal] Add Flash Attention VJP for training"
// (Implementation Notes). The page "[Metal] Add Flash Attention VJP for
// training" also names a dedicated short-query (vector) path beside the tile
// kernels; this is that path, designed for GB300.
//
// Why a separate kernel: with Tq <= 8 a 128-row tensor-core tile is at least
// 94% padding, and the tile kernel walks all keys of a head in one CTA, so a
// decode-shaped call is a serial chain of key tiles on a handful of SMs. Here
// the keys of one (batch, head) are cut into `split` contiguous slices, one per
// CTA of a thread-block cluster (split <= 8, the portable cluster size):
//   - the slice is walked in stages of 128 keys: TMA copies the stage's K and
//     V rows into shared memory (128-byte swizzle); the next stage is loaded
//     once every warp is done with the current one;
//   - each warp takes 32 keys of a stage; a lane computes the scores of one
//     key against the (pre-scaled) query rows held in shared memory, the warp
//     keeps a running max / sum per row (online softmax, exp2 domain), and for
//     P V a lane owns pairs of output columns (the swizzle keeps both the
//     row-per-lane and the column-per-lane reads free of bank conflicts);
//   - the CTA merges its warps' (max, sum, output) per row and stores the
//     result straight into the shared memory of the row's owner, rank
//     (row mod split), through distributed shared memory;
//   - after one cluster barrier every owner merges its rows' partials from
//     its own shared memory and writes O and LSE.
// Waits: the stage loads complete on mbarriers with the library's bounded
// wait (a wait that gives up sets the status word and the CTA skips the rest
// of its keys); the cluster barriers (one at the start, split into arrive and
// wait, so that no CTA writes into a peer that has not started, and one after
// the partial rows are pushed) are reached by every thread of every CTA
// unconditionally.
// The merge is exact: each partial output is rescaled by 2^(m_part - m) to the
// common max m before the sums, and a row no key is visible to gets O = 0 and
// LSE = -inf.
#pragma once

#include "fa_common.cuh"

namespace fa {

constexpr int kDecodeWarps = 4;
constexpr int kDecodeThreads = 32 * kDecodeWarps;
constexpr int kDecodeMaxSplit = 8;    // CTAs per cluster (portable size)

template <int D_, int TQ_, bool BF16_>
struct DecodeFwdCfg {
  static constexpr int D = D_;
  static constexpr int TQ = TQ_;                  // query rows held (Tq rounded up to 1, 2, 4, 8)
  static constexpr bool BF16 = BF16_;
  static constexpr int NP = (D / 2 + 31) / 32;    // output column pairs per lane
  static constexpr int SK = 32 * kDecodeWarps;    // keys per stage
  static constexpr int DP = (D + 63) / 64 * 64;   // row padded to whole 128-byte column blocks
  static constexpr int KREG = DP / 64;
  static constexpr int REGION = SK * 128;         // bytes of one 64-column block of a stage
  static constexpr int TILE = KREG * REGION;      // K (or V) rows of one stage
  // one stage: at D <= 128 two CTAs then fit on an SM, which doubles the warps
  // that hide each other's latency and lets twice as many clusters run at once
  static constexpr int STAGES = 1;
  // shared memory: stages first (1024-byte aligned), then floats
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + STAGES * TILE;
  static constexpr int OFF_F = OFF_V + STAGES * TILE;
  static constexpr int F_Q = 0;                                // [TQ][D] q * scale * log2(e)
  static constexpr int F_P = F_Q + TQ * D;                     // [warps][TQ][32] p of a key block
  static constexpr int F_OW = F_P + kDecodeWarps * TQ * 32;    // [warps][TQ][D] warp partial o
  static constexpr int F_MW = F_OW + kDecodeWarps * TQ * D;    // [warps][TQ] warp max
  static constexpr int F_LW = F_MW + kDecodeWarps * TQ;        // [warps][TQ] warp sum
  // partial rows the cluster pushes to this CTA: slot (i / split) * split + rank
  // of row i's owner (rank i % split) holds rank's o[D], max, sum
  static constexpr int RSLOTS = TQ + kDecodeMaxSplit;
  static constexpr int F_WT = F_LW + kDecodeWarps * TQ;        // [warps][TQ] 2^(warp max - CTA max)
  static constexpr int F_R = F_WT + kDecodeWarps * TQ;         // [RSLOTS][D + 2]
  static constexpr int F_END = F_R + RSLOTS * (D + 2);
  static constexpr int SMEM_BYTES = OFF_F + F_END * 4 + 1024;  // + alignment slack
  static_assert(TQ >= 1 && TQ <= kDecodeMaxTq, "query rows");
  static_assert(D % 8 == 0, "16-byte chunks");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

// Byte offset of element d of row r in a stage tile (64-column blocks of
// 128-byte rows, 128-byte swizzle as TMA writes it).
__device__ __forceinline__ uint32_t stage_offset(int region_bytes, int r, int d) {
  return static_cast<uint32_t>((d >> 6) * region_bytes) +
         sw128_offset(static_cast<uint32_t>(r), static_cast<uint32_t>((d & 63) >> 3)) +
         static_cast<uint32_t>((d & 7) * 2);
}

// Store v to CTA `rank`'s shared memory, at the offset `p` has in this CTA's.
__device__ __forceinline__ void st_peer_f32(float* p, uint32_t rank, float v) {
  uint32_t remote, local = smem_u32(p);
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

// 2^(x - m) with 2^(-inf) = 0 and no NaN when both are -inf.
__device__ __forceinline__ float exp2_rel(float x, float m) {
  return x == -INFINITY ? 0.f : exp2f(x - m);
}

// Grid: B * Hq clusters of `split` CTAs along x (CTA = cluster * split + rank).
// Keys [k_first, k_last) are the ones any of the head's query rows can see;
// CTA `rank` takes [k_first + rank * keys_per_cta, ...) of them. map_k / map_v
// tile the [B * Hkv, Tkv, D] K and V with 64 x 128-row boxes.
template <class C>
__global__ void __launch_bounds__(kDecodeThreads, 1)
fa_fwd_decode_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                     const uint16_t* __restrict__ q, uint16_t* __restrict__ o,
                     float* __restrict__ lse, AttnShape s, int split, int k_first, int k_last,
                     int keys_per_cta, WaitCfg wc) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[C::STAGES];
  __shared__ int abort_flag;
  constexpr int D = C::D, TQ = C::TQ;
  // the swizzle pattern follows shared-memory address bits: align the stages to 1024 bytes
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  float* sm = reinterpret_cast<float*>(smem + C::OFF_F);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int bh = blockIdx.x / split;
  const int b = bh / s.Hq;
  const int g = (bh - b * s.Hq) / (s.Hq / s.Hkv);
  const int zkv = b * s.Hkv + g;
  const int Tq = s.Tq;
  const int64_t q_row0 = static_cast<int64_t>(bh) * Tq;
  const int kbeg = min(k_last, k_first + static_cast<int>(rank) * keys_per_cta);
  const int kend = min(k_last, kbeg + keys_per_cta);
  const int nstage = (kend - kbeg + C::SK - 1) / C::SK;
  const uint64_t tmo = wc.timeout_cycles;
  cluster_arrive_relaxed();  // waited for before the first store into a peer
  grid_wait_prior();  // the previous grid's outputs are complete and visible
  grid_release_next();

  // stage i: K and V rows [kbeg + i * SK, + SK) into slot i % STAGES
  auto issue = [&](int i) {
    const int slot = i % C::STAGES;
    const uint32_t bar = smem_u32(&full[slot]);
    mbar_arrive_expect_tx(bar, 2 * C::TILE);
    for (int r = 0; r < C::KREG; ++r) {
      tma_load_3d(sbase + C::OFF_K + slot * C::TILE + r * C::REGION, &map_k, bar, r * 64,
                  kbeg + i * C::SK, zkv);
      tma_load_3d(sbase + C::OFF_V + slot * C::TILE + r * C::REGION, &map_v, bar, r * 64,
                  kbeg + i * C::SK, zkv);
    }
  };
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < C::STAGES; ++i) mbar_init(smem_u32(&full[i]), 1);
    fence_mbar_init();
    for (int i = 0; i < C::STAGES && i < nstage; ++i) issue(i);
  }

  // query rows, scaled into the exp2 domain; rows past Tq are zero
  float* qs = sm + C::F_Q;
  for (int e = threadIdx.x; e < TQ * D; e += kDecodeThreads) {
    const int i = e / D;
    float x = 0.f;
    if (i < Tq) {
      const uint32_t w = q[(q_row0 + i) * D + (e - i * D)];
      x = unpack2<C::BF16>(w).x * s.scale_log2;
    }
    qs[e] = x;
  }
  __syncthreads();

  float m[TQ], l[TQ], acc[TQ][C::NP][2];
#pragma unroll
  for (int i = 0; i < TQ; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int u = 0; u < C::NP; ++u) acc[i][u][0] = acc[i][u][1] = 0.f;
  }
  float* ps = sm + C::F_P + warp * TQ * 32;

  int done = 0;  // stages consumed
#pragma unroll 1
  for (int st = 0; st < nstage; ++st) {
    const int slot = st % C::STAGES;
    bool ok = mbar_wait(smem_u32(&full[slot]), (st / C::STAGES) & 1, tmo, &abort_flag, wc.status);
    if (!__syncthreads_and(ok)) break;
    done = st + 1;
    const uint32_t ks = sbase + C::OFF_K + slot * C::TILE;
    const uint32_t vs = sbase + C::OFF_V + slot * C::TILE;
    const int blk = kbeg + st * C::SK + 32 * warp;  // this warp's 32 keys
    if (blk < kend) {
      const int rr = 32 * warp + lane;  // this lane's key row in the stage
      const bool in = blk + lane < kend;
      // scores of key blk + lane against every query row (lane = key)
      float sc[TQ];
#pragma unroll
      for (int i = 0; i < TQ; ++i) sc[i] = 0.f;
#pragma unroll 4
      for (int c8 = 0; c8 < D / 8; ++c8) {
        uint32_t w[4];
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                     : "r"(ks + stage_offset(C::REGION, rr, c8 * 8)));
        float kf[8];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float2 f = unpack2<C::BF16>(w[t]);
          kf[2 * t] = f.x;
          kf[2 * t + 1] = f.y;
        }
#pragma unroll
        for (int i = 0; i < TQ; ++i) {
          const float4 qa = *reinterpret_cast<const float4*>(qs + i * D + c8 * 8);
          const float4 qb = *reinterpret_cast<const float4*>(qs + i * D + c8 * 8 + 4);
          sc[i] = fmaf(qa.x, kf[0], sc[i]);
          sc[i] = fmaf(qa.y, kf[1], sc[i]);
          sc[i] = fmaf(qa.z, kf[2], sc[i]);
          sc[i] = fmaf(qa.w, kf[3], sc[i]);
          sc[i] = fmaf(qb.x, kf[4], sc[i]);
          sc[i] = fmaf(qb.y, kf[5], sc[i]);
          sc[i] = fmaf(qb.z, kf[6], sc[i]);
          sc[i] = fmaf(qb.w, kf[7], sc[i]);
        }
      }
      // mask, running max and sum, p of this block to shared memory
#pragma unroll
      for (int i = 0; i < TQ; ++i) {
        int lo, hi;
        visible_keys(s, i, blk, &lo, &hi);
        if (!in || i >= Tq || lane < lo || lane >= hi) sc[i] = -INFINITY;
        const float mn = fmaxf(m[i], warp_max(sc[i]));
        const float alpha = exp2_rel(m[i], mn);
        const float p = exp2_rel(sc[i], mn);
        l[i] = l[i] * alpha + p;
        m[i] = mn;
#pragma unroll
        for (int u = 0; u < C::NP; ++u) {
          acc[i][u][0] *= alpha;
          acc[i][u][1] *= alpha;
        }
        ps[i * 32 + lane] = p;
      }
      __syncwarp();
      // o += p V over the block's keys (lane = output column pairs)
      const int nj = min(32, kend - blk);
#pragma unroll 4
      for (int jj = 0; jj < nj; ++jj) {
        float pj[TQ];
#pragma unroll
        for (int i = 0; i < TQ; ++i) pj[i] = ps[i * 32 + jj];
#pragma unroll
        for (int u = 0; u < C::NP; ++u) {
          const int pidx = lane + 32 * u;
          if (pidx < D / 2) {
            uint32_t w;
            asm volatile("ld.shared.u32 %0, [%1];"
                         : "=r"(w)
                         : "r"(vs + stage_offset(C::REGION, 32 * warp + jj, 2 * pidx)));
            const float2 vf = unpack2<C::BF16>(w);
#pragma unroll
            for (int i = 0; i < TQ; ++i) {
              acc[i][u][0] = fmaf(pj[i], vf.x, acc[i][u][0]);
              acc[i][u][1] = fmaf(pj[i], vf.y, acc[i][u][1]);
            }
          }
        }
      }
      __syncwarp();
    }
    __syncthreads();  // every warp is done with this slot
    if (threadIdx.x == 0 && st + C::STAGES < nstage) issue(st + C::STAGES);
  }
  // after a wait gave up: let the loads still in flight land before the CTA exits
  if (threadIdx.x == 0)
    for (int i = done; i < nstage && i < done + C::STAGES; ++i)
      mbar_wait(smem_u32(&full[i % C::STAGES]), (i / C::STAGES) & 1, wc.drain_cycles, nullptr, wc.status);

  // warp partials to shared memory
  float* ow = sm + C::F_OW + warp * TQ * D;
#pragma unroll
  for (int i = 0; i < TQ; ++i) {
    const float lsum = warp_sum(l[i]);
    if (lane == 0) {
      sm[C::F_MW + warp * TQ + i] = m[i];
      sm[C::F_LW + warp * TQ + i] = lsum;
    }
#pragma unroll
    for (int u = 0; u < C::NP; ++u) {
      const int pidx = lane + 32 * u;
      if (pidx < D / 2) {
        ow[i * D + 2 * pidx] = acc[i][u][0];
        ow[i * D + 2 * pidx + 1] = acc[i][u][1];
      }
    }
  }
  __syncthreads();
  // CTA partial of each row (the warps' rows rescaled to their common max),
  // pushed into the shared memory of the row's owner
  float* recv = sm + C::F_R;
  if (threadIdx.x < Tq) {
    const int i = threadIdx.x;
    float mc = -INFINITY;
    for (int w = 0; w < kDecodeWarps; ++w) mc = fmaxf(mc, sm[C::F_MW + w * TQ + i]);
    float lc = 0.f;
    for (int w = 0; w < kDecodeWarps; ++w) {
      const float wt = exp2_rel(sm[C::F_MW + w * TQ + i], mc);
      sm[C::F_WT + w * TQ + i] = wt;
      lc += sm[C::F_LW + w * TQ + i] * wt;
    }
    sm[C::F_MW + i] = mc;  // warp 0's max is no longer needed
    sm[C::F_LW + i] = lc;
  }
  __syncthreads();
  cluster_wait();  // every CTA of the cluster is running
  for (int e = threadIdx.x; e < Tq * D; e += kDecodeThreads) {
    const int i = e / D;
    float x = 0.f;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w)
      x += sm[C::F_OW + w * TQ * D + e] * sm[C::F_WT + w * TQ + i];
    const int slot = (i / split) * split + static_cast<int>(rank);
    st_peer_f32(recv + slot * (D + 2) + (e - i * D), static_cast<uint32_t>(i % split), x);
  }
  if (threadIdx.x < Tq) {
    const int i = threadIdx.x;
    const int slot = (i / split) * split + static_cast<int>(rank);
    st_peer_f32(recv + slot * (D + 2) + D, static_cast<uint32_t>(i % split), sm[C::F_MW + i]);
    st_peer_f32(recv + slot * (D + 2) + D + 1, static_cast<uint32_t>(i % split), sm[C::F_LW + i]);
  }
  // every partial row has landed in its owner's shared memory; after this no
  // CTA touches another's, so no second barrier is needed before exiting
  cluster_barrier();

  // this CTA owns query rows rank, rank + split, ...: merge the cluster's partials
  using T16 = typename std::conditional<C::BF16, __nv_bfloat16, __half>::type;
  for (int i = static_cast<int>(rank); i < Tq; i += split) {
    const float* rows = recv + (i / split) * split * (D + 2);  // split slots of D + 2
    float mt = -INFINITY;
    for (int c = 0; c < split; ++c) mt = fmaxf(mt, rows[c * (D + 2) + D]);
    float lt = 0.f;
    for (int c = 0; c < split; ++c)
      lt += rows[c * (D + 2) + D + 1] * exp2_rel(rows[c * (D + 2) + D], mt);
    const float inv = lt > 0.f ? 1.f / lt : 0.f;
    T16* orow = reinterpret_cast<T16*>(o) + (q_row0 + i) * D;
    for (int d = threadIdx.x; d < D; d += kDecodeThreads) {
      float x = 0.f;
      for (int c = 0; c < split; ++c)
        x += rows[c * (D + 2) + d] * exp2_rel(rows[c * (D + 2) + D], mt);
      if constexpr (C::BF16)
        orow[d] = __float2bfloat16_rn(x * inv);
      else
        orow[d] = __float2half_rn(x * inv);
    }
    if (threadIdx.x == 0) lse[q_row0 + i] = lt > 0.f ? (mt + __log2f(lt)) * kLn2 : -INFINITY;
  }
}

// ---------------------------------------------------------------------------
// dQ for short query blocks (backward pass 3 of page "mlx-bun 0.0.4:
// package/src/model/flash-attention.ts": dQ_i = scale * sum_j dS_ij K_j with
// P_ij = exp(S_ij - L_i) from the cached LSE and dS_ij = P_ij (dP_ij - D_i),
// dP_ij = dO_i . V_j), split over the keys like the forward above: one cluster
// per (batch, query head), each CTA a slice of the keys staged by TMA, a lane
// per key for S and dP, a lane per output column pair for dS K. No running max
// is needed (LSE is known), so a CTA's partial dQ rows are plain sums; they
// are pushed into the row owner's shared memory and added there after one
// cluster barrier. Needs the D-vector of backward pass 1 (the workspace).
template <int D_, int TQ_, bool BF16_>
struct DecodeDqCfg {
  static constexpr int D = D_;
  static constexpr int TQ = TQ_;
  static constexpr bool BF16 = BF16_;
  static constexpr int NP = (D / 2 + 31) / 32;
  static constexpr int SK = 32 * kDecodeWarps;
  static constexpr int DP = (D + 63) / 64 * 64;
  static constexpr int KREG = DP / 64;
  static constexpr int REGION = SK * 128;
  static constexpr int TILE = KREG * REGION;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + TILE;
  static constexpr int OFF_F = OFF_V + TILE;
  static constexpr int F_Q = 0;                                // [TQ][D] q * scale * log2(e)
  static constexpr int F_DO = F_Q + TQ * D;                    // [TQ][D] dO
  static constexpr int F_NL = F_DO + TQ * D;                   // [TQ] -LSE * log2(e)
  static constexpr int F_DV = F_NL + TQ;                       // [TQ] D-vector
  static constexpr int F_P = F_DV + TQ;                        // [warps][TQ][32] dS of a key block
  static constexpr int F_OW = F_P + kDecodeWarps * TQ * 32;    // [warps][TQ][D] warp partial dQ
  static constexpr int RSLOTS = TQ + kDecodeMaxSplit;
  static constexpr int F_R = F_OW + kDecodeWarps * TQ * D;     // [RSLOTS][D] pushed partial rows
  static constexpr int F_END = F_R + RSLOTS * D;
  static constexpr int SMEM_BYTES = OFF_F + F_END * 4 + 1024;
  static_assert(TQ >= 1 && TQ <= kDecodeMaxTq, "query rows");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

template <class C>
__global__ void __launch_bounds__(kDecodeThreads, 1)
fa_bwd_dq_decode_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                        const uint16_t* __restrict__ q, const uint16_t* __restrict__ dout,
                        const float* __restrict__ lse, const float* __restrict__ dvec,
                        uint16_t* __restrict__ dq, float scale, AttnShape s, int split,
                        int k_first, int k_last, int keys_per_cta, WaitCfg wc, int overlap_prior) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full;
  __shared__ int abort_flag;
  constexpr int D = C::D, TQ = C::TQ;
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  float* sm = reinterpret_cast<float*>(smem + C::OFF_F);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int bh = blockIdx.x / split;
  const int b = bh / s.Hq;
  const int g = (bh - b * s.Hq) / (s.Hq / s.Hkv);
  const int zkv = b * s.Hkv + g;
  const int Tq = s.Tq;
  const int64_t q_row0 = static_cast<int64_t>(bh) * Tq;
  const int kbeg = min(k_last, k_first + static_cast<int>(rank) * keys_per_cta);
  const int kend = min(k_last, kbeg + keys_per_cta);
  const int nstage = (kend - kbeg + C::SK - 1) / C::SK;
  const uint64_t tmo = wc.timeout_cycles;
  cluster_arrive_relaxed();  // waited for before the first store into a peer
  // overlap_prior: the previous grid is the dK/dV launch of the same backward
  // (it and this grid touch disjoint outputs and share only inputs complete
  // before it passed its own wait): start at once, wait for it at exit
  if (!overlap_prior) grid_wait_prior();
  grid_release_next();

  auto issue = [&](int i) {
    const uint32_t bar = smem_u32(&full);
    mbar_arrive_expect_tx(bar, 2 * C::TILE);
    for (int r = 0; r < C::KREG; ++r) {
      tma_load_3d(sbase + C::OFF_K + r * C::REGION, &map_k, bar, r * 64, kbeg + i * C::SK, zkv);
      tma_load_3d(sbase + C::OFF_V + r * C::REGION, &map_v, bar, r * 64, kbeg + i * C::SK, zkv);
    }
  };
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&full), 1);
    fence_mbar_init();
    if (nstage > 0) issue(0);
  }
  // query and dO rows (rows past Tq are zero), their LSE (exp2 domain) and D
  for (int e = threadIdx.x; e < TQ * D; e += kDecodeThreads) {
    const int i = e / D;
    float xq = 0.f, xd = 0.f;
    if (i < Tq) {
      const int64_t at = (q_row0 + i) * D + (e - i * D);
      xq = unpack2<C::BF16>(static_cast<uint32_t>(q[at])).x * s.scale_log2;
      xd = unpack2<C::BF16>(static_cast<uint32_t>(dout[at])).x;
    }
    sm[C::F_Q + e] = xq;
    sm[C::F_DO + e] = xd;
  }
  if (threadIdx.x < TQ) {
    const int i = threadIdx.x;
    float nl = -INFINITY, dv = 0.f;  // no visible key (or past Tq): P = 0
    if (i < Tq) {
      const float L = lse[q_row0 + i];
      if (L != -INFINITY) nl = -L * kLog2e;
      dv = dvec[q_row0 + i];
    }
    sm[C::F_NL + i] = nl;
    sm[C::F_DV + i] = dv;
  }
  __syncthreads();

  float acc[TQ][C::NP][2];
#pragma unroll
  for (int i = 0; i < TQ; ++i)
#pragma unroll
    for (int u = 0; u < C::NP; ++u) acc[i][u][0] = acc[i][u][1] = 0.f;
  const float* qs = sm + C::F_Q;
  const float* dos = sm + C::F_DO;
  float* ps = sm + C::F_P + warp * TQ * 32;

  int done = 0;
#pragma unroll 1
  for (int st = 0; st < nstage; ++st) {
    const bool ok = mbar_wait(smem_u32(&full), st & 1, tmo, &abort_flag, wc.status);
    if (!__syncthreads_and(ok)) break;
    done = st + 1;
    const uint32_t ks = sbase + C::OFF_K, vs = sbase + C::OFF_V;
    const int blk = kbeg + st * C::SK + 32 * warp;
    if (blk < kend) {
      const int rr = 32 * warp + lane;
      const bool in = blk + lane < kend;
      // S and dP of key blk + lane against every query row (lane = key)
      float sc[TQ], dp[TQ];
#pragma unroll
      for (int i = 0; i < TQ; ++i) sc[i] = dp[i] = 0.f;
#pragma unroll 2
      for (int c8 = 0; c8 < D / 8; ++c8) {
        uint32_t wk[4], wv[4];
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(wk[0]), "=r"(wk[1]), "=r"(wk[2]), "=r"(wk[3])
                     : "r"(ks + stage_offset(C::REGION, rr, c8 * 8)));
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(wv[0]), "=r"(wv[1]), "=r"(wv[2]), "=r"(wv[3])
                     : "r"(vs + stage_offset(C::REGION, rr, c8 * 8)));
        float kf[8], vf[8];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float2 a = unpack2<C::BF16>(wk[t]), c = unpack2<C::BF16>(wv[t]);
          kf[2 * t] = a.x;
          kf[2 * t + 1] = a.y;
          vf[2 * t] = c.x;
          vf[2 * t + 1] = c.y;
        }
#pragma unroll
        for (int i = 0; i < TQ; ++i) {
          const float4 qa = *reinterpret_cast<const float4*>(qs + i * D + c8 * 8);
          const float4 qb = *reinterpret_cast<const float4*>(qs + i * D + c8 * 8 + 4);
          const float4 da = *reinterpret_cast<const float4*>(dos + i * D + c8 * 8);
          const float4 db = *reinterpret_cast<const float4*>(dos + i * D + c8 * 8 + 4);
          sc[i] = fmaf(qa.x, kf[0], sc[i]);
          sc[i] = fmaf(qa.y, kf[1], sc[i]);
          sc[i] = fmaf(qa.z, kf[2], sc[i]);
          sc[i] = fmaf(qa.w, kf[3], sc[i]);
          sc[i] = fmaf(qb.x, kf[4], sc[i]);
          sc[i] = fmaf(qb.y, kf[5], sc[i]);
          sc[i] = fmaf(qb.z, kf[6], sc[i]);
          sc[i] = fmaf(qb.w, kf[7], sc[i]);
          dp[i] = fmaf(da.x, vf[0], dp[i]);
          dp[i] = fmaf(da.y, vf[1], dp[i]);
          dp[i] = fmaf(da.z, vf[2], dp[i]);
          dp[i] = fmaf(da.w, vf[3], dp[i]);
          dp[i] = fmaf(db.x, vf[4], dp[i]);
          dp[i] = fmaf(db.y, vf[5], dp[i]);
          dp[i] = fmaf(db.z, vf[6], dp[i]);
          dp[i] = fmaf(db.w, vf[7], dp[i]);
        }
      }
      // dS = P (dP - D) with P = 2^(s c - LSE log2 e); hidden keys give 0
#pragma unroll
      for (int i = 0; i < TQ; ++i) {
        int lo, hi;
        visible_keys(s, i, blk, &lo, &hi);
        const bool vis = in && i < Tq && lane >= lo && lane < hi;
        const float nl = sm[C::F_NL + i];
        const float p = (vis && nl != -INFINITY) ? exp2f(sc[i] + nl) : 0.f;
        ps[i * 32 + lane] = p * (dp[i] - sm[C::F_DV + i]);
      }
      __syncwarp();
      // dQ += dS K over the block's keys (lane = output column pairs)
      const int nj = min(32, kend - blk);
#pragma unroll 4
      for (int jj = 0; jj < nj; ++jj) {
        float dsj[TQ];
#pragma unroll
        for (int i = 0; i < TQ; ++i) dsj[i] = ps[i * 32 + jj];
#pragma unroll
        for (int u = 0; u < C::NP; ++u) {
          const int pidx = lane + 32 * u;
          if (pidx < D / 2) {
            uint32_t w;
            asm volatile("ld.shared.u32 %0, [%1];"
                         : "=r"(w)
                         : "r"(ks + stage_offset(C::REGION, 32 * warp + jj, 2 * pidx)));
            const float2 kv = unpack2<C::BF16>(w);
#pragma unroll
            for (int i = 0; i < TQ; ++i) {
              acc[i][u][0] = fmaf(dsj[i], kv.x, acc[i][u][0]);
              acc[i][u][1] = fmaf(dsj[i], kv.y, acc[i][u][1]);
            }
          }
        }
      }
      __syncwarp();
    }
    __syncthreads();  // every warp is done with the stage
    if (threadIdx.x == 0 && st + 1 < nstage) issue(st + 1);
  }
  // after a wait gave up: let a load still in flight land before the CTA exits
  if (threadIdx.x == 0 && done < nstage) mbar_wait(smem_u32(&full), done & 1, wc.drain_cycles, nullptr, wc.status);

  // warp partials, their sum per CTA pushed into the row owner's shared memory
  float* ow = sm + C::F_OW + warp * TQ * D;
#pragma unroll
  for (int i = 0; i < TQ; ++i)
#pragma unroll
    for (int u = 0; u < C::NP; ++u) {
      const int pidx = lane + 32 * u;
      if (pidx < D / 2) {
        ow[i * D + 2 * pidx] = acc[i][u][0];
        ow[i * D + 2 * pidx + 1] = acc[i][u][1];
      }
    }
  __syncthreads();
  float* recv = sm + C::F_R;
  cluster_wait();  // every CTA of the cluster is running
  for (int e = threadIdx.x; e < Tq * D; e += kDecodeThreads) {
    const int i = e / D;
    float x = 0.f;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) x += sm[C::F_OW + w * TQ * D + e];
    const int slot = (i / split) * split + static_cast<int>(rank);
    st_peer_f32(recv + slot * D + (e - i * D), static_cast<uint32_t>(i % split), x);
  }
  cluster_barrier();  // every partial row has landed in its owner's shared memory

  using T16 = typename std::conditional<C::BF16, __nv_bfloat16, __half>::type;
  for (int i = static_cast<int>(rank); i < Tq; i += split) {
    const float* rows = recv + (i / split) * split * D;
    T16* out = reinterpret_cast<T16*>(dq) + (q_row0 + i) * D;
    for (int d = threadIdx.x; d < D; d += kDecodeThreads) {
      float x = 0.f;
      for (int c = 0; c < split; ++c) x += rows[c * D + d];
      if constexpr (C::BF16)
        out[d] = __float2bfloat16_rn(x * scale);
      else
        out[d] = __float2half_rn(x * scale);
    }
  }
  if (overlap_prior) grid_wait_prior();
}

}  // namespace fa

namespace fa {

// ---------------------------------------------------------------------------
// dK / dV for short query blocks: the vector VJP that page "[Metal] Add Flash
// Attention VJP for training" names for short sequences (Key Features: fp32
// dK/dV accumulation per key row, no padded tiles), computing backward pass 2
// of page "mlx-bun 0.0.4: package/src/model/flash-attention.ts":
//   dV_j = sum_i P_ij dO_i,   dK_j = scale * sum_i dS_ij Q_i,
//   P_ij = exp(S_ij - L_i),   dS_ij = P_ij (dO_i . V_j - D_i),
// the sums running over the query rows of every head that shares key j (GQA).
//
// GB300 design (not the pages'): with Tq <= 8 a KV group has at most 8 r query
// rows, so a 128-row tensor-core tile is mostly padding, and with a causal or
// window mask the heads' rows cannot be folded into one tile either (the mask
// depends on each row's position within its head). One CTA takes kVecKeys
// keys of one (batch, KV group) and walks the group's query rows in chunks of
// RC (8, 16 or 32), staged in shared memory as fp32 (Q pre-scaled by
// scale log2 e):
//   1. S and dP: a lane per key, RC / 8 rows per warp, dot
//      products over D read 16 bytes at a time (K / V rows padded to D + 4
//      floats, so the lanes' rows fall on distinct banks; the row vectors are
//      broadcast);
//   2. P = 2^(S - L log2 e), zero where the mask hides the key from the row's
//      position (or the row has no visible key), and dS = P (dP - D);
//   3. dV_j += P_ij dO_i and dK_j += dS_ij Q_i in fp32 registers, 8 threads
//      per key, each 4 consecutive columns per 32.
// dK is divided by log2 e at the end and both are written in the input dtype.
// Keys that no query position sees are written as zeros.
constexpr int kVecKeys = 32;     // keys per CTA
constexpr int kVecThreads = 256;

// RC: query rows per chunk (8, 16 or 32: the group's rows rounded up, at most 32)
template <int D_, bool BF16_, int RC_>
struct DkvVecCfg {
  static constexpr int D = D_;
  static constexpr bool BF16 = BF16_;
  static constexpr int RC = RC_;
  static constexpr int KS = D + 4;                  // fp32 stride of a K / V row
  static constexpr int PS = RC + 1;           // stride of a P / dS row (one per key)
  static constexpr int F_K = 0;                     // [kVecKeys][KS]
  static constexpr int F_V = F_K + kVecKeys * KS;   // [kVecKeys][KS]
  static constexpr int F_Q = F_V + kVecKeys * KS;   // [RC][D] Q * scale * log2 e
  static constexpr int F_DO = F_Q + RC * D;   // [RC][D]
  static constexpr int F_NL = F_DO + RC * D;  // [RC] -L log2 e (-inf: P = 0)
  static constexpr int F_DV = F_NL + RC;      // [RC] D-vector
  static constexpr int F_POS = F_DV + RC;     // [RC] position within the head (int)
  static constexpr int F_P = F_POS + RC;      // [kVecKeys][PS]
  static constexpr int F_DS = F_P + kVecKeys * PS;  // [kVecKeys][PS]
  static constexpr int F_END = F_DS + kVecKeys * PS;
  static constexpr int SMEM_BYTES = F_END * 4;
  static constexpr int NG = D / 32;                 // 4-column groups a thread accumulates
  static_assert(D % 32 == 0, "head dim");
  static_assert(kVecThreads == 8 * kVecKeys && RC % 8 == 0 && RC <= 32, "thread roles");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

template <class C>
__global__ void __launch_bounds__(kVecThreads)
fa_bwd_dkv_vec_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                      const uint16_t* __restrict__ v, const uint16_t* __restrict__ dout,
                      const float* __restrict__ lse, const float* __restrict__ dvec,
                      uint16_t* __restrict__ dk, uint16_t* __restrict__ dv, AttnShape s) {
  extern __shared__ __align__(16) float sm[];
  constexpr int D = C::D;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int nblk = (s.Tkv + kVecKeys - 1) / kVecKeys;
  const int zkv = blockIdx.x / nblk;  // b * Hkv + g
  const int j0 = (blockIdx.x - zkv * nblk) * kVecKeys;
  const int b = zkv / s.Hkv, g = zkv - b * s.Hkv;
  const int reps = s.Hq / s.Hkv;
  const int rows = reps * s.Tq;       // query rows of the group
  int* smi = reinterpret_cast<int*>(sm);
  // accumulation role: key jj, columns c4 .. c4 + 3 of every 32
  const int jj = t >> 3, c4 = (t & 7) * 4;
  float adk[C::NG][4], adv[C::NG][4];
#pragma unroll
  for (int m = 0; m < C::NG; ++m)
#pragma unroll
    for (int x = 0; x < 4; ++x) adk[m][x] = adv[m][x] = 0.f;
  grid_wait_prior();  // the previous grid's outputs are complete and visible
  grid_release_next();
  int kf, kl;
  key_range(s, 0, s.Tq, &kf, &kl);
  if (j0 < kl && j0 + kVecKeys > kf) {
    // Global loads are issued together (16 bytes each, into registers) and
    // converted afterwards, so staging costs one memory round trip, not one
    // per loop trip.
    constexpr int VPR = D / 8;  // 16-byte vectors per row
    constexpr int NKV = (kVecKeys * VPR + kVecThreads - 1) / kVecThreads;
    constexpr int NQR = (C::RC * VPR + kVecThreads - 1) / kVecThreads;
    auto row_of = [&](int gi) {  // global row of the group's query row gi
      const int hh = gi / s.Tq;
      return (static_cast<int64_t>(b) * s.Hq + g * reps + hh) * s.Tq + (gi - hh * s.Tq);
    };
    auto put8 = [&](float* dst, uint4 w, float mul) {  // dst 16-byte aligned
      const float2 a0 = unpack2<C::BF16>(w.x), a1 = unpack2<C::BF16>(w.y);
      const float2 a2 = unpack2<C::BF16>(w.z), a3 = unpack2<C::BF16>(w.w);
      reinterpret_cast<float4*>(dst)[0] = make_float4(a0.x * mul, a0.y * mul, a1.x * mul, a1.y * mul);
      reinterpret_cast<float4*>(dst)[1] = make_float4(a2.x * mul, a2.y * mul, a3.x * mul, a3.y * mul);
    };
    // K and V rows of the block (rows past Tkv are zero)
    {
      uint4 kw[NKV], vw[NKV];
#pragma unroll
      for (int n = 0; n < NKV; ++n) {
        const int e = t + n * kVecThreads, j = e / VPR;
        kw[n] = vw[n] = make_uint4(0u, 0u, 0u, 0u);
        if (e < kVecKeys * VPR && j0 + j < s.Tkv) {
          const int64_t at = (static_cast<int64_t>(zkv) * s.Tkv + j0 + j) * D + (e - j * VPR) * 8;
          kw[n] = *reinterpret_cast<const uint4*>(k + at);
          vw[n] = *reinterpret_cast<const uint4*>(v + at);
        }
      }
#pragma unroll
      for (int n = 0; n < NKV; ++n) {
        const int e = t + n * kVecThreads, j = e / VPR;
        if (e < kVecKeys * VPR) {
          put8(sm + C::F_K + j * C::KS + (e - j * VPR) * 8, kw[n], 1.f);
          put8(sm + C::F_V + j * C::KS + (e - j * VPR) * 8, vw[n], 1.f);
        }
      }
    }
    for (int i0 = 0; i0 < rows; i0 += C::RC) {
      uint4 qw[NQR], ow[NQR];
#pragma unroll
      for (int n = 0; n < NQR; ++n) {
        const int e = t + n * kVecThreads, i = e / VPR;
        qw[n] = ow[n] = make_uint4(0u, 0u, 0u, 0u);
        if (e < C::RC * VPR && i0 + i < rows) {
          const int64_t at = row_of(i0 + i) * D + (e - i * VPR) * 8;
          qw[n] = *reinterpret_cast<const uint4*>(q + at);
          ow[n] = *reinterpret_cast<const uint4*>(dout + at);
        }
      }
      float nl = -INFINITY, dd = 0.f;
      int pos = 0;
      if (t < C::RC && i0 + t < rows) {
        const int gi = i0 + t;
        pos = gi % s.Tq;
        const int64_t row = row_of(gi);
        const float L = lse[row];
        if (L != -INFINITY) nl = -L * kLog2e;
        dd = dvec[row];
      }
      __syncthreads();  // the previous chunk's rows, P and dS are consumed
#pragma unroll
      for (int n = 0; n < NQR; ++n) {
        const int e = t + n * kVecThreads, i = e / VPR;
        if (e < C::RC * VPR) {
          put8(sm + C::F_Q + i * D + (e - i * VPR) * 8, qw[n], s.scale_log2);
          put8(sm + C::F_DO + i * D + (e - i * VPR) * 8, ow[n], 1.f);
        }
      }
      if (t < C::RC) {
        sm[C::F_NL + t] = nl;
        sm[C::F_DV + t] = dd;
        smi[C::F_POS + t] = pos;
      }
      __syncthreads();
      {
        // S (log2 domain) and dP of key `lane` against rows warp + 8 x (x < RC / 8)
        const float* kr = sm + C::F_K + lane * C::KS;
        const float* vr = sm + C::F_V + lane * C::KS;
        constexpr int RW = C::RC / 8;  // rows per warp
        float sa[RW], pa[RW];
#pragma unroll
        for (int x = 0; x < RW; ++x) sa[x] = pa[x] = 0.f;
#pragma unroll 4
        for (int d = 0; d < D; d += 4) {
          const float4 k4 = *reinterpret_cast<const float4*>(kr + d);
          const float4 v4 = *reinterpret_cast<const float4*>(vr + d);
#pragma unroll
          for (int x = 0; x < RW; ++x) {
            const int i = warp + 8 * x;
            const float4 q4 = *reinterpret_cast<const float4*>(sm + C::F_Q + i * D + d);
            const float4 o4 = *reinterpret_cast<const float4*>(sm + C::F_DO + i * D + d);
            sa[x] = fmaf(q4.x, k4.x, fmaf(q4.y, k4.y, fmaf(q4.z, k4.z, fmaf(q4.w, k4.w, sa[x]))));
            pa[x] = fmaf(o4.x, v4.x, fmaf(o4.y, v4.y, fmaf(o4.z, v4.z, fmaf(o4.w, v4.w, pa[x]))));
          }
        }
        const int key = j0 + lane;
#pragma unroll
        for (int x = 0; x < RW; ++x) {
          const int i = warp + 8 * x;
          const float nl = sm[C::F_NL + i];
          const bool vis = key < s.Tkv && nl != -INFINITY &&
                           key_visible(smi[C::F_POS + i], key, s.causal, s.window);
          const float p = vis ? ex2(sa[x] + nl) : 0.f;
          sm[C::F_P + lane * C::PS + i] = p;
          sm[C::F_DS + lane * C::PS + i] = p * (pa[x] - sm[C::F_DV + i]);
        }
      }
      __syncthreads();
#pragma unroll 4
      for (int i = 0; i < C::RC; ++i) {
        const float p = sm[C::F_P + jj * C::PS + i], ds = sm[C::F_DS + jj * C::PS + i];
#pragma unroll
        for (int m = 0; m < C::NG; ++m) {
          const int d = 32 * m + c4;
          const float4 o4 = *reinterpret_cast<const float4*>(sm + C::F_DO + i * D + d);
          const float4 q4 = *reinterpret_cast<const float4*>(sm + C::F_Q + i * D + d);
          adv[m][0] = fmaf(p, o4.x, adv[m][0]);
          adv[m][1] = fmaf(p, o4.y, adv[m][1]);
          adv[m][2] = fmaf(p, o4.z, adv[m][2]);
          adv[m][3] = fmaf(p, o4.w, adv[m][3]);
          adk[m][0] = fmaf(ds, q4.x, adk[m][0]);
          adk[m][1] = fmaf(ds, q4.y, adk[m][1]);
          adk[m][2] = fmaf(ds, q4.z, adk[m][2]);
          adk[m][3] = fmaf(ds, q4.w, adk[m][3]);
        }
      }
    }
  }
  const int key = j0 + jj;
  if (key < s.Tkv) {
    const int64_t base = (static_cast<int64_t>(zkv) * s.Tkv + key) * D;
#pragma unroll
    for (int m = 0; m < C::NG; ++m) {
      const int d = 32 * m + c4;
      const uint2 wk = make_uint2(pack2<C::BF16>(adk[m][0] * kLn2, adk[m][1] * kLn2),
                                  pack2<C::BF16>(adk[m][2] * kLn2, adk[m][3] * kLn2));
      const uint2 wv = make_uint2(pack2<C::BF16>(adv[m][0], adv[m][1]),
                                  pack2<C::BF16>(adv[m][2], adv[m][3]));
      *reinterpret_cast<uint2*>(dk + base + d) = wk;
      *reinterpret_cast<uint2*>(dv + base + d) = wv;
    }
  }
}

}  // namespace fa
