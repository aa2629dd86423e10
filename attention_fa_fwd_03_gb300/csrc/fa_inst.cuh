// Launch helpers shared by the per-head-dimension instantiation units: build
// the TMA maps a kernel configuration needs and launch it on the caller's
// stream. Each fa_inst_d*.cu picks the tile configuration for its head dim.
#pragma once

#include "fa_bwd.cuh"
#include "fa_fwd.cuh"
#include "fa_launch.h"

namespace fa {

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
  const dim3 grid(bhq, (a.s.Tq + C::NQ * kBM - 1) / (C::NQ * kBM));
  kern<<<grid, C::THREADS, C::SMEM_BYTES, a.stream>>>(mq, mk, mv, a.o, a.lse, a.s, a.wc);
  return cudaGetLastError();
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
  fa_bwd_dvec_kernel<D, BF16><<<blocks, 256, 0, a.stream>>>(
      static_cast<const uint4*>(a.o), static_cast<const uint4*>(a.dout), a.dvec, nrows);
  return cudaGetLastError();
}

template <class C>
cudaError_t run_dkv(const BwdLaunch& a) {
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
  const dim3 grid(bhkv, (a.s.Tkv + kBM - 1) / kBM);
  kern<<<grid, C::THREADS, C::SMEM_BYTES, a.stream>>>(mq, mk, mv, mdo, a.lse, a.dvec, a.dk, a.dv,
                                                       a.scale, a.s, a.wc);
  return cudaGetLastError();
}

template <class C>
cudaError_t run_dq(const BwdLaunch& a) {
  const int bhq = a.s.B * a.s.Hq, bhkv = a.s.B * a.s.Hkv;
  CUtensorMap mq, mk, mv, mdo;
  if (!encode_tile_map(&mq, a.q, C::BF16, C::D, a.s.Tq, bhq, kBM) ||
      !encode_tile_map(&mdo, a.dout, C::BF16, C::D, a.s.Tq, bhq, kBM) ||
      !encode_tile_map(&mk, a.k, C::BF16, C::D, a.s.Tkv, bhkv, C::BN) ||
      !encode_tile_map(&mv, a.v, C::BF16, C::D, a.s.Tkv, bhkv, C::BN))
    return cudaErrorInvalidValue;
  auto kern = fa_bwd_dq_kernel<C>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const dim3 grid(bhq, (a.s.Tq + kBM - 1) / kBM);
  kern<<<grid, C::THREADS, C::SMEM_BYTES, a.stream>>>(mq, mk, mv, mdo, a.lse, a.dvec, a.dq,
                                                       a.scale, a.s, a.wc);
  return cudaGetLastError();
}

}  // namespace fa

// Define launch_fwd_d<D> / launch_bwd_d<D> for one head dim from its tile
// configurations: forward (NQ, BN, STAGES), dK/dV (query tile, STAGES, and
// whether dV and dK share one pass), dQ (BN, STAGES).
#define FA_DEFINE_HEAD_DIM(D, FNQ, FBN, FST, KBMQ, KST_DV, KST_DK, KJOINT, QBN, QST)        \
  namespace fa {                                                                            \
  template <bool BF16>                                                                      \
  static cudaError_t fwd_##D(const FwdLaunch& a) {                                          \
    return run_fwd<FwdCfg<D, FNQ, FBN, FST, BF16>>(a);                                      \
  }                                                                                         \
  template <bool BF16>                                                                      \
  static cudaError_t bwd_##D(const BwdLaunch& a, int phases) {                              \
    cudaError_t e = cudaSuccess;                                                            \
    if (phases & kPhaseDvec) e = run_dvec<D, BF16>(a);                                      \
    if (e != cudaSuccess) return e;                                                         \
    if (phases & kPhaseDkv) {                                                               \
      if constexpr (KJOINT) {                                                               \
        e = run_dkv<DkvCfg<D, KBMQ, KST_DV, BF16, kModeDV | kModeDK>>(a);                   \
      } else {                                                                              \
        e = run_dkv<DkvCfg<D, KBMQ, KST_DV, BF16, kModeDV>>(a);                             \
        if (e == cudaSuccess) e = run_dkv<DkvCfg<D, KBMQ, KST_DK, BF16, kModeDK>>(a);       \
      }                                                                                     \
    }                                                                                       \
    if (e != cudaSuccess) return e;                                                         \
    if (phases & kPhaseDq) e = run_dq<DqCfg<D, QBN, QST, BF16>>(a);                         \
    return e;                                                                               \
  }                                                                                         \
  cudaError_t launch_fwd_d##D(const FwdLaunch& a) {                                         \
    return a.bf16 ? fwd_##D<true>(a) : fwd_##D<false>(a);                                   \
  }                                                                                         \
  cudaError_t launch_bwd_d##D(const BwdLaunch& a, int phases) {                             \
    return a.bf16 ? bwd_##D<true>(a, phases) : bwd_##D<false>(a, phases);                   \
  }                                                                                         \
  }
