// Host-side launch interface between the C ABI (fa_api.cu) and the per-head-
// dimension instantiation units (fa_inst_d*.cu). Internal to the library.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "fa_common.cuh"

namespace fa {

struct FwdLaunch {
  const void *q, *k, *v;
  void* o;
  float* lse;
  AttnShape s;
  bool bf16;
  WaitCfg wc;
  cudaStream_t stream;
};

struct BwdLaunch {
  const void *q, *k, *v, *o, *dout;
  const float* lse;
  void *dq, *dk, *dv;
  float* dvec;  // workspace: [B, Hq, Tq] fp32
  float scale;
  AttnShape s;       // shape the tile kernels run (grouped heads may be folded into rows)
  AttnShape s_rows;  // the call's own shape: Hq heads of Tq rows each
  bool bf16;
  WaitCfg wc;
  cudaStream_t stream;
};

// Encode a TMA map over a dense [z, y, x] = [BH, T, D] 16-bit tensor with a
// 128-byte-swizzled box of 64 x box_rows x 1 elements. Returns false when the
// driver rejects it.
bool encode_tile_map(CUtensorMap* map, const void* base, bool bf16, int D, int T, int BH,
                     int box_rows);

// Number of SMs of the current device (cached per device).
int device_sm_count();

cudaError_t launch_fwd_d64(const FwdLaunch& a);
cudaError_t launch_fwd_d96(const FwdLaunch& a);
cudaError_t launch_fwd_d128(const FwdLaunch& a);
cudaError_t launch_fwd_d256(const FwdLaunch& a);
// Backward phases, launched in this order when several bits are set.
enum : int { kPhaseDvec = 1, kPhaseDkv = 2, kPhaseDq = 4, kPhaseAll = 7 };
cudaError_t launch_bwd_d64(const BwdLaunch& a, int phases);
cudaError_t launch_bwd_d96(const BwdLaunch& a, int phases);
cudaError_t launch_bwd_d128(const BwdLaunch& a, int phases);
cudaError_t launch_bwd_d256(const BwdLaunch& a, int phases);

}  // namespace fa
