// Backward pass 1 for sm_103a: the D-vector preprocess of page "mlx-bun
// 0.0.4: package/src/model/flash-attention.ts", backward pass 1:
//   D_i = rowsum(dO_i o O_i) from the stored O                   (fa_bwd_dvec_kernel)
// Passes 2 (dK/dV) and 3 (dQ) are in fa_bwd_pipelined.cuh (head dims up to
// 128, and dQ at 256) and fa_bwd_d256.cuh (dK/dV at head dim 256).
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

}  // namespace fa
