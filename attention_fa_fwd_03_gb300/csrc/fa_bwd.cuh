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
// A loop trip covers U rows per group, all their loads issued before any
// arithmetic (more bytes in flight per thread: 0.0535 -> 0.0516 ms on a
// B4 Hq32 T4096 D128 call). The loop bound is uniform over the block, so every
// lane of a warp reaches every shuffle (a row past the end loads zeros and
// stores nothing).
template <int D, bool BF16>
__global__ void __launch_bounds__(256)
fa_bwd_dvec_kernel(const uint4* __restrict__ o, const uint4* __restrict__ dout,
                   float* __restrict__ dvec, int64_t nrows) {
  constexpr int CHUNKS = D / 8;  // 16-byte chunks per row
  constexpr int TPR = CHUNKS <= 8 ? 8 : (CHUNKS <= 16 ? 16 : 32);
  constexpr int ROWS_PER_BLOCK = 256 / TPR;
  constexpr int U = 4;  // rows per thread group per loop trip
  grid_wait_prior();  // the previous grid's outputs are complete and visible
  grid_release_next();
  const int sub = threadIdx.x % TPR;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * ROWS_PER_BLOCK;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * ROWS_PER_BLOCK; base < nrows;
       base += U * stride) {
    constexpr int NCH = (CHUNKS + TPR - 1) / TPR;
    uint4 av[U][NCH], bv[U][NCH];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t row = base + u * stride + threadIdx.x / TPR;
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        const int ch = sub + c * TPR;
        av[u][c] = bv[u][c] = make_uint4(0u, 0u, 0u, 0u);
        if (row < nrows && ch < CHUNKS) {
          av[u][c] = __ldg(o + row * CHUNKS + ch);
          bv[u][c] = __ldg(dout + row * CHUNKS + ch);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t row = base + u * stride + threadIdx.x / TPR;
      float acc = 0.f;
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        const uint32_t aw[4] = {av[u][c].x, av[u][c].y, av[u][c].z, av[u][c].w};
        const uint32_t bw[4] = {bv[u][c].x, bv[u][c].y, bv[u][c].z, bv[u][c].w};
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
      if (sub == 0 && row < nrows) dvec[row] = acc;
    }
  }
}

}  // namespace fa
