// Kernels for head dim 64.
//   forward:  two 128-row query tiles per CTA, 128-key tiles, 3-stage K/V ring
//   backward: pipelined 128 x 128 dK/dV and dQ kernels (Q / K rings three
//             tiles deep, dO / V rings two deep)
#include "fa_inst.cuh"

FA_DEFINE_HEAD_DIM(64, 2, 128, 3)
