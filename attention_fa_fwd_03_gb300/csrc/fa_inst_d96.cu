// Kernels for head dim 96.
//   forward:  two 128-row query tiles per CTA, 128-key tiles, 2-stage K/V ring (rows padded to 128 elements in shared memory)
//   backward: pipelined 128 x 128 dK/dV and dQ kernels (Q / K rings three
//             tiles deep, dO / V rings two deep)
#include "fa_inst.cuh"

FA_DEFINE_HEAD_DIM(96, 2, 128, 2)
