// Kernels for head dim 128:
//   forward: two 128-row query tiles per CTA, 128-key tiles, 2-stage K/V ring
//   dK/dV:   128 x 128 tiles, 2-stage Q/dO ring;  dQ: 128 x 128 tiles, 2-stage K/V ring
#include "fa_inst.cuh"

FA_DEFINE_HEAD_DIM(128, 2, 128, 2, 2, 2)
