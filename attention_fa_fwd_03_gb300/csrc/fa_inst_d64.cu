// Kernels for head dim 64 (tile configurations sized for 227 KB of shared
// memory and 512 TMEM columns per SM):
//   forward: two 128-row query tiles per CTA, 128-key tiles, 3-stage K/V ring
//   dK/dV:   128 x 128 tiles, 4-stage Q/dO ring;  dQ: 128 x 128 tiles, 4-stage K/V ring
#include "fa_inst.cuh"

FA_DEFINE_HEAD_DIM(64, 2, 128, 3, 4, 4)
