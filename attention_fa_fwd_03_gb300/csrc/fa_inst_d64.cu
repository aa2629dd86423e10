// Kernels for head dim 64. Tile configuration (chosen for the 227 KB of shared
// memory and 512 TMEM columns of one SM):
//   forward: 2 query tile(s) of 128 rows per CTA, key tiles of 128, 3-stage K/V ring
//   dK/dV:   query tiles of 128 rows, 3-stage Q/dO ring, dV and dK in one pass
//   dQ:      key tiles of 128, 3-stage K/V ring
#include "fa_inst.cuh"

FA_DEFINE_HEAD_DIM(64, 2, 128, 3, 128, 3, 3, 1, 128, 3)
