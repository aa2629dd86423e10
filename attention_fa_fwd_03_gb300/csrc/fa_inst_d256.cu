// Kernels for head dim 256. Tile configuration (chosen for the 227 KB of shared
// memory and 512 TMEM columns of one SM):
//   forward: 1 query tile(s) of 128 rows per CTA, key tiles of 64, 2-stage K/V ring
//   dK/dV:   query tiles of 64 rows, 2-stage Q/dO ring, dV and dK in separate passes (TMEM)
//   dQ:      key tiles of 64, 1-stage K/V ring
#include "fa_inst.cuh"

FA_DEFINE_HEAD_DIM(256, 1, 64, 2, 64, 2, 1, 0, 64, 1)
