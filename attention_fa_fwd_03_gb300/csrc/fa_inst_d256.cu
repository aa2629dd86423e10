// Kernels for head dim 256:
//   forward:  one 128-row query tile per CTA, 64-key tiles with two score
//             buffers in TMEM, 2-stage K/V ring
//   backward: dV and dK in two passes over 64-row query tiles, dQ over
//             64-key tiles (the fp32 accumulators alone fill TMEM at this width)
#include "fa_inst.cuh"

FA_DEFINE_HEAD_DIM(256, 1, 64, 2)
