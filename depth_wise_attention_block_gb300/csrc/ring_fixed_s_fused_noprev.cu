// agg_ring_kernel for bf16 rows of exactly 2 x 448 16-byte vectors
// (d = 7168), a source count fixed at compile time and the block
// bookkeeping fused, its fused source opening a partial sum (the fused source is F alone).  One instantiation per
// S = 1..9.
#include "ring_kernel.cuh"

namespace attnres {

cudaError_t launch_ring_fixed_s_fused_noprev(const RingParams& rp, int grid, int smem, cudaStream_t stream) {
  switch (rp.S) {
    case 1: return launch_ring_t<bf16_t, bf16_t, 2, true, true, 1, 1>(rp, grid, smem, stream);
    case 2: return launch_ring_t<bf16_t, bf16_t, 2, true, true, 2, 1>(rp, grid, smem, stream);
    case 3: return launch_ring_t<bf16_t, bf16_t, 2, true, true, 3, 1>(rp, grid, smem, stream);
    case 4: return launch_ring_t<bf16_t, bf16_t, 2, true, true, 4, 1>(rp, grid, smem, stream);
    case 5: return launch_ring_t<bf16_t, bf16_t, 2, true, true, 5, 1>(rp, grid, smem, stream);
    case 6: return launch_ring_t<bf16_t, bf16_t, 2, true, true, 6, 1>(rp, grid, smem, stream);
    case 7: return launch_ring_t<bf16_t, bf16_t, 2, true, true, 7, 1>(rp, grid, smem, stream);
    case 8: return launch_ring_t<bf16_t, bf16_t, 2, true, true, 8, 1>(rp, grid, smem, stream);
    case 9: return launch_ring_t<bf16_t, bf16_t, 2, true, true, 9, 1>(rp, grid, smem, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace attnres
