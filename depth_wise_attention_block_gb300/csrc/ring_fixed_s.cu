// agg_ring_kernel for bf16 rows of exactly 2 x 448 16-byte vectors
// (d = 7168) and a source count fixed at compile time, without fused bookkeeping.  One
// instantiation per S = 1..9.
#include "ring_kernel.cuh"

namespace attnres {

cudaError_t launch_ring_fixed_s(const RingParams& rp, int grid, int smem, cudaStream_t stream) {
  switch (rp.S) {
    case 1: return launch_ring_t<bf16_t, bf16_t, 2, false, true, 1>(rp, grid, smem, stream);
    case 2: return launch_ring_t<bf16_t, bf16_t, 2, false, true, 2>(rp, grid, smem, stream);
    case 3: return launch_ring_t<bf16_t, bf16_t, 2, false, true, 3>(rp, grid, smem, stream);
    case 4: return launch_ring_t<bf16_t, bf16_t, 2, false, true, 4>(rp, grid, smem, stream);
    case 5: return launch_ring_t<bf16_t, bf16_t, 2, false, true, 5>(rp, grid, smem, stream);
    case 6: return launch_ring_t<bf16_t, bf16_t, 2, false, true, 6>(rp, grid, smem, stream);
    case 7: return launch_ring_t<bf16_t, bf16_t, 2, false, true, 7>(rp, grid, smem, stream);
    case 8: return launch_ring_t<bf16_t, bf16_t, 2, false, true, 8>(rp, grid, smem, stream);
    case 9: return launch_ring_t<bf16_t, bf16_t, 2, false, true, 9>(rp, grid, smem, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace attnres
