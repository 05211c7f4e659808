// Instantiations of the tensor-core decode kernel for f16 KV caches with pages of 8 rows
// (two pages per 16-row tile).
#include "decode_mma.cuh"

namespace pd {

cudaError_t launch_mma_pair_f16(const DecodeParams& p, int q_dtype, dim3 grid, cudaStream_t st,
                                MmaConfig* cfg) {
  (void)q_dtype;
  if (p.D == 64) return launch_mma_r<__half, __half, 64, false, true>(p, grid, st, cfg);
  if (p.D == 128) return launch_mma_r<__half, __half, 128, false, true>(p, grid, st, cfg);
  return cudaErrorInvalidValue;
}

}  // namespace pd
