// Instantiations of the tensor-core decode kernel for fp8 KV caches with pages of 8 rows
// (two pages per 16-row tile).
#include "decode_mma.cuh"

namespace pd {

cudaError_t launch_mma_pair_fp8(const DecodeParams& p, int q_dtype, dim3 grid, cudaStream_t st,
                                MmaConfig* cfg) {
  if (p.D != 128) return cudaErrorInvalidValue;
  if (q_dtype == kBF16) return launch_mma_r<F8, __nv_bfloat16, 128, false, true>(p, grid, st, cfg);
  if (q_dtype == kF16) return launch_mma_r<F8, __half, 128, false, true>(p, grid, st, cfg);
  return cudaErrorInvalidValue;
}

}  // namespace pd
