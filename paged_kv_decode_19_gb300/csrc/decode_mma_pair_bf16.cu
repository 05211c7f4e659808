// Instantiations of the tensor-core decode kernel for bf16 KV caches with pages of 8 rows
// (two pages per 16-row tile).
#include "decode_mma.cuh"

namespace pd {

cudaError_t launch_mma_pair_bf16(const DecodeParams& p, int q_dtype, dim3 grid, cudaStream_t st,
                                MmaConfig* cfg) {
  (void)q_dtype;
  if (p.D == 64) return launch_mma_r<__nv_bfloat16, __nv_bfloat16, 64, false, true>(p, grid, st, cfg);
  if (p.D == 128) return launch_mma_r<__nv_bfloat16, __nv_bfloat16, 128, false, true>(p, grid, st, cfg);
  return cudaErrorInvalidValue;
}

}  // namespace pd
