// Internal launch interface between the host API (api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "decode_common.cuh"

namespace pd {

// SIMT decode (any dtype / D in {64,128,256} / page size / group)
bool simt_supports(int q_dtype, int kv_dtype, int D);
// Launch, or (ctas != nullptr) only report resident blocks per SM.
cudaError_t launch_decode_simt(const DecodeParams& p, int q_dtype, int kv_dtype, dim3 grid,
                               cudaStream_t st, int* ctas = nullptr);

// Tensor-core decode (register-direct page loads + mma.sync); see decode_mma.cuh.
struct MmaConfig {
  int threads;       // block size
  int smem_bytes;    // dynamic shared memory
  int ctas_per_sm;   // occupancy (0 until queried)
};
// Launch (cfg == nullptr) or just query the launch configuration (cfg != nullptr).
cudaError_t launch_mma_bf16(const DecodeParams& p, int q_dtype, dim3 grid, cudaStream_t st,
                           MmaConfig* cfg);
cudaError_t launch_mma_f16(const DecodeParams& p, int q_dtype, dim3 grid, cudaStream_t st,
                           MmaConfig* cfg);
cudaError_t launch_mma_fp8(const DecodeParams& p, int q_dtype, dim3 grid, cudaStream_t st,
                           MmaConfig* cfg);
// The same for pages of 8 rows (single token): two pages per 16-row tile.
cudaError_t launch_mma_pair_bf16(const DecodeParams& p, int q_dtype, dim3 grid, cudaStream_t st,
                                 MmaConfig* cfg);
cudaError_t launch_mma_pair_f16(const DecodeParams& p, int q_dtype, dim3 grid, cudaStream_t st,
                                MmaConfig* cfg);
cudaError_t launch_mma_pair_fp8(const DecodeParams& p, int q_dtype, dim3 grid, cudaStream_t st,
                                MmaConfig* cfg);
// The same for the multi-query form (p.q_len > 1).
cudaError_t launch_mma_mq_bf16(const DecodeParams& p, int q_dtype, dim3 grid, cudaStream_t st,
                               MmaConfig* cfg);
cudaError_t launch_mma_mq_f16(const DecodeParams& p, int q_dtype, dim3 grid, cudaStream_t st,
                              MmaConfig* cfg);
cudaError_t launch_mma_mq_fp8(const DecodeParams& p, int q_dtype, dim3 grid, cudaStream_t st,
                              MmaConfig* cfg);

// Sets the thread's last-error message (api.cu).
void record_error(const char* msg);

// merge_state_inplace and append_paged_kv
cudaError_t launch_merge_state(void* V, float* S, const void* V_other, const float* S_other, int N,
                               int H, int D, int v_dtype, cudaStream_t st);
// R-way merge of fp32 partial states into out (out_dtype) and S_out; partner r's rows
// at V_parts + r * rstride (rstride = N*H*D: [R,N,H,D] with S [R,N,H]; or N*H*(D+1):
// one packed [out | lse] block per partner, S_parts = V_parts + N*H*D).
cudaError_t launch_merge_states(void* out, float* S_out, const float* V_parts, const float* S_parts,
                                int R, int N, int H, int D, int out_dtype, long long rstride,
                                cudaStream_t st);
// RoPE applied to the appended K rows (mode 0: none, 1 rotate-half, 2 interleaved).
struct AppendRope {
  const int32_t* positions;                // [T] position of each new token
  int mode;
  unsigned long long F[kMaxHalfDim];       // fixed-point turns per frequency
};
cudaError_t launch_append(void* pages, const void* k_new, const void* v_new,
                          const int64_t* slot_mapping, int T, int H_kv, int D, int P,
                          long long max_pages, int in_dtype, int kv_dtype, float k_scale,
                          float v_scale, unsigned* err, const AppendRope& rope, cudaStream_t st);

}  // namespace pd
