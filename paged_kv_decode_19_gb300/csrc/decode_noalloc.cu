// pd_batch_decode_paged_kv_noalloc: the decode entry point for callers that must not
// allocate device memory.  Its split scratch (arrival counters and partial out/lse)
// is a fixed array in the library's own device image instead of a cudaMalloc'd
// buffer; everything else is the regular decode path, run with that array passed
// as the caller workspace.
#include <mutex>

#include "kernels.h"
#include "pageddecode.h"

namespace pd {

constexpr size_t kStaticScratchBytes = (size_t)16 << 20;  // 16 MiB per device

// Every device that loads the library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxScratchDevices = 64;
static void* g_scratch_addr[kMaxScratchDevices];
static std::mutex g_scratch_mu;

// Device address of the array on the current device.  Host code may not use the
// array's name as a device pointer (it is a host-side stand-in), so the address is
// looked up once per device, with that device current.
static pd_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices) {
    record_error("pd_batch_decode_paged_kv_noalloc: no usable current CUDA device");
    return PD_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_scratch);
    if (e != cudaSuccess || !ptr) {
      record_error("pd_batch_decode_paged_kv_noalloc: cudaGetSymbolAddress of the static scratch failed");
      return PD_ERR_CUDA;
    }
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return PD_OK;
}

}  // namespace pd

extern "C" pd_status pd_batch_decode_paged_kv_noalloc(
    const void* Q, const void* pages, const int32_t* page_table_indptr,
    const int32_t* page_table_values, const int32_t* length_info,
    const int32_t* k_rope_pos_offset, const int32_t* q_rope_position, void* output, float* lse,
    int32_t rotary_mode, float rope_scale, float rope_theta, float sm_scale,
    const pd_decode_desc* desc, pd_stream_t stream) {
  if (!desc) {
    pd::record_error("desc is NULL");
    return PD_ERR_INVALID_ARG;
  }
  if (desc->workspace) {
    pd::record_error("pd_batch_decode_paged_kv_noalloc uses its own static scratch: desc->workspace must be NULL");
    return PD_ERR_INVALID_ARG;
  }
  void* scratch = nullptr;
  pd_status st = pd::scratch_address(&scratch);
  if (st != PD_OK) return st;
  const size_t need = pd_workspace_size(desc);
  if (need > pd::kStaticScratchBytes) {
    pd::record_error("pd_batch_decode_paged_kv_noalloc: this batch needs more split scratch than the "
                     "16 MiB static array holds; lower desc->num_splits or use pd_batch_decode_paged_kv");
    return PD_ERR_WORKSPACE;
  }
  pd_decode_desc d = *desc;
  d.workspace = scratch;
  d.workspace_bytes = pd::kStaticScratchBytes;
  return pd_batch_decode_paged_kv(Q, pages, page_table_indptr, page_table_values, length_info,
                                  k_rope_pos_offset, q_rope_position, output, lse, rotary_mode,
                                  rope_scale, rope_theta, sm_scale, &d, stream);
}
