// merge_state_inplace and append_paged_kv kernels.
//
// merge_states: the same formula over R partners at once (the combine step of a
//   decode split across ranks); fp32 partial rows in, the output type out.
// merge: Apache TVM `_decode_kernels.py`, `merge_state_inplace` — one warp per
//   (n, h) row: both log-sum-exps are read, the row of V is rescaled and summed in
//   fp32, and S is written last (after the warp's reads).
// append: vllm-cpu `nki_flash_attn.py`, `reshape_and_cache`, on the TVM page layout
//   [max_pages, 2, H_kv, P, D]; FP8 encode per the NKI Attention Block TKG reference
//   (per-tensor k_scale / v_scale, OCP e4m3fn): IEEE fp32 division, then the hardware
//   round-to-nearest-even saturating conversion.  A negative slot skips the token.
//   With RoPE (append_paged_kv_rope) each K row is rotated at its token's position
//   before the conversion, the order of the NKI TKG block (RoPE, then the cache update).
#include "common.cuh"
#include "kernels.h"

namespace pd {

template <typename VT>
__global__ void merge_state_kernel(VT* __restrict__ V, float* __restrict__ S,
                                   const VT* __restrict__ Vo, const float* __restrict__ So,
                                   int rows, int D) {
  pdl_wait();
  pdl_release();
  const int warps = blockDim.x >> 5;
  const int row = blockIdx.x * warps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float s = S[row], so = So[row];
  const float smax = fmaxf(s, so);
  const float w = exp2f(s - smax), wo = exp2f(so - smax);
  const float a = w / (w + wo), ao = wo / (w + wo);
  VT* v = V + (size_t)row * D;
  const VT* vo = Vo + (size_t)row * D;
  for (int d = lane; d < D; d += 32) v[d] = from_f32<VT>(to_f32(v[d]) * a + to_f32(vo[d]) * ao);
  __syncwarp();
  if (lane == 0) S[row] = log2f(w + wo) + smax;
}

cudaError_t launch_merge_state(void* V, float* S, const void* V_other, const float* S_other, int N,
                               int H, int D, int v_dtype, cudaStream_t st) {
  const int rows = N * H;
  if (rows == 0) return cudaSuccess;
  const int threads = 256, per = threads / 32;
  const dim3 grid((rows + per - 1) / per);
  if (v_dtype == kF32)
    return launch_pdl(merge_state_kernel<float>, grid, dim3(threads), 0, st, (float*)V, S,
                      (const float*)V_other, S_other, rows, D);
  if (v_dtype == kBF16)
    return launch_pdl(merge_state_kernel<__nv_bfloat16>, grid, dim3(threads), 0, st,
                      (__nv_bfloat16*)V, S, (const __nv_bfloat16*)V_other, S_other, rows, D);
  if (v_dtype == kF16)
    return launch_pdl(merge_state_kernel<__half>, grid, dim3(threads), 0, st, (__half*)V, S,
                      (const __half*)V_other, S_other, rows, D);
  return cudaErrorInvalidValue;
}

// merge_states: the merge formula over R partners at once (one warp per (n, h) row): the
// R log-sum-exps are read by the lanes (r = lane, lane + 32, ...), M and the weight sum
// come from warp reductions, then each lane accumulates its dims over the R fp32
// partial rows and writes the output type.  All partners empty: out 0, lse -5e4.
template <typename OT, int DPL>
__global__ void merge_states_kernel(OT* __restrict__ out, float* __restrict__ S_out,
                                    const float* __restrict__ Vp, const float* __restrict__ Sp,
                                    int R, int rows, int D, long long rstride) {
  pdl_wait();
  pdl_release();
  const int warps = blockDim.x >> 5;
  const int row = blockIdx.x * warps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  // partner r: S at Sp + r * sstride, V rows at Vp + r * rstride (rstride = rows * D, or
  // one packed [out | lse] block per partner: rstride = sstride = rows * (D + 1))
  const long long sstride = rstride == (long long)rows * D ? rows : rstride;
  // lane r holds S_r of the first 32 partners (the common case: one load per lane)
  const float s_lane = lane < R ? Sp[lane * sstride + row] : kEmptyM;
  float M = s_lane;
  for (int r = lane + 32; r < R; r += 32) M = fmaxf(M, Sp[r * sstride + row]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  OT* o = out + (size_t)row * D;
  if (!(M > kEmptyM)) {
    for (int d = lane; d < D; d += 32) o[d] = from_f32<OT>(0.f);
    if (lane == 0) S_out[row] = kEmptyM;
    return;
  }
  // the partners' weights 2^(S_r - M), each computed once: lane r's for r < 32
  const float w_lane = lane < R ? exp2f(s_lane - M) : 0.f;
  float den = w_lane;
  for (int r = lane + 32; r < R; r += 32) den += exp2f(Sp[r * sstride + row] - M);
  den = warp_sum(den);
  const float inv = 1.f / den;
  // each lane owns DPL dims of a chunk of 32 DPL (d = d0 + lane + 32 e); the rows of four
  // partners are requested before any is accumulated, so the loads overlap instead of
  // queueing one L2 round trip behind another
  for (int d0 = 0; d0 < D; d0 += 32 * DPL) {
    float acc[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e) acc[e] = 0.f;
    const float* vrow = Vp + (long long)row * D + d0 + lane;
    for (int r0 = 0; r0 < R; r0 += 4) {
      float v[4][DPL];
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int e = 0; e < DPL; ++e)
          v[u][e] = r0 + u < R && d0 + lane + 32 * e < D ? vrow[(r0 + u) * rstride + 32 * e] : 0.f;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int r = r0 + u;
        float w = __shfl_sync(0xffffffffu, w_lane, r & 31);
        if (r >= 32) w = r < R ? exp2f(Sp[r * sstride + row] - M) : 0.f;
        if (r >= R) w = 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[e] = fmaf(w, v[u][e], acc[e]);
      }
    }
#pragma unroll
    for (int e = 0; e < DPL; ++e)
      if (d0 + lane + 32 * e < D) o[d0 + lane + 32 * e] = from_f32<OT>(acc[e] * inv);
  }
  if (lane == 0) S_out[row] = M + log2f(den);
}

template <typename OT>
static cudaError_t launch_merge_states_t(dim3 grid, dim3 block, cudaStream_t st, OT* out,
                                         float* S_out, const float* V_parts,
                                         const float* S_parts, int R, int rows, int D,
                                         long long rstride) {
  // dims per lane and chunk: D = 64 and 128 in one chunk, anything larger in chunks of 256
  if (D <= 64)
    return launch_pdl(merge_states_kernel<OT, 2>, grid, block, 0, st, out, S_out, V_parts,
                      S_parts, R, rows, D, rstride);
  if (D <= 128)
    return launch_pdl(merge_states_kernel<OT, 4>, grid, block, 0, st, out, S_out, V_parts,
                      S_parts, R, rows, D, rstride);
  return launch_pdl(merge_states_kernel<OT, 8>, grid, block, 0, st, out, S_out, V_parts,
                    S_parts, R, rows, D, rstride);
}

cudaError_t launch_merge_states(void* out, float* S_out, const float* V_parts, const float* S_parts,
                                int R, int N, int H, int D, int out_dtype, long long rstride,
                                cudaStream_t st) {
  const int rows = N * H;
  if (rows == 0) return cudaSuccess;
  const int threads = 256, per = threads / 32;
  const dim3 grid((rows + per - 1) / per);
  if (out_dtype == kF32)
    return launch_merge_states_t(grid, dim3(threads), st, (float*)out, S_out, V_parts, S_parts,
                                 R, rows, D, rstride);
  if (out_dtype == kBF16)
    return launch_merge_states_t(grid, dim3(threads), st, (__nv_bfloat16*)out, S_out, V_parts,
                                 S_parts, R, rows, D, rstride);
  if (out_dtype == kF16)
    return launch_merge_states_t(grid, dim3(threads), st, (__half*)out, S_out, V_parts, S_parts,
                                 R, rows, D, rstride);
  return cudaErrorInvalidValue;
}

template <typename IT, typename OT>
__device__ __forceinline__ OT convert_elem(IT x, float scale) {
  if constexpr (std::is_same<IT, OT>::value) {
    return x;
  } else if constexpr (std::is_same<OT, F8>::value) {
    F8 r;
    r.v = f32_to_e4m3(to_f32(x) / scale);  // IEEE division (no fast-math), then RNE satfinite
    return r;
  } else {
    return from_f32<OT>(to_f32(x));
  }
}

template <typename OT>
__device__ __forceinline__ OT convert_f32(float x, float scale) {
  if constexpr (std::is_same<OT, F8>::value) {
    F8 r;
    r.v = f32_to_e4m3(x / scale);
    return r;
  } else {
    return from_f32<OT>(x);
  }
}

// grid: (T * H_kv) blocks; block threads stride over D.  blockIdx.y: 0 = K, 1 = V.
// With rope.mode (1 rotate-half, 2 interleaved) each K row is rotated first, in fp32,
// at positions[t] (angle from the fixed-point turns F[i], to fp32 accuracy).
template <typename IT, typename OT>
__global__ void append_kernel(OT* __restrict__ pages, const IT* __restrict__ k_new,
                              const IT* __restrict__ v_new, const int64_t* __restrict__ slots,
                              int T, int H_kv, int D, int P, long long max_pages, float k_scale,
                              float v_scale, unsigned* err, const __grid_constant__ AppendRope rope) {
  pdl_wait();  // inputs and pages are the previous kernel's to write until it completes
  pdl_release();
  const int th = blockIdx.x;
  const int t = th / H_kv, h = th - t * H_kv;
  const int kv = blockIdx.y;
  const long long slot = slots[t];
  if (slot < 0) return;
  const long long page = slot / P, off = slot % P;
  if (page >= max_pages) {
    if (threadIdx.x == 0 && kv == 0 && h == 0) set_error(err, kErrBadSlot);
    return;
  }
  const IT* src = (kv == 0 ? k_new : v_new) + ((size_t)t * H_kv + h) * D;
  OT* dst = pages + ((((size_t)page * 2 + kv) * H_kv + h) * P + off) * D;
  const float scale = kv == 0 ? k_scale : v_scale;
  if (kv == 0 && rope.mode) {
    const int pos = rope.positions[t];
    for (int i = threadIdx.x; i < D / 2; i += blockDim.x) {
      const int a = rope.mode == 1 ? i : 2 * i, b = rope.mode == 1 ? i + D / 2 : 2 * i + 1;
      float c, sn;
      rope_cos_sin_accurate(pos, rope.F[i], c, sn);
      const float x = to_f32(src[a]), y = to_f32(src[b]);
      dst[a] = convert_f32<OT>(x * c - y * sn, scale);
      dst[b] = convert_f32<OT>(y * c + x * sn, scale);
    }
    return;
  }
  for (int d = threadIdx.x; d < D; d += blockDim.x) dst[d] = convert_elem<IT, OT>(src[d], scale);
}

template <typename IT>
static cudaError_t append_in(void* pages, const void* k, const void* v, const int64_t* slots, int T,
                             int H, int D, int P, long long max_pages, int kv_dtype, float ks,
                             float vs, unsigned* err, const AppendRope& rope, cudaStream_t st) {
  const dim3 grid((unsigned)T * H, 2);
  const int threads = D < 128 ? D : 128;
  const IT* kk = (const IT*)k;
  const IT* vv = (const IT*)v;
  const dim3 block(threads);
  switch (kv_dtype) {
    case kF32: return launch_pdl(append_kernel<IT, float>, grid, block, 0, st, (float*)pages, kk, vv, slots, T, H, D, P, max_pages, ks, vs, err, rope);
    case kF16: return launch_pdl(append_kernel<IT, __half>, grid, block, 0, st, (__half*)pages, kk, vv, slots, T, H, D, P, max_pages, ks, vs, err, rope);
    case kBF16: return launch_pdl(append_kernel<IT, __nv_bfloat16>, grid, block, 0, st, (__nv_bfloat16*)pages, kk, vv, slots, T, H, D, P, max_pages, ks, vs, err, rope);
    case kE4M3: return launch_pdl(append_kernel<IT, F8>, grid, block, 0, st, (F8*)pages, kk, vv, slots, T, H, D, P, max_pages, ks, vs, err, rope);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_append(void* pages, const void* k_new, const void* v_new,
                          const int64_t* slot_mapping, int T, int H_kv, int D, int P,
                          long long max_pages, int in_dtype, int kv_dtype, float k_scale,
                          float v_scale, unsigned* err, const AppendRope& rope, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  switch (in_dtype) {
    case kF32: return append_in<float>(pages, k_new, v_new, slot_mapping, T, H_kv, D, P, max_pages, kv_dtype, k_scale, v_scale, err, rope, st);
    case kF16: return append_in<__half>(pages, k_new, v_new, slot_mapping, T, H_kv, D, P, max_pages, kv_dtype, k_scale, v_scale, err, rope, st);
    case kBF16: return append_in<__nv_bfloat16>(pages, k_new, v_new, slot_mapping, T, H_kv, D, P, max_pages, kv_dtype, k_scale, v_scale, err, rope, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace pd
