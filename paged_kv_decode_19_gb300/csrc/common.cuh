// Device-side building blocks shared by the libpageddecode kernels (sm_103a).
//
// Everything here is inline PTX or CUDA intrinsics: mma.sync for the small dense
// contractions, packed fp32x2 arithmetic, FP8/bf16/f16 conversions, the RoPE angle,
// L2 prefetches and the device error word.  No kernel of this library waits on a
// flag or barrier that another block sets.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <climits>
#include <stdint.h>

#include <utility>

namespace pd {

// dtype codes (mirror pd_dtype in include/pageddecode.h)
enum : int { kF32 = 0, kF16 = 1, kBF16 = 2, kE4M3 = 3 };

// device error word bits
// (kErrTimeout is reserved: the current kernels have no wait that could time out)
enum : unsigned { kErrBadPage = 1u, kErrBadLength = 2u, kErrBadSlot = 4u, kErrTimeout = 8u };

// Initial running max of the online softmax (the TVM decode kernel's -5e4 sentinel);
// together with d = 0 it is the empty state and the merge identity.
constexpr float kEmptyM = -5e4f;

struct F8 { uint8_t v; };  // storage type of an e4m3 element

template <typename T> struct ElemBytes { static constexpr int v = sizeof(T); };
template <> struct ElemBytes<F8> { static constexpr int v = 1; };

// ----------------------------------------------------------------------------- conversions
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }

// two e4m3 codes (low byte = first) -> f16x2 (exact)
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}
__device__ __forceinline__ float to_f32(F8 x) {
  uint32_t h = e4m3x2_to_f16x2((uint16_t)x.v);
  return __half2float(__ushort_as_half((unsigned short)(h & 0xffff)));
}

// f32 -> one e4m3 code, round to nearest even, saturating to +-448.
__device__ __forceinline__ uint8_t f32_to_e4m3(float x) {
  uint16_t r;
  // first source -> upper byte, second source -> lower byte
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(x));
  return (uint8_t)(r & 0xff);
}

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}
template <> __device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }

// pack two f32 into a 16-bit-pair register (lo = first) of the MMA input type
template <typename T> __device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <> __device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
template <> __device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
template <typename T> __device__ __forceinline__ float2 unpack2(uint32_t v);
template <> __device__ __forceinline__ float2 unpack2<__nv_bfloat16>(uint32_t v) {
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}
template <> __device__ __forceinline__ float2 unpack2<__half>(uint32_t v) {
  __half2 h = *reinterpret_cast<__half2*>(&v);
  return __half22float2(h);
}

// Packed fp32x2 arithmetic (sm_100+): one instruction operates on a register pair.
__device__ __forceinline__ unsigned long long f2_pack(float2 v) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(v.x), "f"(v.y));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(unsigned long long r) {
  float2 v;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
  return v;
}
__device__ __forceinline__ float2 mul_f2(float2 a, float2 b) {
  unsigned long long r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2_pack(a)), "l"(f2_pack(b)));
  return f2_unpack(r);
}
__device__ __forceinline__ float2 sub_f2(float2 a, float2 b) {
  unsigned long long r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2_pack(a)), "l"(f2_pack(b)));
  return f2_unpack(r);
}
__device__ __forceinline__ float2 fma_f2(float2 a, float2 b, float2 c) {  // a * b + c
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(f2_pack(a)), "l"(f2_pack(b)), "l"(f2_pack(c)));
  return f2_unpack(r);
}

// Split x into hi + lo of the MMA input type (hi = RN(x), lo = RN(x - hi)); the pair
// carries ~2x the mantissa bits, so products of split operands are near-fp32 exact.
template <typename T>
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = pack2<T>(x0, x1);
  float2 h = unpack2<T>(hi);
  lo = pack2<T>(x0 - h.x, x1 - h.y);
}
// Same split of a pair, with the residual taken by one packed subtraction.
template <typename T>
__device__ __forceinline__ void split2(float2 x, uint32_t& hi, uint32_t& lo) {
  hi = pack2<T>(x.x, x.y);
  const float2 r = sub_f2(x, unpack2<T>(hi));
  lo = pack2<T>(r.x, r.y);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ----------------------------------------------------------------------------- RoPE angle
// Angle of frequency i at integer position pos, from the frequency's fixed-point
// "turns per position" F (2^64 * frac(rope_scale / rope_theta^(2i/D) / (2 pi))):
// pos * F mod 2^64 is the exact fraction of a revolution, so the angle is reduced
// to [-pi, pi) without any precision loss, whatever the position.
__device__ __forceinline__ void rope_cos_sin(int pos, unsigned long long F, float& c, float& s) {
  unsigned long long t = (unsigned long long)(long long)pos * F;
  int hi = (int)(unsigned)(t >> 32);
  float ang = (float)hi * 1.4629180792671596e-09f;  // 2*pi / 2^32
  __sincosf(ang, &s, &c);
}

// Same angle with fp32-level accuracy (for the fp32 path): the turn fraction is split
// into a 24-bit head and an 8-bit tail, sin/cos(pi*x) of the head come from the
// accurate sincospif, and the tail (< 2^-23 half-turns) is added to first order.
__device__ __forceinline__ void rope_cos_sin_accurate(int pos, unsigned long long F, float& c,
                                                      float& s) {
  const unsigned long long t = (unsigned long long)(long long)pos * F;
  const int hi = (int)(unsigned)(t >> 32);  // half-turns * 2^31, signed: x in [-1, 1)
  const float xa = (float)(hi & ~0xff) * 4.656612873077393e-10f;  // exact (<= 24 bits) * 2^-31
  const float xb = (float)(hi & 0xff) * 4.656612873077393e-10f;
  float sa, ca;
  sincospif(xa, &sa, &ca);
  const float d = xb * 3.14159265358979f;
  s = fmaf(ca, d, sa);
  c = fmaf(-sa, d, ca);
}

// Acquire-release fence at GPU scope: with a relaxed atomic after it (release) or
// before it (acquire) it orders a worker's partial results against the arrival
// counter, without the sequentially consistent fence of __threadfence().
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// ----------------------------------------------------------------------------- launch order
// Programmatic dependent launch: every kernel of the library is launched with
// programmatic stream serialisation, so it may start while the kernel before it on the
// stream is still finishing.  pdl_wait() returns once every grid it depends on has
// completed with its writes visible (at once when launched without the attribute);
// a kernel reads nothing that its predecessor may write, and writes nothing, before it.
// pdl_release() lets the next such kernel start; it is called only after pdl_wait(),
// so a kernel that starts early knows that everything before its predecessor is done.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_release() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... Params, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ----------------------------------------------------------------------------- error word
// Prefetch `bytes` (a multiple of 16) of global memory from a 16-byte aligned address
// into L2 (bulk async prefetch; no completion to wait for).
__device__ __forceinline__ void prefetch_l2_bulk(const void* ptr, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(ptr), "r"(bytes) : "memory");
}

// Block `part` of `parts` prefetches its share of [base, base + bytes) into L2 (the
// 16-byte aligned interior only: nothing outside the array is touched).
__device__ __forceinline__ void prefetch_l2_share(const void* base, size_t bytes, unsigned part,
                                                  unsigned parts) {
  const uintptr_t b0 = reinterpret_cast<uintptr_t>(base);
  const uintptr_t lo = (b0 + 15) & ~(uintptr_t)15, hi = (b0 + bytes) & ~(uintptr_t)15;
  if (hi <= lo || parts == 0) return;
  const uintptr_t chunk = (((hi - lo) + parts - 1) / parts + 15) & ~(uintptr_t)15;
  const uintptr_t s = lo + chunk * part;
  if (s >= hi) return;
  const uintptr_t e = s + chunk < hi ? s + chunk : hi;
  prefetch_l2_bulk(reinterpret_cast<const void*>(s), (uint32_t)(e - s));
}

__device__ __forceinline__ void set_error(unsigned* err, unsigned bits) {
  if (err) atomicOr(err, bits);
}

// ----------------------------------------------------------------------------- mma.sync
template <typename T> struct Mma;
template <> struct Mma<__nv_bfloat16> {
  static __device__ __forceinline__ void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7},"
        " {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
};
template <> struct Mma<__half> {
  static __device__ __forceinline__ void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7},"
        " {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
};

// warp-wide max / sum over lanes that share (lane & 3)  (xor 4, 8, 16)
__device__ __forceinline__ float max_over_groups(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
  return v;
}
__device__ __forceinline__ float sum_over_groups(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  v += __shfl_xor_sync(0xffffffffu, v, 8);
  v += __shfl_xor_sync(0xffffffffu, v, 16);
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace pd
