// SIMT decode kernel: any element type (fp32 / f16 / bf16 / e4m3 KV), head dim
// 64/128/256, any page size, any GQA group.  Used for fp32 (where the 16-bit tensor
// path would lose the 1e-5 accuracy the fp32 path keeps) and for shapes the MMA
// kernel does not take.
//
// A block walks its share of (sequence, KV head, slice of <= 8 query heads) segments
// (see block_range); warps take groups of rows of a share; a lane holds D/32 elements of a row:
// D/64 from each half, so a RoPE pair (d, d + D/2) sits in one lane.  Per row: the
// q.k dot product is a warp sum, then the base-2 online softmax update of the TVM
// `batch_decode_paged_kv` kernel (m, d, O) and the PV accumulate; the warps' states
// are merged at the end (same formula as `merge_state_inplace`).
#include "decode_common.cuh"
#include "kernels.h"

namespace pd {

template <typename T, int N>
struct RowHalf {  // N consecutive elements of a row, loaded with one vector access
  static constexpr int kBytes = N * ElemBytes<T>::v;
  __device__ __forceinline__ static void load(const T* src, float (&dst)[N]) {
    if constexpr (kBytes == 16) {
      uint4 v = __ldg(reinterpret_cast<const uint4*>(src));
      unpack(reinterpret_cast<const uint8_t*>(&v), dst);
    } else if constexpr (kBytes == 8) {
      uint2 v = __ldg(reinterpret_cast<const uint2*>(src));
      unpack(reinterpret_cast<const uint8_t*>(&v), dst);
    } else if constexpr (kBytes == 4) {
      unsigned v = __ldg(reinterpret_cast<const unsigned*>(src));
      unpack(reinterpret_cast<const uint8_t*>(&v), dst);
    } else if constexpr (kBytes == 2) {
      unsigned short v = __ldg(reinterpret_cast<const unsigned short*>(src));
      unpack(reinterpret_cast<const uint8_t*>(&v), dst);
    } else {
      uint8_t v = *reinterpret_cast<const uint8_t*>(src);
      unpack(&v, dst);
    }
  }
  __device__ __forceinline__ static void unpack(const uint8_t* b, float (&dst)[N]) {
#pragma unroll
    for (int i = 0; i < N; ++i) dst[i] = to_f32(reinterpret_cast<const T*>(b)[i]);
  }
};

// A lane's Q or K values of one row: halves [d0, d0 + H2) and [d1, d1 + H2) (rotate-half
// pairs (d, d + D/2) share a lane slot e), or, for the interleaved RoPE layout, the
// element pairs (2i, 2i + 1) for i in [d0, d0 + H2), even elements in `a` and odd in
// `b`: the RoPE pair again shares slot e with frequency d0 + e.  Q and K take the same
// order, so q.k is unchanged; V and the output keep the halves.
template <typename T, int H2>
__device__ __forceinline__ void load_qk_row(const T* row, int d0, int d1, bool interleaved,
                                            float (&a)[H2], float (&b)[H2]) {
  if (!interleaved) {
    RowHalf<T, H2>::load(row + d0, a);
    RowHalf<T, H2>::load(row + d1, b);
    return;
  }
  float lo[H2], hi[H2];  // elements 2 d0 .. 2 d0 + 2 H2 - 1
  RowHalf<T, H2>::load(row + 2 * d0, lo);
  RowHalf<T, H2>::load(row + 2 * d0 + H2, hi);
#pragma unroll
  for (int e = 0; e < H2; ++e) {
    const float x = 2 * e < H2 ? lo[2 * e] : hi[2 * e - H2];
    const float y = 2 * e + 1 < H2 ? lo[2 * e + 1] : hi[2 * e + 1 - H2];
    a[e] = x;
    b[e] = y;
  }
}

template <typename KT, typename QT, int D, int NW>
__global__ void __launch_bounds__(NW * 32) decode_simt_kernel(const __grid_constant__ DecodeParams p) {
  constexpr int NT = NW * 32;
  constexpr int H2 = D / 64;  // elements per lane per half
  constexpr int E = 2 * H2;
  __shared__ float sm_m[NW * 8], sm_d[NW * 8];
  __shared__ float sm_o[NW * 8 * D];

  pdl_wait();  // nothing of the caller's is read before the previous kernel completes
  pdl_release();
  const BlockRange br = block_range<NT>(p);
  if (br.x0 >= br.x1) return;  // no units for this block
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int d0 = lane * H2, d1 = D / 2 + lane * H2;  // this lane's dims: [d0,d0+H2) and [d1,d1+H2)

  // rope frequencies of this lane
  unsigned long long F[H2];
#pragma unroll
  for (int e = 0; e < H2; ++e) F[e] = p.rope_F[d0 + e];

  // The block walks the segments (sequence, head slice) its unit range [x0, x1) touches;
  // a share of pieces [ua, pend) is the contiguous attended-row range [r0, r1).
  Segment sg = br.seg;
  for (;;) {
  const int ua = (int)max(br.x0 - sg.off, 0ll);
  const int ub = (int)min(br.x1 - sg.off, (long long)sg.n);
  const int hk = sg.hz / p.n_z, z = sg.hz - (sg.hz / p.n_z) * p.n_z;
  const int hq0 = hk * p.group + z * kMaxGroupPerCta;
  const int hcount = min(kMaxGroupPerCta, p.group - z * kMaxGroupPerCta);
  int r0 = 0, r1 = 0;
  if (sg.seq.L > 0) {
    const Pieces pcs = make_pieces(0, sg.seq.L, sg.seq, p.P);
    const int pend = min(ub, pcs.count());
    if (pend > ua) {
      const Piece first = get_piece(pcs, ua, p.P), last = get_piece(pcs, pend - 1, p.P);
      r0 = first.r_lo;
      r1 = last.r_lo + (last.s_hi - last.s_lo);
    }
  }
  const SeqInfo& wseq = sg.seq;

  // Q rows of this block's heads, roped, in log2 units
  float q[kMaxGroupPerCta][E];
  const int qpos = p.rotary ? p.q_rope_position[sg.b] : 0;
#pragma unroll
  for (int j = 0; j < kMaxGroupPerCta; ++j) {
    float a[H2], bb[H2];
    if (j < hcount) {
      const QT* qrow = reinterpret_cast<const QT*>(p.Q) + ((size_t)sg.b * p.H_qo + hq0 + j) * D;
      load_qk_row<QT, H2>(qrow, d0, d1, p.rotary == 2, a, bb);
    } else {
#pragma unroll
      for (int e = 0; e < H2; ++e) a[e] = bb[e] = 0.f;
    }
#pragma unroll
    for (int e = 0; e < H2; ++e) {
      float x = a[e], y = bb[e];
      if (p.rotary) {
        float c, s;
        if (std::is_same<KT, float>::value) rope_cos_sin_accurate(qpos, F[e], c, s);
        else rope_cos_sin(qpos, F[e], c, s);
        const float xr = x * c - y * s, yr = y * c + x * s;
        x = xr;
        y = yr;
      }
      q[j][e] = x * p.score_scale;
      q[j][H2 + e] = y * p.score_scale;
    }
  }

  float m[kMaxGroupPerCta], dsum[kMaxGroupPerCta], o[kMaxGroupPerCta][E];
#pragma unroll
  for (int j = 0; j < kMaxGroupPerCta; ++j) {
    m[j] = kEmptyM;
    dsum[j] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) o[j][e] = 0.f;
  }

  const int kpos0 = p.rotary && !p.k_rotated ? p.k_rope_pos_offset[sg.b] : 0;
  const KT* pages = reinterpret_cast<const KT*>(p.pages);
  const size_t kv_stride = (size_t)p.H_kv * p.P * D;  // K block -> V block of a page
  constexpr int R = 4;  // rows a warp loads before computing them (latency hiding)
  for (int rbase = r0 + warp * R; rbase < r1; rbase += NW * R) {
    float k[R][E], v[R][E];
    bool ok[R];
#pragma unroll
    for (int u = 0; u < R; ++u) {
      const int r = rbase + u;
      ok[u] = false;
#pragma unroll
      for (int e = 0; e < E; ++e) k[u][e] = v[u][e] = 0.f;  // rows outside the share stay 0
      if (r < r1) {
        const int so = r < wseq.sink ? r : r - wseq.sink + wseq.win_off;
        const int page = lookup_page(p, wseq, so / p.P);
        if (page >= 0) {
          ok[u] = true;
          const size_t kofs = (((size_t)page * 2 * p.H_kv + hk) * p.P + (so % p.P)) * D;
          float ka[H2], kb[H2], va[H2], vb[H2];
          load_qk_row<KT, H2>(pages + kofs, d0, d1, p.rotary == 2, ka, kb);
          RowHalf<KT, H2>::load(pages + kofs + kv_stride + d0, va);
          RowHalf<KT, H2>::load(pages + kofs + kv_stride + d1, vb);
#pragma unroll
          for (int e = 0; e < H2; ++e) {
            k[u][e] = ka[e];
            k[u][H2 + e] = kb[e];
            v[u][e] = va[e];
            v[u][H2 + e] = vb[e];
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < R; ++u) {
      if (ok[u] && p.rotary && !p.k_rotated) {  // (else the cache holds K rotated)
#pragma unroll
        for (int e = 0; e < H2; ++e) {
          float c, s;
          if (std::is_same<KT, float>::value) rope_cos_sin_accurate(kpos0 + rbase + u, F[e], c, s);
          else rope_cos_sin(kpos0 + rbase + u, F[e], c, s);
          const float x = k[u][e], y = k[u][H2 + e];
          k[u][e] = x * c - y * s;
          k[u][H2 + e] = y * c + x * s;
        }
      }
    }
    // the group's scores, then one max / rescale for the group (the group's weights
    // are independent of each other, so their exponentials overlap)
    float sc[kMaxGroupPerCta][R], mg[kMaxGroupPerCta];
#pragma unroll
    for (int j = 0; j < kMaxGroupPerCta; ++j) {
      mg[j] = m[j];
#pragma unroll
      for (int u = 0; u < R; ++u) {
        float s = 0.f;
        if (j < hcount) {
#pragma unroll
          for (int e = 0; e < E; ++e) s = fmaf(q[j][e], k[u][e], s);
          s = warp_sum(s);
        }
        sc[j][u] = s;
        if (ok[u]) mg[j] = fmaxf(mg[j], s);
      }
    }
    // weights: w[j][u] = 2^(s - mg) for the rows, w[j][R] = 2^(m - mg) rescales the state
    float w[kMaxGroupPerCta][R + 1];
    if constexpr (std::is_same<KT, float>::value) {
      // fp32 cache: the accurate exp2f (hardware ex2 is a few ulp short of fp32)
#pragma unroll
      for (int j = 0; j < kMaxGroupPerCta; ++j) {
#pragma unroll
        for (int u = 0; u < R; ++u) w[j][u] = ok[u] ? exp2f(sc[j][u] - mg[j]) : 0.f;
        w[j][R] = exp2f(m[j] - mg[j]);
      }
    } else {
#pragma unroll
      for (int j = 0; j < kMaxGroupPerCta; ++j) {
#pragma unroll
        for (int u = 0; u < R; ++u) w[j][u] = ok[u] ? fast_exp2(sc[j][u] - mg[j]) : 0.f;
        w[j][R] = fast_exp2(m[j] - mg[j]);
      }
    }
#pragma unroll
    for (int j = 0; j < kMaxGroupPerCta; ++j) {
      if (j < hcount) {
        const float a = w[j][R];
        float dsum_g = 0.f;
#pragma unroll
        for (int u = 0; u < R; ++u) dsum_g += w[j][u];
        dsum[j] = dsum[j] * a + dsum_g;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          float acc = o[j][e] * a;
#pragma unroll
          for (int u = 0; u < R; ++u) acc = fmaf(w[j][u], v[u][e], acc);
          o[j][e] = acc;
        }
        m[j] = mg[j];
      }
    }
  }

  // warp states -> shared memory
#pragma unroll
  for (int j = 0; j < kMaxGroupPerCta; ++j) {
    if (lane == 0) {
      sm_m[warp * 8 + j] = m[j];
      sm_d[warp * 8 + j] = dsum[j];
    }
#pragma unroll
    for (int e = 0; e < H2; ++e) {
      sm_o[(warp * 8 + j) * D + d0 + e] = o[j][e];
      sm_o[(warp * 8 + j) * D + d1 + e] = o[j][H2 + e];
    }
  }
  __syncthreads();
  finish_share<NT, NW>(p, br, sg, ua, ub, hq0, hcount, sm_m, sm_d, sm_o);
  if (sg.off + sg.n >= br.x1 || !next_segment(p, sg)) break;
  }  // segments
}

// ------------------------------------------------------------------------- dispatch
// Launch, or (ctas != nullptr) report how many blocks of the variant fit on one SM.
template <typename KT, typename QT, int D>
static cudaError_t launch_simt_d(const DecodeParams& p, dim3 grid, cudaStream_t st, int* ctas) {
  constexpr int NW = 4;
  auto kern = decode_simt_kernel<KT, QT, D, NW>;
  if (ctas) return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, kern, NW * 32, 0);
  return launch_pdl(kern, grid, dim3(NW * 32), 0, st, p);
}

template <typename KT, typename QT>
static cudaError_t launch_simt_t(const DecodeParams& p, dim3 grid, cudaStream_t st, int* ctas) {
  switch (p.D) {
    case 64: return launch_simt_d<KT, QT, 64>(p, grid, st, ctas);
    case 128: return launch_simt_d<KT, QT, 128>(p, grid, st, ctas);
    case 256: return launch_simt_d<KT, QT, 256>(p, grid, st, ctas);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode_simt(const DecodeParams& p, int q_dtype, int kv_dtype, dim3 grid,
                               cudaStream_t st, int* ctas) {
  if (kv_dtype == kF32 && q_dtype == kF32) return launch_simt_t<float, float>(p, grid, st, ctas);
  if (kv_dtype == kBF16 && q_dtype == kBF16) return launch_simt_t<__nv_bfloat16, __nv_bfloat16>(p, grid, st, ctas);
  if (kv_dtype == kF16 && q_dtype == kF16) return launch_simt_t<__half, __half>(p, grid, st, ctas);
  if (kv_dtype == kE4M3 && q_dtype == kBF16) return launch_simt_t<F8, __nv_bfloat16>(p, grid, st, ctas);
  if (kv_dtype == kE4M3 && q_dtype == kF16) return launch_simt_t<F8, __half>(p, grid, st, ctas);
  if (kv_dtype == kE4M3 && q_dtype == kF32) return launch_simt_t<F8, float>(p, grid, st, ctas);
  return cudaErrorInvalidValue;
}

bool simt_supports(int q_dtype, int kv_dtype, int D) {
  if (D != 64 && D != 128 && D != 256) return false;
  if (kv_dtype == q_dtype && kv_dtype != kE4M3) return true;
  return kv_dtype == kE4M3 && (q_dtype == kBF16 || q_dtype == kF16 || q_dtype == kF32);
}

}  // namespace pd
