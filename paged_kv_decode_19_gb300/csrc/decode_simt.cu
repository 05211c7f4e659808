// SIMT decode kernel: any element type (fp32 / f16 / bf16 / e4m3 KV), head dim
// 64/128/256, any page size, any GQA group.  Used for fp32 (where the 16-bit tensor
// path would lose the 1e-5 accuracy the fp32 path keeps) and for shapes the MMA
// kernel does not take (page size not a multiple of 16, D = 256).
//
// A block walks its share of (sequence, KV head, slice of <= 8 query heads) segments
// (see block_range); its warps take 32-row tiles of the share in turn.  Within a tile
// the lanes first own ROWS: lane i gathers row i's page, reads its K row in chunks,
// rotates it (RoPE) and computes the scores of all the slice's heads with Q read from
// shared memory (no cross-lane reduction per row).  The base-2 online softmax of the
// TVM `batch_decode_paged_kv` kernel (running max m, sum d, output O) then needs one
// warp maximum per head per tile; each lane keeps its own rows' share of d.  For P.V
// the lanes own DIMS: each lane accumulates its D/32 output dims over the tile's rows,
// with the probabilities and row addresses read back from shared memory as broadcasts.
// The warps' states are merged at the end (same formula as `merge_state_inplace`).
#include <type_traits>

#include "decode_common.cuh"
#include "kernels.h"

namespace pd {

// N consecutive elements of a row as floats, loaded with the widest vector accesses
// their byte count allows (the chunk starts at a multiple of its own size).
template <typename T, int N>
__device__ __forceinline__ void load_row_f32(const T* src, float (&dst)[N]) {
  constexpr int kBytes = N * ElemBytes<T>::v;
  if constexpr (kBytes < 4) {  // 1 or 2 bytes (E4M3 rows at D = 32, 64)
#pragma unroll
    for (int k = 0; k < N; ++k) dst[k] = to_f32(src[k]);
  } else if constexpr (kBytes % 16 == 0) {
#pragma unroll
    for (int i = 0; i < kBytes / 16; ++i) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(src) + i);
      const T* e = reinterpret_cast<const T*>(&v);
#pragma unroll
      for (int k = 0; k < 16 / (int)ElemBytes<T>::v; ++k) dst[i * (16 / ElemBytes<T>::v) + k] = to_f32(e[k]);
    }
  } else if constexpr (kBytes % 8 == 0) {
#pragma unroll
    for (int i = 0; i < kBytes / 8; ++i) {
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(src) + i);
      const T* e = reinterpret_cast<const T*>(&v);
#pragma unroll
      for (int k = 0; k < 8 / (int)ElemBytes<T>::v; ++k) dst[i * (8 / ElemBytes<T>::v) + k] = to_f32(e[k]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < kBytes / 4; ++i) {
      const unsigned v = __ldg(reinterpret_cast<const unsigned*>(src) + i);
      const T* e = reinterpret_cast<const T*>(&v);
#pragma unroll
      for (int k = 0; k < 4 / (int)ElemBytes<T>::v; ++k) dst[i * (4 / ElemBytes<T>::v) + k] = to_f32(e[k]);
    }
  }
}

template <typename KT>
__device__ __forceinline__ void rope_cs(int pos, unsigned long long F, float& c, float& s) {
  if constexpr (std::is_same<KT, float>::value) rope_cos_sin_accurate(pos, F, c, s);
  else rope_cos_sin(pos, F, c, s);
}

template <typename KT>
__device__ __forceinline__ float exp2_kv(float x) {
  if constexpr (std::is_same<KT, float>::value) return exp2f(x);  // fp32: the accurate exp2
  else return fast_exp2(x);
}

constexpr int kSimtChunk = 16;  // K dims (per half, with RoPE) a lane reads at a time

template <typename KT, typename QT, int D, int NW>
__global__ void __launch_bounds__(NW * 32, 2) decode_simt_kernel(const __grid_constant__ DecodeParams p) {
  constexpr int NT = NW * 32;
  constexpr int E = D / 32;  // output dims per lane in P.V
  constexpr int G8 = kMaxGroupPerCta;
  // The tile loop's Q rows and probabilities share their space with the warps' final
  // states (a block barrier separates the two uses).
  static_assert(G8 * D + NW * 32 * G8 <= NW * G8 * D, "shared layout");
  __shared__ __align__(16) float s_buf[NW * G8 * D];
  float (*s_q)[D] = reinterpret_cast<float (*)[D]>(s_buf);                 // [G8][D] Q rows (rotated, log2-scaled)
  float (*s_p)[32][G8] = reinterpret_cast<float (*)[32][G8]>(s_buf + G8 * D);  // [NW][32][G8] probabilities
  float* sm_o = s_buf;                                                       // [NW][G8][D] warp states
  __shared__ long long s_row[NW][32];                // element offset of each tile row's K row, -1: none
  __shared__ unsigned long long s_F[D / 2];          // RoPE turns per position, per frequency
  __shared__ float sm_m[NW * G8], sm_d[NW * G8];

  pdl_wait();  // nothing of the caller's is read before the previous kernel completes
  pdl_release();
  if (p.rotary)
    for (int i = threadIdx.x; i < D / 2; i += NT) s_F[i] = p.rope_F[i];
  const BlockRange br = block_range<NT>(p);
  if (br.x0 >= br.x1) return;  // no units for this block
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool il = p.rotary == 2;
  const bool krot = p.rotary && !p.k_rotated;
  const KT* pages = reinterpret_cast<const KT*>(p.pages);
  const size_t kv_stride = (size_t)p.H_kv * p.P * D;  // K block -> V block of a page

  // The block walks the segments (sequence, head slice) its unit range [x0, x1) touches;
  // its share of a segment, pieces [ua, pend), is the contiguous attended-row range [r0, r1).
  Segment sg = br.seg;
  for (;;) {
  const int ua = (int)max(br.x0 - sg.off, 0ll);
  const int ub = (int)min(br.x1 - sg.off, (long long)sg.n);
  const int hk = sg.hz / p.n_z, z = sg.hz - (sg.hz / p.n_z) * p.n_z;
  const int hq0 = hk * p.group + z * G8;
  const int hcount = min(G8, p.group - z * G8);
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
  const SeqInfo wseq = sg.seq;

  // Q rows of the slice -> shared memory, rotated at q_rope_position and scaled to log2
  // units; heads beyond the slice are zero.  Thread t takes (head, RoPE pair) items.
  {
    const int qpos = p.rotary ? __ldg(p.q_rope_position + sg.b) : 0;
    for (int it = tid; it < G8 * (D / 2); it += NT) {
      const int j = it / (D / 2), i = it - j * (D / 2);
      const int dx = il ? 2 * i : i, dy = il ? 2 * i + 1 : i + D / 2;  // the pair of frequency i
      float x = 0.f, y = 0.f;
      if (j < hcount) {
        const QT* qrow = reinterpret_cast<const QT*>(p.Q) + ((size_t)sg.b * p.H_qo + hq0 + j) * D;
        x = to_f32(qrow[dx]);
        y = to_f32(qrow[dy]);
        if (p.rotary) {
          float c, s;
          rope_cs<KT>(qpos, s_F[i], c, s);
          const float xr = x * c - y * s, yr = y * c + x * s;
          x = xr;
          y = yr;
        }
      }
      s_q[j][dx] = x * p.score_scale;
      s_q[j][dy] = y * p.score_scale;
    }
  }
  __syncthreads();

  const int kpos0 = krot ? __ldg(p.k_rope_pos_offset + sg.b) : 0;
  float m[G8], dl[G8], o[G8][E];
#pragma unroll
  for (int j = 0; j < G8; ++j) {
    m[j] = kEmptyM;
    dl[j] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) o[j][e] = 0.f;
  }

  // the tile loop for slices of at most HM heads (4 or 8: the scores' registers)
  auto tiles = [&](auto hm_tag) {
    constexpr int HM = decltype(hm_tag)::value;
    for (int rb = r0 + warp * 32; rb < r1; rb += NW * 32) {
      // ---- rows on lanes: gather, K . Q for every head
      const int r = rb + lane;
      long long off = -1;
      if (r < r1) {
        const int so = r < wseq.sink ? r : r - wseq.sink + wseq.win_off;
        const int page = lookup_page(p, wseq, so / p.P);
        if (page >= 0) off = ((((long long)page * 2 * p.H_kv + hk) * p.P) + (so % p.P)) * D;
      }
      s_row[warp][lane] = off;
      float sc[HM];
#pragma unroll
      for (int j = 0; j < HM; ++j) sc[j] = 0.f;
      if (off >= 0) {
        const KT* krow = pages + off;
        if (!krot) {
#pragma unroll 2
          for (int c = 0; c < D; c += kSimtChunk) {
            float k[kSimtChunk];
            load_row_f32<KT, kSimtChunk>(krow + c, k);
#pragma unroll
            for (int j = 0; j < HM; ++j) {
#pragma unroll
              for (int e = 0; e < kSimtChunk; e += 4) {
                const float4 q = *reinterpret_cast<const float4*>(&s_q[j][c + e]);
                sc[j] = fmaf(q.x, k[e], sc[j]);
                sc[j] = fmaf(q.y, k[e + 1], sc[j]);
                sc[j] = fmaf(q.z, k[e + 2], sc[j]);
                sc[j] = fmaf(q.w, k[e + 3], sc[j]);
              }
            }
          }
        } else {
          // RoPE pairs: frequency i rotates (i, i + D/2), or (2i, 2i + 1) interleaved
          const int pos = kpos0 + r;
#pragma unroll 1
          for (int c = 0; c < D / 2; c += kSimtChunk) {
            float kx[kSimtChunk], ky[kSimtChunk];
            if (!il) {
              load_row_f32<KT, kSimtChunk>(krow + c, kx);
              load_row_f32<KT, kSimtChunk>(krow + D / 2 + c, ky);
            } else {
              float a[2 * kSimtChunk];
              load_row_f32<KT, 2 * kSimtChunk>(krow + 2 * c, a);
#pragma unroll
              for (int e = 0; e < kSimtChunk; ++e) {
                kx[e] = a[2 * e];
                ky[e] = a[2 * e + 1];
              }
            }
#pragma unroll
            for (int e = 0; e < kSimtChunk; ++e) {
              float cs, sn;
              rope_cs<KT>(pos, s_F[c + e], cs, sn);
              const float x = kx[e], y = ky[e];
              kx[e] = x * cs - y * sn;
              ky[e] = y * cs + x * sn;
            }
#pragma unroll
            for (int j = 0; j < HM; ++j) {
#pragma unroll
              for (int e = 0; e < kSimtChunk; ++e) {
                const int dx = il ? 2 * (c + e) : c + e, dy = il ? dx + 1 : c + e + D / 2;
                sc[j] = fmaf(s_q[j][dx], kx[e], sc[j]);
                sc[j] = fmaf(s_q[j][dy], ky[e], sc[j]);
              }
            }
          }
        }
      }
      // ---- online softmax: one warp maximum per head per tile
#pragma unroll
      for (int j = 0; j < HM; ++j) {
        const float s = off >= 0 ? sc[j] : -INFINITY;
        float tm = s;
#pragma unroll
        for (int k = 16; k > 0; k >>= 1) tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, k));
        const float mn = fmaxf(m[j], tm);
        const float a = exp2_kv<KT>(m[j] - mn);  // 1 when the maximum did not move
        dl[j] *= a;
#pragma unroll
        for (int e = 0; e < E; ++e) o[j][e] *= a;
        m[j] = mn;
        const float pr = off >= 0 ? exp2_kv<KT>(s - mn) : 0.f;
        dl[j] += pr;
        s_p[warp][lane][j] = pr;
      }
      __syncwarp();
      // ---- dims on lanes: O[:, lane's dims] += p[:, row] v[row, lane's dims]
      const int nrow = min(32, r1 - rb);
#pragma unroll 4
      for (int i = 0; i < nrow; ++i) {
        const long long ro = s_row[warp][i];
        if (ro < 0) continue;  // bad page: the row is skipped (error recorded)
        float v[E];
        load_row_f32<KT, E>(pages + ro + kv_stride + lane * E, v);
        float pj[HM];
#pragma unroll
        for (int j = 0; j < HM; j += 4) {
          const float4 q4 = *reinterpret_cast<const float4*>(&s_p[warp][i][j]);
          pj[j] = q4.x;
          pj[j + 1] = q4.y;
          pj[j + 2] = q4.z;
          pj[j + 3] = q4.w;
        }
#pragma unroll
        for (int j = 0; j < HM; ++j)
#pragma unroll
          for (int e = 0; e < E; ++e) o[j][e] = fmaf(pj[j], v[e], o[j][e]);
      }
      __syncwarp();  // s_p / s_row are rewritten by the next tile
    }
  };
  if (hcount <= 4) tiles(std::integral_constant<int, 4>{});
  else tiles(std::integral_constant<int, 8>{});

  // warp states -> shared memory (unnormalised O, m, d = the lanes' shares summed), over
  // the Q rows and probabilities, once every warp is done with them
  __syncthreads();
#pragma unroll
  for (int j = 0; j < G8; ++j) {
    const float d = warp_sum(dl[j]);
    if (lane == 0) {
      sm_m[warp * G8 + j] = m[j];
      sm_d[warp * G8 + j] = d;
    }
#pragma unroll
    for (int e = 0; e < E; ++e) sm_o[(warp * G8 + j) * D + lane * E + e] = o[j][e];
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
