// SIMT decode kernel: any element type (fp32 / f16 / bf16 / e4m3 KV), head dim
// 64/128/256, any page size, any GQA group.  Used for fp32 (where the 16-bit tensor
// path would lose the 1e-5 accuracy the fp32 path keeps) and for shapes the MMA
// kernel does not take (page sizes other than 8 and multiples of 16, D = 256).
//
// A block walks its share of (sequence, KV head, slice of <= 8 query heads) segments
// (see block_range); its warps take tiles of the share's rows in turn (4 KB of K rows
// per tile, 2 KB at D = 256: 32 rows of 128 bytes down to 2 rows of 1 KB).  Each warp has
// two shared-memory stages: while it computes a tile from one, the next tile's K and V
// rows are gathered through the page table into the other with cp.async (every row of
// the tile in flight at once), and the page-table entries of the tile after that are
// loaded.  The lanes then own ROWS (one to sixteen lanes per row): each reads its share
// of its K row, rotates it (RoPE) and computes the scores of all the slice's heads with
// Q read from shared memory (no reduction across the warp per row).  The base-2 online
// softmax of the TVM `batch_decode_paged_kv` kernel (running max m, sum d, output O)
// then needs one warp maximum per head per tile; each lane keeps its own rows' share of
// d.  For P.V the lanes own DIMS: each lane accumulates its D/32 output dims over the
// tile's rows, with the probabilities and row addresses read back from shared memory as
// broadcasts.
// The warps' states are merged at the end (same formula as `merge_state_inplace`).
#include <type_traits>

#include "decode_common.cuh"
#include "kernels.h"

namespace pd {

// N consecutive elements of a row in shared memory as floats (the chunk starts at a
// multiple of its own size, at most 16 bytes apart from it).
template <typename T, int N>
__device__ __forceinline__ void load_smem_f32(const T* src, float (&dst)[N]) {
  constexpr int kBytes = N * ElemBytes<T>::v;
  if constexpr (kBytes >= 16 && kBytes % 16 == 0) {
#pragma unroll
    for (int i = 0; i < kBytes / 16; ++i) {
      const uint4 v = reinterpret_cast<const uint4*>(src)[i];
      const T* e = reinterpret_cast<const T*>(&v);
#pragma unroll
      for (int k = 0; k < 16 / (int)ElemBytes<T>::v; ++k) dst[i * (16 / ElemBytes<T>::v) + k] = to_f32(e[k]);
    }
  } else if constexpr (kBytes == 8) {
    const uint2 v = *reinterpret_cast<const uint2*>(src);
    const T* e = reinterpret_cast<const T*>(&v);
#pragma unroll
    for (int k = 0; k < N; ++k) dst[k] = to_f32(e[k]);
  } else if constexpr (kBytes == 4) {
    const unsigned v = *reinterpret_cast<const unsigned*>(src);
    const T* e = reinterpret_cast<const T*>(&v);
#pragma unroll
    for (int k = 0; k < N; ++k) dst[k] = to_f32(e[k]);
  } else {
#pragma unroll
    for (int k = 0; k < N; ++k) dst[k] = to_f32(src[k]);
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

// cp.async: 16 bytes global -> shared, through L2 only.  A thread's copies since its
// last commit form a group; cp_async_wait<N> returns once all but its N most recent
// groups have landed.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Tile geometry of the SIMT kernel for rows of RB bytes: TR rows per warp tile (each
// row's K and V copied into one of the warp's two shared-memory stages), LPR = 32 / TR
// lanes per row in the K.Q phase; a stage is about 4 KB of K plus 4 KB of V (2 KB each
// at D = 256, where the per-warp Q rows take the room).
template <int RB, int D>
struct SimtTile {
  static constexpr int kKBytes = D >= 256 ? 2048 : 4096;
  static constexpr int TR = RB * 32 <= kKBytes ? 32 : kKBytes / RB;
  static constexpr int LPR = 32 / TR;
  static constexpr int KS = RB + 16;  // K row stride in shared memory (16 bytes apart per row:
                                      // the lanes' 16-byte reads of 8 rows cover all banks)
  static constexpr int kStage = TR * (KS + RB);
};

template <typename KT, int D, int NW>
struct SimtSmem {
  static constexpr int RB = D * ElemBytes<KT>::v;
  using Tl = SimtTile<RB, D>;
  static constexpr int G8 = kMaxGroupPerCta;
  // [Q rows G8 x D f32][probabilities NW x 32 x G8 f32][row offsets 2 x NW x 32 i64]
  // [stages 2 x NW] and, with RoPE on K, [per-warp Q rows NW x G8 x D f32][row rotations
  // TR x D/2 float2]; stage b of warp w is at kStage + (b NW + w) Tl::kStage
  static constexpr int kQ = 0;
  static constexpr int kP = kQ + G8 * D * 4;
  static constexpr int kRow = kP + NW * 32 * G8 * 4;
  static constexpr int kStage = kRow + 2 * NW * 32 * 8;
  static constexpr int kBytes = kStage + 2 * NW * Tl::kStage;
  static constexpr int kQW = kBytes;
  static constexpr int kRT = kQW + NW * G8 * D * 4;
  static constexpr int kBytesRope = kRT + Tl::TR * (D / 2) * 8;
  // the warps' final states [NW][G8][D] f32 reuse the space from the start
  static_assert(NW * G8 * D * 4 <= kBytes, "state overlay");
  // with the kernel's static shared memory (12 KB, start-up scan and merge scratch), within
  // the 227 KB a block may hold
  static_assert(kBytesRope + 16 * 1024 <= 227 * 1024, "shared memory");
};

template <typename KT, typename QT, int D, int NW>
__global__ void __launch_bounds__(NW * 32, 1) decode_simt_kernel(const __grid_constant__ DecodeParams p) {
  constexpr int NT = NW * 32;
  constexpr int E = D / 32;  // output dims per lane in P.V
  constexpr int G8 = kMaxGroupPerCta;
  using SM = SimtSmem<KT, D, NW>;
  using Tl = typename SM::Tl;
  constexpr int RB = SM::RB, TR = Tl::TR, LPR = Tl::LPR, KS = Tl::KS;
  constexpr int FP = (D / 2) / LPR;  // RoPE frequencies (pairs) per lane of a row
  constexpr int CH = FP < 8 ? FP : 8;
  extern __shared__ __align__(16) unsigned char s_dyn[];
  float (*s_q)[D] = reinterpret_cast<float (*)[D]>(s_dyn + SM::kQ);
  float (*s_p)[32][G8] = reinterpret_cast<float (*)[32][G8]>(s_dyn + SM::kP);
  long long (*s_row)[NW][32] = reinterpret_cast<long long (*)[NW][32]>(s_dyn + SM::kRow);
  // RoPE on K: a tile's rows sit at positions base + t (t = 0 .. TR-1); K row t is turned
  // by t positions (s_rt, the same for every tile) and each warp's Q rows by -base
  // (s_qw), since R(qpos) q . R(base + t) k = R(qpos - base) q . R(t) k
  float (*s_qw)[G8][D] = reinterpret_cast<float (*)[G8][D]>(s_dyn + SM::kQW);
  float2 (*s_rt)[D / 2] = reinterpret_cast<float2 (*)[D / 2]>(s_dyn + SM::kRT);
  float* sm_o = reinterpret_cast<float*>(s_dyn);  // [NW][G8][D] after the tiles
  __shared__ unsigned long long s_F[D / 2];       // RoPE turns per position, per frequency
  __shared__ float sm_m[NW * G8], sm_d[NW * G8];

  // Q and the page table are needed right after the start-up: each block prefetches its
  // share into L2 while it waits for the previous kernel (a prefetch reads nothing into
  // the program, and L2 sees that kernel's writes)
  if (threadIdx.x == 0) {
    prefetch_l2_share(p.Q, (size_t)p.B * p.H_qo * D * sizeof(QT), blockIdx.x, gridDim.x);
    if (p.values) prefetch_l2_share(p.values, (size_t)p.nnz_pages * sizeof(int32_t), blockIdx.x, gridDim.x);
  }
  pdl_wait();  // nothing of the caller's is read before the previous kernel completes
  pdl_release();
  if (p.rotary)
    for (int i = threadIdx.x; i < D / 2; i += NT) s_F[i] = p.rope_F[i];
  const BlockRange br = block_range<NT>(p);  // (its barriers also publish s_F)
  if (br.x0 >= br.x1) return;  // no units for this block
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (p.rotary && !p.k_rotated)  // published by the barrier after the first Q build
    for (int it = tid; it < TR * (D / 2); it += NT) {
      float c, sn;
      rope_cs<KT>(it / (D / 2), s_F[it % (D / 2)], c, sn);
      s_rt[it / (D / 2)][it % (D / 2)] = make_float2(c, sn);
    }
  const int trow = lane / LPR, part = lane % LPR;  // K.Q phase: this lane's row and part
  // this warp's two stages: K rows [TR][KS], then V rows [TR][RB]
  auto stage_k = [&](int buf) { return s_dyn + SM::kStage + (buf * NW + warp) * Tl::kStage; };
  auto stage_v = [&](int buf) { return stage_k(buf) + TR * KS; };
  const bool il = p.rotary == 2;
  const bool krot = p.rotary && !p.k_rotated;
  const unsigned char* pages = reinterpret_cast<const unsigned char*>(p.pages);
  const size_t kv_stride = (size_t)p.H_kv * p.P * RB;  // K block -> V block of a page (bytes)

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

  // A row's page-table entry is loaded first (row_entry) and used later (row_offset), so
  // that the load is in flight during other work; so < 0: no row.
  struct RowRef {
    int page, so;
  };
  auto row_entry = [&](int r) -> RowRef {
    RowRef e{-1, -1};
    if (r >= r1) return e;
    e.so = r < wseq.sink ? r : r - wseq.sink + wseq.win_off;
    const int pidx = e.so / p.P;
    if (pidx < 0 || pidx >= wseq.npages || (long long)wseq.page_begin + pidx >= p.nnz_pages)
      set_error(p.err, kErrBadPage);  // page stays -1
    else
      e.page = __ldg(p.values + wseq.page_begin + pidx);
    return e;
  };
  // byte offset in the pages of the row's K row (-1: no row / bad page, error recorded)
  auto row_offset = [&](const RowRef& e) -> long long {
    if (e.so < 0) return -1;
    if (e.page < 0 || (long long)e.page >= p.max_pages) {
      set_error(p.err, kErrBadPage);
      return -1;
    }
    return ((((long long)e.page * 2 * p.H_kv + hk) * p.P) + (e.so % p.P)) * RB;
  };
  // a tile's K and V rows -> stage `buf` of this warp (each row by its LPR lanes), as
  // one cp.async group of this thread
  auto issue_tile = [&](int buf, long long off) {
    if (part == 0) s_row[buf][warp][trow] = off;
    if (off >= 0) {
#pragma unroll
      for (int k = 0; k < RB / (16 * LPR); ++k) {
        const int c = (k * LPR + part) * 16;
        cp_async16(stage_k(buf) + trow * KS + c, pages + off + c);
        cp_async16(stage_v(buf) + trow * RB + c, pages + off + kv_stride + c);
      }
    }
    cp_async_commit();
  };

  // Q rows of the slice -> shared memory, rotated at q_rope_position and scaled to log2
  // units; heads beyond the slice are zero.  Thread t takes (head, RoPE pair) items.  The
  // raw Q elements and the page-table entries of this warp's first two tiles are loaded
  // together; the first tile's gather then streams in while Q is rotated and stored.
  const int rb_first = r0 + warp * TR;
  const RowRef e_first = row_entry(rb_first + trow);
  const RowRef e_second = row_entry(rb_first + NW * TR + trow);
  long long off_first;
  {
    constexpr int kQI = (G8 * (D / 2) + NT - 1) / NT;  // items per thread
    float qx[kQI], qy[kQI];
    const int qpos = p.rotary ? __ldg(p.q_rope_position + sg.b) : 0;
#pragma unroll
    for (int k = 0; k < kQI; ++k) {
      const int it = tid + k * NT;
      const int j = it / (D / 2), i = it - j * (D / 2);
      const int dx = il ? 2 * i : i, dy = il ? 2 * i + 1 : i + D / 2;  // the pair of frequency i
      qx[k] = qy[k] = 0.f;
      if (it < G8 * (D / 2) && j < hcount) {
        const QT* qrow = reinterpret_cast<const QT*>(p.Q) + ((size_t)sg.b * p.H_qo + hq0 + j) * D;
        qx[k] = to_f32(qrow[dx]);
        qy[k] = to_f32(qrow[dy]);
      }
    }
    off_first = row_offset(e_first);
    issue_tile(0, off_first);
#pragma unroll
    for (int k = 0; k < kQI; ++k) {
      const int it = tid + k * NT;
      if (it >= G8 * (D / 2)) break;
      const int j = it / (D / 2), i = it - j * (D / 2);
      const int dx = il ? 2 * i : i, dy = il ? 2 * i + 1 : i + D / 2;
      float x = qx[k], y = qy[k];
      if (p.rotary && j < hcount) {
        float c, sn;
        rope_cs<KT>(qpos, s_F[i], c, sn);
        const float xr = x * c - y * sn, yr = y * c + x * sn;
        x = xr;
        y = yr;
      }
      s_q[j][dx] = x * p.score_scale;
      s_q[j][dy] = y * p.score_scale;
    }
  }
  __syncthreads();

  const int kpos0 = krot ? __ldg(p.k_rope_pos_offset + sg.b) : 0;

  // the tile loop for slices of at most HM heads (4 or 8: the scores' registers)
  auto tiles = [&](auto hm_tag) {
    constexpr int HM = decltype(hm_tag)::value;
    float m[HM], dl[HM], o[HM][E];  // this warp's state of the slice's (first HM) heads
#pragma unroll
    for (int j = 0; j < HM; ++j) {
      m[j] = kEmptyM;
      dl[j] = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) o[j][e] = 0.f;
    }
    // Two stages per warp: tile i computes from stage i & 1 while tile i + 1 streams into
    // the other, and the page-table entries of tile i + 2 are loaded meanwhile.
    long long off = off_first;  // this lane's row of the current tile
    RowRef e_next = e_second;             // ... of the next tile
    int buf = 0;
    for (int rb = rb_first; rb < r1; rb += NW * TR, buf ^= 1) {
      if (krot) {  // this tile's Q rows, turned by -(position of its row 0)
        const int base = kpos0 + rb;
        for (int i = lane; i < D / 2; i += 32) {
          float c, sn;
          rope_cs<KT>(-base, s_F[i], c, sn);
          const int dx = il ? 2 * i : i, dy = il ? 2 * i + 1 : i + D / 2;
#pragma unroll
          for (int j = 0; j < HM; ++j) {
            const float x = s_q[j][dx], y = s_q[j][dy];
            s_qw[warp][j][dx] = x * c - y * sn;
            s_qw[warp][j][dy] = y * c + x * sn;
          }
        }
      }
      // the next tile's rows -> the other stage (read by the previous tile, whose last
      // __syncwarp has passed); an empty group past the last tile
      const long long off_next = row_offset(e_next);
      issue_tile(buf ^ 1, off_next);
      e_next = row_entry(rb + 2 * NW * TR + trow);
      cp_async_wait<1>();  // this tile's rows have landed
      __syncwarp();
      const unsigned char* st_k = stage_k(buf);
      const unsigned char* st_v = stage_v(buf);
      // ---- rows on lanes: K . Q over this lane's share of the row, summed over the row's lanes
      float sc[HM];
#pragma unroll
      for (int j = 0; j < HM; ++j) sc[j] = 0.f;
      if (off >= 0) {
        const KT* krow = reinterpret_cast<const KT*>(st_k + trow * KS);
        const float* qbase = krot ? &s_qw[warp][0][0] : &s_q[0][0];
#pragma unroll
        for (int c0 = 0; c0 < FP; c0 += CH) {
          const int f0 = part * FP + c0;  // first frequency of this chunk
          float kx[CH], ky[CH];
          if (!il) {
            load_smem_f32<KT, CH>(krow + f0, kx);
            load_smem_f32<KT, CH>(krow + D / 2 + f0, ky);
          } else {
            float a[2 * CH];
            load_smem_f32<KT, 2 * CH>(krow + 2 * f0, a);
#pragma unroll
            for (int e = 0; e < CH; ++e) {
              kx[e] = a[2 * e];
              ky[e] = a[2 * e + 1];
            }
          }
          if (krot) {
#pragma unroll
            for (int e = 0; e < CH; ++e) {
              const float2 cs = s_rt[trow][f0 + e];
              const float x = kx[e], y = ky[e];
              kx[e] = x * cs.x - y * cs.y;
              ky[e] = y * cs.x + x * cs.y;
            }
          }
#pragma unroll
          for (int j = 0; j < HM; ++j) {
            float qx[CH], qy[CH];  // Q of the chunk's pairs, read as 16-byte vectors
            const float* qj = qbase + j * D;
            if (!il) {
#pragma unroll
              for (int e = 0; e < CH; e += 4) {
                const float4 a = *reinterpret_cast<const float4*>(qj + f0 + e);
                const float4 b = *reinterpret_cast<const float4*>(qj + D / 2 + f0 + e);
                qx[e] = a.x; qx[e + 1] = a.y; qx[e + 2] = a.z; qx[e + 3] = a.w;
                qy[e] = b.x; qy[e + 1] = b.y; qy[e + 2] = b.z; qy[e + 3] = b.w;
              }
            } else {
#pragma unroll
              for (int e = 0; e < CH; e += 2) {
                const float4 a = *reinterpret_cast<const float4*>(qj + 2 * (f0 + e));
                qx[e] = a.x; qy[e] = a.y; qx[e + 1] = a.z; qy[e + 1] = a.w;
              }
            }
#pragma unroll
            for (int e = 0; e < CH; ++e) {
              sc[j] = fmaf(qx[e], kx[e], sc[j]);
              sc[j] = fmaf(qy[e], ky[e], sc[j]);
            }
          }
        }
      }
#pragma unroll
      for (int j = 0; j < HM; ++j)
#pragma unroll
        for (int k = 1; k < LPR; k <<= 1) sc[j] += __shfl_xor_sync(0xffffffffu, sc[j], k);
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
        if (part == 0) {
          dl[j] += pr;
          s_p[warp][trow][j] = pr;
        }
      }
      __syncwarp();
      // ---- dims on lanes: O[:, lane's dims] += p[:, row] v[row, lane's dims]
      const int nrow = min(TR, r1 - rb);
#pragma unroll 4
      for (int i = 0; i < nrow; ++i) {
        if (s_row[buf][warp][i] < 0) continue;  // no row (bad page: error recorded)
        float v[E];
        load_smem_f32<KT, E>(reinterpret_cast<const KT*>(st_v + i * RB) + lane * E, v);
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
      __syncwarp();  // s_p is rewritten by the next tile, this stage by the one after
      off = off_next;
    }
    // warp states -> shared memory (unnormalised O, m, d = the lanes' shares summed),
    // over the Q rows, probabilities and stages, once every warp is done with them
    __syncthreads();
#pragma unroll
    for (int j = 0; j < G8; ++j) {
      const float d = j < HM ? warp_sum(dl[j < HM ? j : 0]) : 0.f;
      if (lane == 0) {
        sm_m[warp * G8 + j] = j < HM ? m[j < HM ? j : 0] : kEmptyM;
        sm_d[warp * G8 + j] = d;
      }
#pragma unroll
      for (int e = 0; e < E; ++e)
        sm_o[(warp * G8 + j) * D + lane * E + e] = j < HM ? o[j < HM ? j : 0][e] : 0.f;
    }
  };
  if (hcount <= 4) tiles(std::integral_constant<int, 4>{});
  else tiles(std::integral_constant<int, 8>{});
  __syncthreads();
  finish_share<NT, NW>(p, br, sg, ua, ub, hq0, hcount, sm_m, sm_d, sm_o);
  if (sg.off + sg.n >= br.x1 || !next_segment(p, sg)) break;
  }  // segments
}

// ------------------------------------------------------------------------- dispatch
// Launch, or (ctas != nullptr) report how many blocks of the variant fit on one SM.
template <typename KT, typename QT, int D>
static cudaError_t launch_simt_d(const DecodeParams& p, dim3 grid, cudaStream_t st, int* ctas) {
  // 8 warps per block: a sequence's rows spread over twice the warps when each block
  // serves one (sequence, head slice) whole (no split), and one block of 8 warps holds
  // an SM like two of 4 would (registers)
  constexpr int NW = 8;
  using SM = SimtSmem<KT, D, NW>;
  const int smem = p.rotary && !p.k_rotated ? SM::kBytesRope : SM::kBytes;
  auto kern = decode_simt_kernel<KT, QT, D, NW>;
  // the dynamic shared memory above the default 48 KB is opted into once per device
  static bool opted[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!opted[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kBytesRope);
    if (e != cudaSuccess) return e;
    opted[dev] = true;
  }
  if (ctas) return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, kern, NW * 32, smem);
  return launch_pdl(kern, grid, dim3(NW * 32), smem, st, p);
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
