// Tensor-core decode kernel for 16-bit and FP8 KV caches (sm_103a).
//
// Block = one (work item, KV head, slice of <= 8 query heads): up to 8 query heads
// that share one KV head, over one chunk of a sequence's attended rows; every K/V
// byte of the chunk is read once per block.
//
// Every warp streams its own 16-row tiles (one page = P/16 tiles; pages go to the
// warps round-robin) straight from HBM into registers with 16-byte loads: on GB300
// this gathers scattered 4 KB page blocks faster than TMA, bulk copies or cp.async
// staging (see profiles/page_gather_probe.md).  The loads are laid out so that the
// registers already are mma.sync fragments:
//   - S^T = K Q^T (m16n8k16, fp32 accumulate): A = the K tile (16 rows x 16 dims per
//     k-tile), B = Q^T with the <= 8 query heads of the KV group as the n dimension.
//     A thread loads 16 contiguous bytes of its rows per chunk; the dot product's
//     k order is permuted to match, and Q's B fragments use the same permutation.
//   - online base-2 softmax on the accumulator fragments (TVM `batch_decode_paged_kv`:
//     running max m, sum d, output O), P^T rebuilt as a B fragment with 4 shuffles;
//   - O^T += V^T P^T: A = V^T built from 16-byte row loads with byte permutes (the
//     output dims are permuted and written back in order at the end).
// The next tile's K loads are issued right after QK and its V loads right after PV,
// so each warp keeps about one tile in flight while it computes.
// RoPE (rotate-half) is applied to K in registers before the MMA; rotated K and Q are
// split into hi + lo 16-bit parts so the products keep ~16 mantissa bits.  FP8 codes
// become f16 in registers (exact); k_scale folds into the score scale, v_scale into
// the output.  The warps' states are merged at the end (finish_block).
//
// Limits: head dim 64/128 for 16-bit KV, 128 for FP8; page size a multiple of 16.
#pragma once

#include "decode_common.cuh"
#include "kernels.h"

namespace pd {

constexpr int kMmaWarps = 4;

template <typename KVT, typename QT, int D, bool ROPE>
struct MmaTraits {
  static constexpr bool kFp8 = sizeof(KVT) == 1;
  using MT = typename std::conditional<std::is_same<KVT, __nv_bfloat16>::value, __nv_bfloat16,
                                       __half>::type;  // tensor-core input type
  static constexpr int kRowBytes = D * ElemBytes<KVT>::v;
  static constexpr int kKT = D / 16;             // k-tiles of QK, m-tiles of PV
  static constexpr int kKCh = kRowBytes / 64;    // 16-byte K chunks per row per thread
  static constexpr int kVCh = kRowBytes / 128;   // 16-byte V chunks per row per thread
  static constexpr bool kQSplit = ROPE || kFp8 || !std::is_same<QT, MT>::value;
  static_assert(kRowBytes == 128 || kRowBytes == 256, "row must be 128 or 256 bytes");
};

// Dim of A-fragment element (k-tile kt, half 0: k-pos 2q..2q+1 / half 1: 2q+8..2q+9,
// element e) for thread quad index q4: thread q4 owns 16-byte chunks 4c + q4 of a row.
template <bool FP8>
__device__ __forceinline__ int frag_dim(int kt, int half, int e, int q4) {
  return FP8 ? 16 * (4 * (kt >> 2) + q4) + 4 * (kt & 3) + 2 * half + e
             : 8 * (4 * (kt >> 1) + q4) + 4 * (kt & 1) + 2 * half + e;
}

// Output dim of O^T fragment row (m-tile mt, row g_id or g_id + 8 when `hi`).
template <bool FP8>
__device__ __forceinline__ int out_dim(int mt, int g_id, int hi) {
  return FP8 ? 16 * g_id + 2 * mt + hi : 8 * (g_id + 8 * (mt >> 2)) + 2 * (mt & 3) + hi;
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ uint32_t comp(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

template <typename KVT, typename QT, int D, bool ROPE, int NW>
__global__ void __launch_bounds__(NW * 32)
    decode_mma_kernel(const __grid_constant__ DecodeParams p) {
  using Tr = MmaTraits<KVT, QT, D, ROPE>;
  using MT = typename Tr::MT;
  constexpr int NT = NW * 32;
  constexpr int KT = Tr::kKT;
  constexpr int RB = Tr::kRowBytes;
  constexpr int KCH = Tr::kKCh;
  constexpr int VCH = Tr::kVCh;
  constexpr bool FP8 = Tr::kFp8;
  __shared__ float sm_m[NW * 8], sm_d[NW * 8];
  __shared__ float sm_o[NW * 8 * D];

  const BlockRange br = block_range<NT>(p);
  if (br.x0 >= br.x1) return;  // no units for this block

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g_id = lane >> 2, q4 = lane & 3;
  const int P = p.P;
  const uint8_t* kv_base = reinterpret_cast<const uint8_t*>(p.pages);
  const size_t block_bytes = (size_t)P * RB;                 // one (page, K|V, head) block
  const size_t v_off = (size_t)p.H_kv * block_bytes;         // K block -> V block
  __shared__ uint4 s_qf[KT][32];
  __shared__ unsigned long long s_ropeF[ROPE ? D / 2 : 1];  // RoPE frequencies (fixed point)
  __shared__ float2 s_rot8[ROPE ? D / 2 : 1];               // e^(i * 8 * omega_f)
  if (ROPE) {
    for (int i = threadIdx.x; i < D / 2; i += NT) {
      const unsigned long long F = p.rope_F[i];
      s_ropeF[i] = F;
      float c8, s8;
      rope_cos_sin(8, F, c8, s8);
      s_rot8[i] = make_float2(c8, s8);
    }
  }

  // The block walks the segments (sequence, head slice) its unit range [x0, x1) touches.
  Segment sg = br.seg;
  for (;;) {
  const int ua = (int)max(br.x0 - sg.off, 0ll);
  const int ub = (int)min(br.x1 - sg.off, (long long)sg.n);
  const int hk = sg.hz / p.n_z, z = sg.hz - (sg.hz / p.n_z) * p.n_z;
  const Pieces pcs = make_pieces(0, sg.seq.L, sg.seq, P);
  const int pend = min(ub, sg.seq.L > 0 ? pcs.count() : 0);  // pieces [ua, pend) here
  const int hq0 = hk * p.group + z * kMaxGroupPerCta;
  const int hcount = min(kMaxGroupPerCta, p.group - z * kMaxGroupPerCta);

  // ---------------------------------------------------------------- Q^T B fragments
  // Per k-tile and lane: {hi b0, hi b1, lo b0, lo b1} with b0 = (k 2q..2q+1, head g_id),
  // b1 = (k 2q+8..2q+9, head g_id) in the permuted dim order.  Built once per segment in
  // shared memory (k-tile pairs kt / kt + KT/2 spread over the warps), read per k-tile.
  {
    const bool have = g_id < hcount;
    const QT* qrow = reinterpret_cast<const QT*>(p.Q) + ((size_t)sg.b * p.H_qo + hq0 + (have ? g_id : 0)) * D;
    const int qpos = ROPE ? p.q_rope_position[sg.b] : 0;
    for (int kt = warp; kt < KT / 2; kt += NW) {
      float qv[2][2][2];  // [pair member u: kt, kt + KT/2][half][e]
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int e = 0; e < 2; ++e)
            qv[u][h][e] = have ? to_f32(qrow[frag_dim<FP8>(kt + u * (KT / 2), h, e, q4)]) : 0.f;
      if (ROPE) {
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float c, sn;
            rope_cos_sin(qpos, p.rope_F[frag_dim<FP8>(kt, h, e, q4)], c, sn);
            const float x = qv[0][h][e], y = qv[1][h][e];
            qv[0][h][e] = x * c - y * sn;
            qv[1][h][e] = y * c + x * sn;
          }
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        uint32_t hi[2], lo[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (Tr::kQSplit) {
            split2<MT>(qv[u][h][0] * p.q_prescale, qv[u][h][1] * p.q_prescale, hi[h], lo[h]);
          } else {
            hi[h] = pack2<MT>(qv[u][h][0], qv[u][h][1]);
            lo[h] = 0u;
          }
        }
        s_qf[kt + u * (KT / 2)][lane] = make_uint4(hi[0], hi[1], lo[0], lo[1]);
      }
    }
  }
  __syncthreads();
  const float post_scale = Tr::kQSplit ? 1.f : p.score_scale;
  const int kpos0 = ROPE ? p.k_rope_pos_offset[sg.b] : 0;

  float st_m[2] = {kEmptyM, kEmptyM}, st_d[2] = {0.f, 0.f};
  float oacc[KT][4];
#pragma unroll
  for (int i = 0; i < KT; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;

  // ---------------------------------------------------------------- tile stream
  // This warp's pieces are warp, warp + NW, ...; their page ids are looked up 32 at
  // a time (one per lane) and handed out with a shuffle.
  struct Tile {
    int piece, t, s_lo, s_hi, r_lo;
    const uint8_t* kblk;  // K block of (page, hk); nullptr = no more tiles
  };
  const int my_pieces = pend - ua > warp ? (pend - ua - warp + NW - 1) / NW : 0;
  int batch_base = -32, batch_page = -1;
  auto page_for = [&](int j) -> int {  // j = index among this warp's pieces (warp-uniform)
    if (j >= batch_base + 32) {
      batch_base = j - (j % 32);
      const int jj = batch_base + lane;
      batch_page = jj < my_pieces ? lookup_page(p, sg.seq, get_piece(pcs, ua + warp + jj * NW, P).page_idx) : -1;
    }
    return __shfl_sync(0xffffffffu, batch_page, j - batch_base);
  };
  auto first_tile_from = [&](int j) -> Tile {  // first tile of this warp's piece j or later
    Tile tl;
    tl.kblk = nullptr;
    for (; j < my_pieces; ++j) {
      const int pg = page_for(j);
      if (pg < 0) continue;  // bad page id: its rows are skipped (error already recorded)
      const Piece pc = get_piece(pcs, ua + warp + j * NW, P);
      tl.piece = j;
      tl.t = pc.s_lo >> 4;
      tl.s_lo = pc.s_lo;
      tl.s_hi = pc.s_hi;
      tl.r_lo = pc.r_lo;
      tl.kblk = kv_base + (((size_t)pg * 2) * p.H_kv + hk) * block_bytes;
      break;
    }
    return tl;
  };
  auto next_tile = [&](const Tile& c) -> Tile {
    if ((c.t + 1) * 16 < c.s_hi) {
      Tile n = c;
      n.t = c.t + 1;
      return n;
    }
    return first_tile_from(c.piece + 1);
  };
  uint4 kr[2][KCH];      // K rows t*16 + g_id (+8): chunks 4c + q4
  uint4 vr[4][VCH];      // V rows t*16 + 2q4, +1, +8, +9: chunks g_id + 8j
  auto load_k = [&](const Tile& c) {
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const uint8_t* row = c.kblk + (size_t)(c.t * 16 + g_id + 8 * rr) * RB;
#pragma unroll
      for (int ch = 0; ch < KCH; ++ch) kr[rr][ch] = ldg_stream(row + (4 * ch + q4) * 16);
    }
  };
  auto load_v = [&](const Tile& c) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int slot = c.t * 16 + 2 * q4 + (i & 1) + 8 * (i >> 1);
      const uint8_t* row = c.kblk + v_off + (size_t)slot * RB;
#pragma unroll
      for (int j = 0; j < VCH; ++j) vr[i][j] = ldg_stream(row + (g_id + 8 * j) * 16);
    }
  };

  Tile cur = first_tile_from(0);
  if (cur.kblk) {
    load_k(cur);
    load_v(cur);
  }
  while (cur.kblk) {
    const int slot0 = cur.t * 16 + g_id, slot1 = slot0 + 8;
    const bool v0 = slot0 >= cur.s_lo && slot0 < cur.s_hi;
    const bool v1 = slot1 >= cur.s_lo && slot1 < cur.s_hi;
    // ------------------------------------------------------------ S^T = K Q^T
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if constexpr (!ROPE) {
#pragma unroll
      for (int kt = 0; kt < KT; ++kt) {
        uint32_t a[4];
        if constexpr (FP8) {
          const uint32_t r0w = comp(kr[0][kt >> 2], kt & 3), r1w = comp(kr[1][kt >> 2], kt & 3);
          a[0] = e4m3x2_to_f16x2((uint16_t)(r0w & 0xffff));
          a[2] = e4m3x2_to_f16x2((uint16_t)(r0w >> 16));
          a[1] = e4m3x2_to_f16x2((uint16_t)(r1w & 0xffff));
          a[3] = e4m3x2_to_f16x2((uint16_t)(r1w >> 16));
        } else {
          a[0] = comp(kr[0][kt >> 1], 2 * (kt & 1));
          a[2] = comp(kr[0][kt >> 1], 2 * (kt & 1) + 1);
          a[1] = comp(kr[1][kt >> 1], 2 * (kt & 1));
          a[3] = comp(kr[1][kt >> 1], 2 * (kt & 1) + 1);
        }
        const uint4 qf = s_qf[kt][lane];
        Mma<MT>::run(acc, a, qf.x, qf.y);
        if (Tr::kQSplit) Mma<MT>::run(acc, a, qf.z, qf.w);
      }
    } else {
      // RoPE on K in registers: k-tiles kt and kt + KT/2 hold dims d and d + D/2
      const int pos0 = kpos0 + cur.r_lo + (slot0 - cur.s_lo);  // row g_id; row g_id + 8 is pos0 + 8
#pragma unroll
      for (int kt = 0; kt < KT / 2; ++kt) {
        uint32_t araw[2][4];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int ktu = kt + u * (KT / 2);
          if constexpr (FP8) {
            const uint32_t r0w = comp(kr[0][ktu >> 2], ktu & 3), r1w = comp(kr[1][ktu >> 2], ktu & 3);
            araw[u][0] = e4m3x2_to_f16x2((uint16_t)(r0w & 0xffff));
            araw[u][2] = e4m3x2_to_f16x2((uint16_t)(r0w >> 16));
            araw[u][1] = e4m3x2_to_f16x2((uint16_t)(r1w & 0xffff));
            araw[u][3] = e4m3x2_to_f16x2((uint16_t)(r1w >> 16));
          } else {
            araw[u][0] = comp(kr[0][ktu >> 1], 2 * (ktu & 1));
            araw[u][2] = comp(kr[0][ktu >> 1], 2 * (ktu & 1) + 1);
            araw[u][1] = comp(kr[1][ktu >> 1], 2 * (ktu & 1));
            araw[u][3] = comp(kr[1][ktu >> 1], 2 * (ktu & 1) + 1);
          }
        }
        uint32_t ahi[2][4], alo[2][4];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          // (cos, sin) of this half's two frequencies at rows g_id (direct) and g_id + 8
          float cs[2][2][2];  // [row][e][cos|sin]
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int f = frag_dim<FP8>(kt, half, e, q4);
            rope_cos_sin(pos0, s_ropeF[f], cs[0][e][0], cs[0][e][1]);
            const float2 r8 = s_rot8[f];
            cs[1][e][0] = cs[0][e][0] * r8.x - cs[0][e][1] * r8.y;
            cs[1][e][1] = cs[0][e][1] * r8.x + cs[0][e][0] * r8.y;
          }
#pragma unroll
          for (int row = 0; row < 2; ++row) {
            const int ai = 2 * half + row;
            const float2 x = unpack2<MT>(araw[0][ai]);
            const float2 y = unpack2<MT>(araw[1][ai]);
            const float c0 = cs[row][0][0], s0 = cs[row][0][1], c1 = cs[row][1][0], s1 = cs[row][1][1];
            split2<MT>(x.x * c0 - y.x * s0, x.y * c1 - y.y * s1, ahi[0][ai], alo[0][ai]);
            split2<MT>(y.x * c0 + x.x * s0, y.y * c1 + x.y * s1, ahi[1][ai], alo[1][ai]);
          }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const uint4 qf = s_qf[kt + u * (KT / 2)][lane];
          Mma<MT>::run(acc, ahi[u], qf.x, qf.y);
          Mma<MT>::run(acc, alo[u], qf.x, qf.y);
          Mma<MT>::run(acc, ahi[u], qf.z, qf.w);
        }
      }
    }
    // K registers are free: start the next tile's K loads
    const Tile nxt = next_tile(cur);
    if (nxt.kblk) load_k(nxt);
    // ------------------------------------------------------------ online softmax (log2)
    float sc[4];
    sc[0] = v0 ? acc[0] * post_scale : -INFINITY;  // row g_id, heads 2q, 2q+1
    sc[1] = v0 ? acc[1] * post_scale : -INFINITY;
    sc[2] = v1 ? acc[2] * post_scale : -INFINITY;  // row g_id + 8
    sc[3] = v1 ? acc[3] * post_scale : -INFINITY;
    const float tm0 = max_over_groups(fmaxf(sc[0], sc[2]));
    const float tm1 = max_over_groups(fmaxf(sc[1], sc[3]));
    const float mn0 = fmaxf(st_m[0], tm0), mn1 = fmaxf(st_m[1], tm1);
    const float al0 = fast_exp2(st_m[0] - mn0), al1 = fast_exp2(st_m[1] - mn1);
    float pr[4];
    pr[0] = fast_exp2(sc[0] - mn0);
    pr[1] = fast_exp2(sc[1] - mn1);
    pr[2] = fast_exp2(sc[2] - mn0);
    pr[3] = fast_exp2(sc[3] - mn1);
    st_d[0] = st_d[0] * al0 + pr[0] + pr[2];
    st_d[1] = st_d[1] * al1 + pr[1] + pr[3];
    st_m[0] = mn0;
    st_m[1] = mn1;
    if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
      for (int mt = 0; mt < KT; ++mt) {
        oacc[mt][0] *= al0;
        oacc[mt][1] *= al1;
        oacc[mt][2] *= al0;
        oacc[mt][3] *= al1;
      }
    }
    // P^T as a B fragment: rows 2q,2q+1 | 2q+8,2q+9 of head g_id
    uint32_t pb0, pb1;
    {
      const uint32_t x0 = pack2<MT>(pr[0], pr[2]);  // head 2q: rows g_id, g_id+8
      const uint32_t x1 = pack2<MT>(pr[1], pr[3]);  // head 2q+1
      const int srcA = 8 * q4 + (g_id >> 1), srcB = srcA + 4;
      const uint32_t a0 = __shfl_sync(0xffffffffu, x0, srcA);
      const uint32_t a1 = __shfl_sync(0xffffffffu, x1, srcA);
      const uint32_t b0 = __shfl_sync(0xffffffffu, x0, srcB);
      const uint32_t b1 = __shfl_sync(0xffffffffu, x1, srcB);
      const uint32_t va = (g_id & 1) ? a1 : a0, vb = (g_id & 1) ? b1 : b0;
      pb0 = __byte_perm(va, vb, 0x5410);
      pb1 = __byte_perm(va, vb, 0x7632);
    }
    // rows of this thread's V^T halves: 2q, 2q+1 (a0, a1) and 2q+8, 2q+9 (a2, a3);
    // rows outside the piece may hold anything (even NaN): zero them
    uint32_t vm01 = 0xffffffffu, vm23 = 0xffffffffu;
    if ((cur.t * 16 < cur.s_lo) || (cur.t * 16 + 16 > cur.s_hi)) {
      const int rA = cur.t * 16 + 2 * q4, rB = rA + 8;
      vm01 = ((rA >= cur.s_lo && rA < cur.s_hi) ? 0x0000ffffu : 0u) |
             ((rA + 1 >= cur.s_lo && rA + 1 < cur.s_hi) ? 0xffff0000u : 0u);
      vm23 = ((rB >= cur.s_lo && rB < cur.s_hi) ? 0x0000ffffu : 0u) |
             ((rB + 1 >= cur.s_lo && rB + 1 < cur.s_hi) ? 0xffff0000u : 0u);
    }
    // ------------------------------------------------------------ O^T += V^T P^T
#pragma unroll
    for (int mt = 0; mt < KT; ++mt) {
      uint32_t a[4];
      if constexpr (FP8) {
        const int ci = mt >> 1;
        const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
        const uint32_t xy01 = __byte_perm(comp(vr[0][0], ci), comp(vr[1][0], ci), sel);
        const uint32_t xy23 = __byte_perm(comp(vr[2][0], ci), comp(vr[3][0], ci), sel);
        a[0] = e4m3x2_to_f16x2((uint16_t)(xy01 & 0xffff)) & vm01;
        a[1] = e4m3x2_to_f16x2((uint16_t)(xy01 >> 16)) & vm01;
        a[2] = e4m3x2_to_f16x2((uint16_t)(xy23 & 0xffff)) & vm23;
        a[3] = e4m3x2_to_f16x2((uint16_t)(xy23 >> 16)) & vm23;
      } else {
        const int j = mt >> 2, ci = mt & 3;
        const uint32_t x0 = comp(vr[0][j], ci), x1 = comp(vr[1][j], ci);
        const uint32_t y0 = comp(vr[2][j], ci), y1 = comp(vr[3][j], ci);
        a[0] = __byte_perm(x0, x1, 0x5410) & vm01;
        a[1] = __byte_perm(x0, x1, 0x7632) & vm01;
        a[2] = __byte_perm(y0, y1, 0x5410) & vm23;
        a[3] = __byte_perm(y0, y1, 0x7632) & vm23;
      }
      Mma<MT>::run(oacc[mt], a, pb0, pb1);
    }
    if (nxt.kblk) load_v(nxt);
    cur = nxt;
  }
  st_d[0] = sum_over_groups(st_d[0]);
  st_d[1] = sum_over_groups(st_d[1]);

  // ---------------------------------------------------------------- merge + finish
  if (g_id == 0) {
    sm_m[warp * 8 + 2 * q4] = st_m[0];
    sm_m[warp * 8 + 2 * q4 + 1] = st_m[1];
    sm_d[warp * 8 + 2 * q4] = st_d[0];
    sm_d[warp * 8 + 2 * q4 + 1] = st_d[1];
  }
#pragma unroll
  for (int mt = 0; mt < KT; ++mt) {
    const int dA = out_dim<FP8>(mt, g_id, 0), dB = out_dim<FP8>(mt, g_id, 1);
    sm_o[(warp * 8 + 2 * q4) * D + dA] = oacc[mt][0];
    sm_o[(warp * 8 + 2 * q4 + 1) * D + dA] = oacc[mt][1];
    sm_o[(warp * 8 + 2 * q4) * D + dB] = oacc[mt][2];
    sm_o[(warp * 8 + 2 * q4 + 1) * D + dB] = oacc[mt][3];
  }
  __syncthreads();
  finish_share<NT, NW>(p, br, sg, ua, ub, hq0, hcount, sm_m, sm_d, sm_o);
  if (sg.off + sg.n >= br.x1 || !next_segment(p, sg)) break;
  }  // segments
}

template <typename KVT, typename QT, int D, bool ROPE>
static cudaError_t launch_mma_t(const DecodeParams& p, dim3 grid, cudaStream_t st, MmaConfig* cfg) {
  constexpr int NW = kMmaWarps;
  auto kern = decode_mma_kernel<KVT, QT, D, ROPE, NW>;
  if (cfg) {
    cfg->threads = NW * 32;
    cfg->smem_bytes = 0;
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, NW * 32, 0);
    if (e != cudaSuccess) return e;
    cfg->ctas_per_sm = n;
    return cudaSuccess;
  }
  kern<<<grid, NW * 32, 0, st>>>(p);
  return cudaGetLastError();
}

template <typename KVT, typename QT, int D>
static cudaError_t launch_mma_r(const DecodeParams& p, dim3 grid, cudaStream_t st, MmaConfig* cfg) {
  if (p.rotary) return launch_mma_t<KVT, QT, D, true>(p, grid, st, cfg);
  return launch_mma_t<KVT, QT, D, false>(p, grid, st, cfg);
}

}  // namespace pd
