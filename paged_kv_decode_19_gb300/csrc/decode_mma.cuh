// Tensor-core decode kernel for 16-bit and FP8 KV caches (sm_103a).
//
// Block = one (work item, KV head, slice of <= 8 query heads) = up to 8 query heads
// that share one KV head, over one chunk of a sequence's attended rows; every K/V
// byte of the chunk is read once per block.
//
//   warp NC (producer): walks the chunk's pages ("pieces"), looks the page ids up in
//     the page table (32 at a time, one per lane, prefetched a batch ahead) and
//     streams each page's K and V tiles into a ring of NS shared-memory stages with
//     TMA (cp.async.bulk.tensor, 128B-swizzled), completion on an mbarrier;
//   warps 0..NC-1 (consumers): take pieces round-robin; per 16-row tile
//     S^T = K Q^T with mma.sync m16n8k16 (A = K tile by ldmatrix, B = Q^T: the 8 heads
//     are the n dimension), online base-2 softmax on the accumulator fragments
//     (TVM `batch_decode_paged_kv`: m, d, O), P^T rebuilt as a B fragment with four
//     shuffles, then O^T += V^T P^T (A = V^T by ldmatrix.trans, or for FP8 by byte
//     permutes).  RoPE (rotate-half) is applied to K in registers before the MMA; the
//     rotated K and Q are then split into hi + lo 16-bit parts so that the tensor-core
//     products keep ~16 mantissa bits.  FP8 codes are converted to f16 in registers
//     (exact); k_scale folds into the score scale and v_scale into the output.
//   finish: the consumers' states are merged through shared memory, then the block
//     writes the output or a partial state (see finish_block).
//
// Limits: head dim 64/128 for 16-bit KV, 128 for FP8; page size a multiple of 16
// (<= 256); row bytes D * elem a multiple of 128.
#pragma once

#include "decode_common.cuh"
#include "kernels.h"

namespace pd {

constexpr int kMmaConsumers = 4;
constexpr int kMaxStages = 16;
constexpr int kStageBudgetBytes = 48 * 1024;

// Byte address of (row, byte) inside a TMA box region laid out with 128B swizzle:
// boxes of 128-byte rows, P rows each, 1024-byte aligned.
__device__ __forceinline__ uint32_t swz(uint32_t base, int P, int row, int byte) {
  return base + (uint32_t)((byte >> 7) * P * 128 + row * 128 +
                           ((((byte & 127) >> 4) ^ (row & 7)) << 4) + (byte & 15));
}

template <typename KVT, typename QT, int D, bool ROPE>
struct MmaTraits {
  static constexpr bool kFp8 = sizeof(KVT) == 1;
  using MT = typename std::conditional<std::is_same<KVT, __nv_bfloat16>::value, __nv_bfloat16,
                                       __half>::type;  // tensor-core input type
  static constexpr int kElem = ElemBytes<KVT>::v;
  static constexpr int kRowBytes = D * kElem;
  static constexpr int kKT = D / 16;  // k-tiles of QK, m-tiles of PV
  static constexpr bool kQSplit = ROPE || kFp8 || !std::is_same<QT, MT>::value;
  static constexpr bool kKSplit = ROPE;
  static_assert(kRowBytes % 128 == 0, "row bytes must be a multiple of 128");
  static_assert(kMaxStages % kMmaConsumers == 0, "stage ring must split evenly over consumers");
};

// dim held by fragment half `half` (0: k-pos 2q..2q+1, 1: 2q+8..2q+9), element e, k-tile kt
template <bool FP8>
__device__ __forceinline__ int frag_dim(int kt, int half, int e, int q4) {
  return FP8 ? kt * 16 + 4 * q4 + half * 2 + e : kt * 16 + 2 * q4 + half * 8 + e;
}

template <typename KVT, typename QT, int D, bool ROPE, int NC>
__global__ void __launch_bounds__((NC + 1) * 32)
    decode_mma_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap kv_map,
                      int ns) {
  using Tr = MmaTraits<KVT, QT, D, ROPE>;
  using MT = typename Tr::MT;
  constexpr int NT = (NC + 1) * 32;
  constexpr int KT = Tr::kKT;
  constexpr bool FP8 = Tr::kFp8;
  extern __shared__ uint8_t dyn_smem[];

  const int item = blockIdx.x, hk = blockIdx.y, z = blockIdx.z;
  Work w;
  if (!locate_item<NT>(p, item, w)) return;

  const int P = p.P;
  const int stage_bytes = 2 * P * Tr::kRowBytes;
  const uint32_t smem0 = (smem_u32(dyn_smem) + 1023u) & ~1023u;
  uint8_t* smem_gen = dyn_smem + (smem0 - smem_u32(dyn_smem));
  int* meta = reinterpret_cast<int*>(smem_gen + ns * stage_bytes);
  unsigned long long* ropeF = reinterpret_cast<unsigned long long*>(meta + kMaxStages);
  __shared__ __align__(8) unsigned long long bars[2 * kMaxStages];
  __shared__ int s_abort;
  const uint32_t full0 = smem_u32(&bars[0]), empty0 = smem_u32(&bars[kMaxStages]);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int s = 0; s < ns; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    s_abort = 0;
    fence_barrier_init();
  }
  if (ROPE)
    for (int i = tid; i < D / 2; i += NT) ropeF[i] = p.rope_F[i];
  __syncthreads();

  const int r0 = w.chunk * p.chunk_rows;
  const int r1 = (w.seq.L - r0 > p.chunk_rows) ? r0 + p.chunk_rows : w.seq.L;
  const Pieces pcs = make_pieces(r0, r1, w.seq, P);
  const int npieces = pcs.count();
  const int hq0 = hk * p.group + z * kMaxGroupPerCta;
  const int hcount = min(kMaxGroupPerCta, p.group - z * kMaxGroupPerCta);

  float st_m[2] = {kEmptyM, kEmptyM}, st_d[2] = {0.f, 0.f};
  float oacc[KT][4];
#pragma unroll
  for (int i = 0; i < KT; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;

  if (warp == NC) {
    // ------------------------------------------------------------------ producer
    int issued = 0;
    bool ok = true;
    auto page_of = [&](int i) -> int {
      if (i >= npieces) return -1;
      return lookup_page(p, w.seq, get_piece(pcs, i, P).page_idx);
    };
    int cur = page_of(lane);
    for (int base = 0; base < npieces && ok; base += 32) {
      const int nxt = page_of(base + 32 + lane);
      const int nb = min(32, npieces - base);
      for (int k = 0; k < nb; ++k) {
        const int pg = __shfl_sync(0xffffffffu, cur, k);
        const int i = base + k, s = i % ns, use = i / ns;
        if (lane == 0) {
          if (use > 0 && !mbar_wait(empty0 + 8 * s, (use - 1) & 1)) {
            set_error(p.err, kErrTimeout);
            s_abort = 1;
            ok = false;
          }
          if (ok) {
            meta[s] = pg;
            const uint32_t bar = full0 + 8 * s;
            if (pg >= 0) {
              mbar_arrive_expect_tx(bar, stage_bytes);
              const uint32_t dst = smem0 + s * stage_bytes;
#pragma unroll
              for (int kv = 0; kv < 2; ++kv)
#pragma unroll
                for (int bx = 0; bx < Tr::kRowBytes / 128; ++bx)
                  tma_load_3d(dst + kv * P * Tr::kRowBytes + bx * P * 128, &kv_map, bar,
                              bx * (128 / Tr::kElem), 0, (pg * 2 + kv) * p.H_kv + hk);
            } else {
              mbar_arrive(bar);
            }
            ++issued;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
      cur = nxt;
    }
    // drain: the most recent use of every stage must have landed before smem reuse
    if (lane == 0) {
      for (int i = max(0, issued - ns); i < issued; ++i)
        if (!mbar_wait(full0 + 8 * (i % ns), (i / ns) & 1)) set_error(p.err, kErrTimeout);
    }
  } else {
    // ------------------------------------------------------------------ consumers
    const int g_id = lane >> 2, q4 = lane & 3;
    // Q^T as B fragments: b0 = (k 2q..2q+1, head g_id), b1 = (k 2q+8..2q+9, head g_id)
    uint32_t qhi[KT][2], qlo[KT][2];
    {
      const int qpos = ROPE ? p.q_rope_position[w.b] : 0;
      const bool have = g_id < hcount;
      const QT* qrow = reinterpret_cast<const QT*>(p.Q) + ((size_t)w.b * p.H_qo + hq0 + (have ? g_id : 0)) * D;
      float qv[KT][2][2];
#pragma unroll
      for (int kt = 0; kt < KT; ++kt)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int e = 0; e < 2; ++e)
            qv[kt][h][e] = have ? to_f32(qrow[frag_dim<FP8>(kt, h, e, q4)]) : 0.f;
      if (ROPE) {
#pragma unroll
        for (int kt = 0; kt < KT / 2; ++kt)
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              float c, s;
              rope_cos_sin(qpos, ropeF[frag_dim<FP8>(kt, h, e, q4)], c, s);
              const float x = qv[kt][h][e], y = qv[kt + KT / 2][h][e];
              qv[kt][h][e] = x * c - y * s;
              qv[kt + KT / 2][h][e] = y * c + x * s;
            }
      }
#pragma unroll
      for (int kt = 0; kt < KT; ++kt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (Tr::kQSplit) {
            split2<MT>(qv[kt][h][0] * p.q_prescale, qv[kt][h][1] * p.q_prescale, qhi[kt][h], qlo[kt][h]);
          } else {
            qhi[kt][h] = pack2<MT>(qv[kt][h][0], qv[kt][h][1]);
            qlo[kt][h] = 0u;
          }
        }
    }
    const float post_scale = Tr::kQSplit ? 1.f : p.score_scale;
    const int kpos0 = ROPE ? p.k_rope_pos_offset[w.b] : 0;

    for (int i = warp; i < npieces; i += NC) {
      const int s = i % ns, use = i / ns;
      if (!mbar_wait(full0 + 8 * s, use & 1)) {
        set_error(p.err, kErrTimeout);
        s_abort = 1;
        break;
      }
      if (*(volatile int*)&s_abort) break;
      const int pg = meta[s];
      const Piece pc = get_piece(pcs, i, P);
      if (pg >= 0) {
        const uint32_t kbase = smem0 + s * stage_bytes;
        const uint32_t vbase = kbase + P * Tr::kRowBytes;
        for (int t = pc.s_lo >> 4; t * 16 < pc.s_hi; ++t) {
          const int slot0 = t * 16 + g_id, slot1 = slot0 + 8;
          const bool v0 = slot0 >= pc.s_lo && slot0 < pc.s_hi;
          const bool v1 = slot1 >= pc.s_lo && slot1 < pc.s_hi;
          // ---------------- S^T = K Q^T
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
          if constexpr (!ROPE) {
            if constexpr (!FP8) {
#pragma unroll
              for (int kt = 0; kt < KT; ++kt) {
                const int mi = lane >> 3;
                const uint32_t addr = swz(kbase, P, t * 16 + (mi & 1) * 8 + (lane & 7), (kt * 16 + (mi >> 1) * 8) * 2);
                uint32_t a[4];
                ldsm_x4(addr, a[0], a[1], a[2], a[3]);
                Mma<MT>::run(acc, a, qhi[kt][0], qhi[kt][1]);
                if (Tr::kQSplit) Mma<MT>::run(acc, a, qlo[kt][0], qlo[kt][1]);
              }
            } else {
#pragma unroll
              for (int c = 0; c < KT / 2; ++c) {
                const int mi = lane >> 3;
                const uint32_t addr = swz(kbase, P, t * 16 + (mi & 1) * 8 + (lane & 7), c * 32 + (mi >> 1) * 16);
                uint32_t r[4];
                ldsm_x4(addr, r[0], r[1], r[2], r[3]);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                  const int kt = 2 * c + u;
                  uint32_t a[4];
                  a[0] = e4m3x2_to_f16x2((uint16_t)(r[2 * u] & 0xffff));
                  a[2] = e4m3x2_to_f16x2((uint16_t)(r[2 * u] >> 16));
                  a[1] = e4m3x2_to_f16x2((uint16_t)(r[2 * u + 1] & 0xffff));
                  a[3] = e4m3x2_to_f16x2((uint16_t)(r[2 * u + 1] >> 16));
                  Mma<MT>::run(acc, a, qhi[kt][0], qhi[kt][1]);
                  Mma<MT>::run(acc, a, qlo[kt][0], qlo[kt][1]);
                }
              }
            }
          } else {
            // RoPE on K in registers: k-tiles kt and kt + KT/2 hold dims d and d + D/2
            const int pos0 = kpos0 + pc.r_lo + (slot0 - pc.s_lo);
            const int pos1 = pos0 + 8;
#pragma unroll
            for (int kt = 0; kt < KT / 2; ++kt) {
              uint32_t araw[2][4];
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                const int ktu = kt + u * (KT / 2);
                if constexpr (!FP8) {
                  const int mi = lane >> 3;
                  const uint32_t addr = swz(kbase, P, t * 16 + (mi & 1) * 8 + (lane & 7), (ktu * 16 + (mi >> 1) * 8) * 2);
                  ldsm_x4(addr, araw[u][0], araw[u][1], araw[u][2], araw[u][3]);
                } else {
                  // one x2 load per k-tile: matrix 0 rows 0-7, matrix 1 rows 8-15
                  const int mi = (lane >> 3) & 1;
                  const uint32_t addr = swz(kbase, P, t * 16 + mi * 8 + (lane & 7), ktu * 16);
                  uint32_t r0, r1;
                  ldsm_x2(addr, r0, r1);
                  araw[u][0] = e4m3x2_to_f16x2((uint16_t)(r0 & 0xffff));
                  araw[u][2] = e4m3x2_to_f16x2((uint16_t)(r0 >> 16));
                  araw[u][1] = e4m3x2_to_f16x2((uint16_t)(r1 & 0xffff));
                  araw[u][3] = e4m3x2_to_f16x2((uint16_t)(r1 >> 16));
                }
              }
              uint32_t ahi[2][4], alo[2][4];
#pragma unroll
              for (int ai = 0; ai < 4; ++ai) {
                const int half = ai >> 1;
                const int pos = (ai & 1) ? pos1 : pos0;
                const float2 x = unpack2<MT>(araw[0][ai]);
                const float2 y = unpack2<MT>(araw[1][ai]);
                float c0, s0, c1, s1;
                rope_cos_sin(pos, ropeF[frag_dim<FP8>(kt, half, 0, q4)], c0, s0);
                rope_cos_sin(pos, ropeF[frag_dim<FP8>(kt, half, 1, q4)], c1, s1);
                split2<MT>(x.x * c0 - y.x * s0, x.y * c1 - y.y * s1, ahi[0][ai], alo[0][ai]);
                split2<MT>(y.x * c0 + x.x * s0, y.y * c1 + x.y * s1, ahi[1][ai], alo[1][ai]);
              }
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                const int ktu = kt + u * (KT / 2);
                Mma<MT>::run(acc, ahi[u], qhi[ktu][0], qhi[ktu][1]);
                Mma<MT>::run(acc, alo[u], qhi[ktu][0], qhi[ktu][1]);
                Mma<MT>::run(acc, ahi[u], qlo[ktu][0], qlo[ktu][1]);
              }
            }
          }
          // ---------------- online softmax (log2 units); c0,c1: row g_id; c2,c3: row g_id+8
          float sc[4];
          sc[0] = v0 ? acc[0] * post_scale : -INFINITY;
          sc[1] = v0 ? acc[1] * post_scale : -INFINITY;
          sc[2] = v1 ? acc[2] * post_scale : -INFINITY;
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
          // ---------------- P^T as B fragment: rows 2q,2q+1 | 2q+8,2q+9 of head g_id
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
          // rows of this thread's V^T fragment halves: 2q, 2q+1 (a0,a1) and 2q+8, 2q+9 (a2,a3)
          const bool partial = (t * 16 < pc.s_lo) || (t * 16 + 16 > pc.s_hi);
          uint32_t vm01 = 0xffffffffu, vm23 = 0xffffffffu;
          if (partial) {
            const int rA = t * 16 + 2 * q4, rB = rA + 8;
            vm01 = ((rA >= pc.s_lo && rA < pc.s_hi) ? 0x0000ffffu : 0u) |
                   ((rA + 1 >= pc.s_lo && rA + 1 < pc.s_hi) ? 0xffff0000u : 0u);
            vm23 = ((rB >= pc.s_lo && rB < pc.s_hi) ? 0x0000ffffu : 0u) |
                   ((rB + 1 >= pc.s_lo && rB + 1 < pc.s_hi) ? 0xffff0000u : 0u);
          }
          // ---------------- O^T += V^T P^T
          if constexpr (!FP8) {
#pragma unroll
            for (int mt = 0; mt < KT; ++mt) {
              const int mi = lane >> 3;
              const uint32_t addr = swz(vbase, P, t * 16 + (mi >> 1) * 8 + (lane & 7), (mt * 16 + (mi & 1) * 8) * 2);
              uint32_t a[4];
              ldsm_x4_t(addr, a[0], a[1], a[2], a[3]);
              a[0] &= vm01;
              a[1] &= vm01;
              a[2] &= vm23;
              a[3] &= vm23;
              Mma<MT>::run(oacc[mt], a, pb0, pb1);
            }
          } else {
            const int rA = t * 16 + 2 * q4;
#pragma unroll
            for (int j = 0; j < KT / 2; ++j) {
              const int byte = 32 * j + 4 * g_id;
              const uint32_t w0 = lds_u32(swz(vbase, P, rA, byte));
              const uint32_t w1 = lds_u32(swz(vbase, P, rA + 1, byte));
              const uint32_t w2 = lds_u32(swz(vbase, P, rA + 8, byte));
              const uint32_t w3 = lds_u32(swz(vbase, P, rA + 9, byte));
              const uint32_t x01 = __byte_perm(w0, w1, 0x5140), x23 = __byte_perm(w0, w1, 0x7362);
              const uint32_t y01 = __byte_perm(w2, w3, 0x5140), y23 = __byte_perm(w2, w3, 0x7362);
              uint32_t a[4];
              a[0] = e4m3x2_to_f16x2((uint16_t)(x01 & 0xffff)) & vm01;
              a[1] = e4m3x2_to_f16x2((uint16_t)(x01 >> 16)) & vm01;
              a[2] = e4m3x2_to_f16x2((uint16_t)(y01 & 0xffff)) & vm23;
              a[3] = e4m3x2_to_f16x2((uint16_t)(y01 >> 16)) & vm23;
              Mma<MT>::run(oacc[2 * j], a, pb0, pb1);
              a[0] = e4m3x2_to_f16x2((uint16_t)(x23 & 0xffff)) & vm01;
              a[1] = e4m3x2_to_f16x2((uint16_t)(x23 >> 16)) & vm01;
              a[2] = e4m3x2_to_f16x2((uint16_t)(y23 & 0xffff)) & vm23;
              a[3] = e4m3x2_to_f16x2((uint16_t)(y23 >> 16)) & vm23;
              Mma<MT>::run(oacc[2 * j + 1], a, pb0, pb1);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * s);
    }
    st_d[0] = sum_over_groups(st_d[0]);
    st_d[1] = sum_over_groups(st_d[1]);
  }

  // ------------------------------------------------------------------ merge + finish
  __syncthreads();  // all stages consumed (or abandoned and drained): smem reusable
  float* sm_m = reinterpret_cast<float*>(smem_gen);
  float* sm_d = sm_m + NC * 8;
  float* sm_o = sm_d + NC * 8;
  if (warp < NC) {
    const int g_id = lane >> 2, q4 = lane & 3;
    if (g_id == 0) {
      sm_m[warp * 8 + 2 * q4] = st_m[0];
      sm_m[warp * 8 + 2 * q4 + 1] = st_m[1];
      sm_d[warp * 8 + 2 * q4] = st_d[0];
      sm_d[warp * 8 + 2 * q4 + 1] = st_d[1];
    }
#pragma unroll
    for (int mt = 0; mt < KT; ++mt) {
      int dA, dB;
      if (FP8) {
        dA = 32 * (mt >> 1) + 4 * g_id + 2 * (mt & 1);
        dB = dA + 1;
      } else {
        dA = mt * 16 + g_id;
        dB = dA + 8;
      }
      sm_o[(warp * 8 + 2 * q4) * D + dA] = oacc[mt][0];
      sm_o[(warp * 8 + 2 * q4 + 1) * D + dA] = oacc[mt][1];
      sm_o[(warp * 8 + 2 * q4) * D + dB] = oacc[mt][2];
      sm_o[(warp * 8 + 2 * q4 + 1) * D + dB] = oacc[mt][3];
    }
  }
  __syncthreads();
  finish_block<NT, NC>(p, w, item, hk, z, hq0, hcount, sm_m, sm_d, sm_o);
}

template <typename KVT, typename QT, int D, bool ROPE>
static int mma_smem_bytes(int P, int* ns_out) {
  // The stage count is a multiple of the consumer count: stage s is then always
  // consumed by warp s % NC, in order, which the parity waits rely on.
  const int stage = 2 * P * D * ElemBytes<KVT>::v;
  int ns = kStageBudgetBytes / stage / kMmaConsumers * kMmaConsumers;
  ns = ns < kMmaConsumers ? kMmaConsumers : (ns > kMaxStages ? kMaxStages : ns);
  const int merge = kMmaConsumers * 8 * (D + 2) * 4;
  int body = ns * stage;
  if (body < merge) body = merge;
  if (ns_out) *ns_out = ns;
  return 1024 + body + kMaxStages * 4 + (D / 2) * 8;
}

template <typename KVT, typename QT, int D, bool ROPE>
static cudaError_t launch_mma_t(const DecodeParams& p, const CUtensorMap& map, dim3 grid,
                                cudaStream_t st, MmaConfig* cfg) {
  constexpr int NC = kMmaConsumers;
  auto kern = decode_mma_kernel<KVT, QT, D, ROPE, NC>;
  int ns = 0;
  const int smem = mma_smem_bytes<KVT, QT, D, ROPE>(p.P, &ns);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  if (cfg) {
    cfg->threads = (NC + 1) * 32;
    cfg->smem_bytes = smem;
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, (NC + 1) * 32, smem);
    if (e != cudaSuccess) return e;
    cfg->ctas_per_sm = n;
    return cudaSuccess;
  }
  kern<<<grid, (NC + 1) * 32, smem, st>>>(p, map, ns);
  return cudaGetLastError();
}

template <typename KVT, typename QT, int D>
static cudaError_t launch_mma_r(const DecodeParams& p, const CUtensorMap& map, dim3 grid,
                                cudaStream_t st, MmaConfig* cfg) {
  if (p.rotary) return launch_mma_t<KVT, QT, D, true>(p, map, grid, st, cfg);
  return launch_mma_t<KVT, QT, D, false>(p, map, grid, st, cfg);
}

}  // namespace pd
