// Tensor-core decode kernel for 16-bit and FP8 KV caches (sm_103a).
//
// Work split: the attended pages of every segment (sequence, KV head, slice of <= 8
// query columns that share the KV head) lie on one cost line (each segment: a fixed
// set-up cost, then one unit per page), cut into W equal contiguous ranges, one per
// warp (W = blocks x 4).  Each warp is an independent
// worker: it walks the segments its range touches, streams their pages in order and
// finishes each segment on its own -- a segment it covers whole is written straight
// to out/lse; otherwise it leaves a partial state (normalised O, lse) in one of its two
// slots, and the worker that completes the segment's page count merges the slots
// (merge_state over S partials).  Apart from the start-up scan that finds each
// worker's first segment there is no block-wide barrier, so a worker switching
// segments or merging never stalls the other warps of its block.
//
// Every warp streams its 16-row tiles straight from HBM into registers with 16-byte
// loads (on GB300 this streams scattered 4 KB page blocks faster than staging them in
// shared memory with cp.async, which measured 19% slower on long contexts), and
// prefetches the K and V blocks of the next page into L2.  The loads are laid out so
// that the registers already are mma.sync fragments:
//   - S^T = K Q^T (m16n8k16, fp32 accumulate): A = the K tile (16 rows x 16 dims per
//     k-tile), B = Q^T with the <= 8 query columns of the slice as the n dimension:
//     the query heads of the KV group, or in the multi-query form (MQ) its (token,
//     head) pairs, each token t masked beyond its causal limit L - q_len + 1 + t.
//     A thread loads 16 contiguous bytes of its rows per chunk; the dot product's
//     k order is permuted to match, and Q's B fragments use the same permutation.
//   - online base-2 softmax on the accumulator fragments (TVM `batch_decode_paged_kv`:
//     running max m, sum d, output O), P^T rebuilt as a B fragment with 4 shuffles;
//   - O^T += V^T P^T: A = V^T built from 16-byte row loads with byte permutes.  The
//     output dims are permuted: m-tile mt row g_id (+8) holds dim 16 g_id + 2 mt (+1)
//     for FP8, 8 (g_id + 8 (mt >> 2)) + 2 (mt & 3) (+1) otherwise, so each thread ends
//     up with whole runs of 16 or 8 consecutive output dims (16-byte stores).
// The next tile's K loads are issued right after QK and its V loads right after PV,
// so each warp keeps about one tile in registers in flight while it computes.  The
// tile loop is kept nearly branch-free (its instruction fetch and branch stalls
// measurably limit it): the next piece comes from a per-lane cache by shuffles, the
// Q-packing mode is a compile-time parameter, and only partial tiles take a branch.
// RoPE (rotate-half pairs (d, d + D/2) or interleaved pairs (2i, 2i + 1)) is applied to
// K in registers before the MMA; rotated K is rounded once to f16 (11 significant bits;
// a score error of about 2^-12 of |q| |k| sqrt(D) scale) and multiplied with Q split
// into f16 hi + lo parts, one MMA per k-tile when the hi and lo parts share the n
// dimension (<= 4 columns).  The rotated K of a bf16 cache must stay inside the f16
// range (|k| < 46000).  A cache that holds K rotated at append time skips the K
// rotation (RoPE modes 3 and 4: Q only).  The frequency tables sit in shared memory
// padded against bank conflicts (rope_slot).  FP8 codes
// become f16 in registers (exact); k_scale folds into the score scale, v_scale into
// the output.
//
// Limits: head dim 64/128 for 16-bit KV, 128 for FP8; page size a multiple of 16, or 8
// (PAIR: two pages per 16-row tile).
#pragma once

#include <type_traits>

#include "decode_common.cuh"
#include "kernels.h"

namespace pd {

#ifndef PD_PREFETCH_PIECES
#define PD_PREFETCH_PIECES 1
#endif
constexpr int kPrefetchPieces = PD_PREFETCH_PIECES;  // L2 prefetch distance, in pages
#ifndef PD_QK_CHAINS
#define PD_QK_CHAINS 2
#endif
constexpr int kQChains = PD_QK_CHAINS;  // independent accumulators of a tile's K Q^T
constexpr float kLazyMax = 8.f;  // slack of the lazy running max (log2 units)
#ifndef PD_MIN_BLOCKS_PLAIN
#define PD_MIN_BLOCKS_PLAIN 1
#endif
#ifndef PD_MIN_BLOCKS_ROPE
#define PD_MIN_BLOCKS_ROPE 1
#endif
// Resident blocks per SM the register allocation targets.  The FP8 kernel moves half
// the bytes per tile of the 16-bit one, so it needs the extra warps of a third block
// to keep enough loads in flight (measured: 3 blocks of <= 168 registers beat 2 of
// 213 by ~15% on a 256-sequence FP8 cache).
template <bool ROPE, bool FP8>
struct MinBlocks {
  static constexpr int v = ROPE ? PD_MIN_BLOCKS_ROPE : FP8 ? 3 : PD_MIN_BLOCKS_PLAIN;
};

// ROPE: Q is rotated (its hi + lo split keeps the rotation exact); KROT: K is rotated
// in the kernel too (else the cache holds it rotated, or there is no RoPE).
template <typename KVT, typename QT, int D, bool ROPE, bool KROT = ROPE>
struct MmaTraits {
  static constexpr bool kFp8 = sizeof(KVT) == 1;
  using MT = typename std::conditional<std::is_same<KVT, __nv_bfloat16>::value, __nv_bfloat16,
                                       __half>::type;  // tensor-core input type
  static constexpr int kRowBytes = D * ElemBytes<KVT>::v;
  static constexpr int kKT = D / 16;             // k-tiles of QK, m-tiles of PV
  static constexpr int kKCh = kRowBytes / 64;    // 16-byte K chunks per row per thread
  static constexpr int kVCh = kRowBytes / 128;   // 16-byte V chunks per row per thread
  static constexpr bool kQSplit = ROPE || kFp8 || !std::is_same<QT, MT>::value;
  // QK tensor-core type: rotated K is rounded once to f16 (11-bit significand, against
  // bf16's 8), Q is split into f16 hi + lo, so a score keeps about 11 bits of K'
  using QKT = typename std::conditional<KROT, __half, MT>::type;
  static_assert(kRowBytes == 128 || kRowBytes == 256, "row must be 128 or 256 bytes");
};

// Slot of frequency f in the shared RoPE tables: two spare 8-byte words after every 16
// frequencies, so that the four quad lanes, which read frequencies 8 apart (rotate-half)
// or 4 apart (interleaved), hit different banks; slots stay even (16-byte reads of
// s_rot8 at an even f stay aligned).
__device__ __forceinline__ int rope_slot(int f) { return f + 2 * (f >> 4); }
constexpr int rope_slots(int D) { return D / 2 + 2 * (D / 32); }

// Dim of A-fragment element (k-tile kt, half 0: k-pos 2q..2q+1 / half 1: 2q+8..2q+9,
// element e) for thread quad index q4: thread q4 owns 16-byte chunks 4c + q4 of a row.
template <bool FP8>
__device__ __forceinline__ int frag_dim(int kt, int half, int e, int q4) {
  return FP8 ? 16 * (4 * (kt >> 2) + q4) + 4 * (kt & 3) + 2 * half + e
             : 8 * (4 * (kt >> 1) + q4) + 4 * (kt & 1) + 2 * half + e;
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ uint32_t comp(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Store a run of RL consecutive output dims of one (sequence, head) row.
template <int RL>
__device__ __forceinline__ void store_run(const DecodeParams& p, size_t idx, const float* v) {
  if (p.out_vec16) {
    if (p.out_dtype == kF32) {
      float4* o = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + idx);
#pragma unroll
      for (int i = 0; i < RL / 4; ++i) o[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    } else {
      uint4* o = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.out) + idx);
#pragma unroll
      for (int i = 0; i < RL / 8; ++i) {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          w[k] = p.out_dtype == kBF16 ? pack2<__nv_bfloat16>(v[8 * i + 2 * k], v[8 * i + 2 * k + 1])
                                      : pack2<__half>(v[8 * i + 2 * k], v[8 * i + 2 * k + 1]);
        o[i] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < RL; ++i) store_out(p, idx + i, v[i]);
  }
}

// Merge of every worker's partial state of one segment into out/lse, by one warp:
// lse = M + log2 sum_s 2^(lse_s - M), out = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M),
// over the workers s whose ranges hold the segment's units (cost-line positions
// seg_off + seg_c ... seg_off + seg_c + seg_n - 1; W workers on a line of U positions).
// HMAX bounds the heads of the slice (hcount), BATCH the slots whose partial rows are in
// flight together.  With at most 32 slots, lane s reads slot s's lse and the weights come
// from warp reductions; the first batch of partial rows is requested before that, so
// the merge costs about one L2 round trip per batch.  s_w: this warp's shared scratch
// of 34 x 8 floats, s_sl: 32 ints.
template <int D, int HMAX, int BATCH, bool MQ>
__device__ void warp_merge(const DecodeParams& p, int seg_b, long long seg_off, int seg_c, int seg_n,
                           long long U, long long W, int hk, int c0, int hcount,
                           float (*s_w)[kMaxGroupPerCta], int* s_sl, int zg, int zw) {
  constexpr int G8 = kMaxGroupPerCta;
  constexpr int D4 = D / 4;
  constexpr int kV = (HMAX * D4 + 31) / 32;  // float4 outputs per lane
  static_assert(HMAX % 4 == 0 && HMAX <= G8, "HMAX");
  const int lane = threadIdx.x & 31;
  const long long w0 = share_of(seg_off + seg_c, U, W);
  const int ns = (int)(share_of(seg_off + seg_c + seg_n - 1, U, W) - w0 + 1);
  // line worker w's slot for this slice: worker w * zg + zw (zg = 1: w itself)
  const long long sl0 = share_slot_z(w0, seg_off, U, W, zg, zw);  // worker w0 always holds units
  float* s_M = s_w[32];
  float* s_den = s_w[33];
  float4 acc[kV];
#pragma unroll
  for (int e = 0; e < kV; ++e) acc[e] = make_float4(0.f, 0.f, 0.f, 0.f);
  auto load_rows = [&](float4 (&o)[BATCH][kV], int i0, int cnt) {
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const float* po = p.part_o + (size_t)s_sl[min(i0 + u, cnt - 1)] * D;
#pragma unroll
      for (int e = 0; e < kV; ++e) {
        const int vi = lane + 32 * e;
        o[u][e] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (vi < hcount * D4) o[u][e] = __ldcg(reinterpret_cast<const float4*>(po + (size_t)(vi / D4) * D) + vi % D4);
      }
    }
  };
  auto add_rows = [&](const float4 (&o)[BATCH][kV], int i0, int cnt) {
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      if (i0 + u < cnt) {
#pragma unroll
        for (int e = 0; e < kV; ++e) {
          const int vi = lane + 32 * e;
          if (vi < hcount * D4) {
            const float w = s_w[i0 + u][vi / D4];
            acc[e].x += w * o[u][e].x;
            acc[e].y += w * o[u][e].y;
            acc[e].z += w * o[u][e].z;
            acc[e].w += w * o[u][e].w;
          }
        }
      }
    }
  };
  if (ns <= 32) {
    long long sl = -1;
    float v[HMAX];
#pragma unroll
    for (int j = 0; j < HMAX; ++j) v[j] = kEmptyM;
    if (lane < ns) {
      sl = share_slot_z(w0 + lane, seg_off, U, W, zg, zw);
      if (sl >= 0) {
#pragma unroll
        for (int q = 0; q < HMAX / 4; ++q) {
          const float4 a = __ldcg(reinterpret_cast<const float4*>(p.part_lse + sl) + q);
          v[4 * q] = a.x;
          v[4 * q + 1] = a.y;
          v[4 * q + 2] = a.z;
          v[4 * q + 3] = a.w;
        }
      }
    }
    s_sl[lane] = (int)(sl >= 0 ? sl : sl0);  // a worker with no units: weight 0, a written slot
    __syncwarp();
    float4 o[BATCH][kV];
    load_rows(o, 0, ns);  // independent of the weights: in flight during the reductions
#pragma unroll
    for (int j = 0; j < HMAX; ++j) {
      const bool ok = sl >= 0 && j < hcount;
      float M = ok ? v[j] : kEmptyM;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
      const float w = ok ? merge_exp2(p, v[j] - M) : 0.f;
      float den = w;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
      s_w[lane][j] = den > 0.f ? w / den : 0.f;  // normalised weight of slot `lane`
      if (lane == 0) {
        s_M[j] = M;
        s_den[j] = den;
      }
    }
    __syncwarp();
    add_rows(o, 0, ns);
    for (int i0 = BATCH; i0 < ns; i0 += BATCH) {
      load_rows(o, i0, ns);
      add_rows(o, i0, ns);
    }
  } else {
    // more than 32 slots: per-head maximum, then weights chunk by chunk (unnormalised)
    float M[HMAX], den[HMAX];
#pragma unroll
    for (int j = 0; j < HMAX; ++j) {
      M[j] = kEmptyM;
      den[j] = 0.f;
    }
    for (int s = lane; s < ns; s += 32) {
      const long long sl = share_slot_z(w0 + s, seg_off, U, W, zg, zw);
      if (sl < 0) continue;
#pragma unroll
      for (int j = 0; j < HMAX; ++j) M[j] = fmaxf(M[j], j < hcount ? __ldcg(p.part_lse + sl + j) : kEmptyM);
    }
#pragma unroll
    for (int j = 0; j < HMAX; ++j)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) M[j] = fmaxf(M[j], __shfl_xor_sync(0xffffffffu, M[j], off));
    for (int base = 0; base < ns; base += 32) {
      const int s = base + lane;
      const long long sl = s < ns ? share_slot_z(w0 + s, seg_off, U, W, zg, zw) : -1;
#pragma unroll
      for (int j = 0; j < HMAX; ++j) {
        const float w = (sl >= 0 && j < hcount) ? merge_exp2(p, __ldcg(p.part_lse + sl + j) - M[j]) : 0.f;
        den[j] += w;
        s_w[lane][j] = w;
      }
      s_sl[lane] = (int)(sl >= 0 ? sl : sl0);
      __syncwarp();
      const int cnt = min(32, ns - base);
      float4 o[BATCH][kV];
      for (int i0 = 0; i0 < cnt; i0 += BATCH) {
        load_rows(o, i0, cnt);
        add_rows(o, i0, cnt);
      }
      __syncwarp();
    }
#pragma unroll
    for (int j = 0; j < HMAX; ++j)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) den[j] += __shfl_xor_sync(0xffffffffu, den[j], off);
    if (lane == 0) {
#pragma unroll
      for (int j = 0; j < HMAX; ++j) {
        s_M[j] = M[j];
        s_den[j] = den[j];
      }
    }
    __syncwarp();
#pragma unroll
    for (int e = 0; e < kV; ++e) {  // weights were not normalised on this path
      const int vi = lane + 32 * e;
      if (vi < hcount * D4) {
        const float dj = s_den[vi / D4];
        const float r = dj > 0.f ? 1.f / dj : 0.f;
        acc[e].x *= r;
        acc[e].y *= r;
        acc[e].z *= r;
        acc[e].w *= r;
      }
    }
  }
  // per column: output scale and final lse (with the head's sink, if any), by lane j
  __syncwarp();
  if (lane < hcount) {
    const float Mj = s_M[lane], dj = s_den[lane];
    const bool empty = !(Mj > kEmptyM);
    float sc = empty ? 0.f : p.out_scale;
    float l = empty ? kEmptyM : Mj + log2f(dj);
    if (p.sink) {
      const SinkAdj sa = apply_sink(p, col_head<MQ>(p, hk, c0 + lane), l);
      sc *= sa.scale;
      l = sa.lse;
    }
    s_w[0][lane] = sc;  // the weight rows are free again
    s_w[1][lane] = l;
  }
  __syncwarp();
#pragma unroll
  for (int e = 0; e < kV; ++e) {
    const int vi = lane + 32 * e;
    if (vi < hcount * D4) {
      const int j = vi / D4, d4 = vi % D4;
      const float sc = s_w[0][j];
      const size_t row = col_row<MQ>(p, seg_b, hk, c0 + j);
      const size_t o = row * D + 4 * d4;
      store_out(p, o + 0, acc[e].x * sc);
      store_out(p, o + 1, acc[e].y * sc);
      store_out(p, o + 2, acc[e].z * sc);
      store_out(p, o + 3, acc[e].w * sc);
      if (d4 == 0) p.lse[row] = s_w[1][j];
    }
  }
  __syncwarp();
}

// RM: 0 no RoPE; 1 rotate-half, 2 interleaved pairs (Q and K rotated here); 3, 4 the same
// layouts with K rotated in the cache already (only Q rotated here).
// PAIR: pages of 8 rows; a 16-row tile takes two consecutive pages (rows 0-7 from the
// first, rows 8-15 from the second) when their attended rows follow each other, else one.
template <typename KVT, typename QT, int D, int RM, int NW, bool MQ, bool PAIR = false>
__global__ void __launch_bounds__(NW * 32, MinBlocks<(RM == 1 || RM == 2), (sizeof(KVT) == 1)>::v)
    decode_mma_kernel(const __grid_constant__ DecodeParams p) {
  constexpr bool ROPE = RM != 0;               // Q is rotated
  constexpr bool KROT = RM == 1 || RM == 2;    // K is rotated in the tile loop
  constexpr bool IL = RM == 2 || RM == 4;      // interleaved pairs (2i, 2i + 1)
  using Tr = MmaTraits<KVT, QT, D, ROPE, KROT>;
  using MT = typename Tr::MT;
  using QKT = typename Tr::QKT;
  constexpr int NT = NW * 32;
  constexpr int KT = Tr::kKT;
  constexpr int RB = Tr::kRowBytes;
  constexpr int KCH = Tr::kKCh;
  constexpr int VCH = Tr::kVCh;
  constexpr bool FP8 = Tr::kFp8;
  constexpr int RL = FP8 ? 16 : 8;  // output run: consecutive dims a thread holds
  constexpr int NR = 2 * KT / RL;   // runs per head and thread
  __shared__ uint4 s_qf[NW][KT][32];                        // per-warp Q^T B fragments
  __shared__ int s_units[kStartCacheB];                     // start-up scan scratch
  __shared__ float s_mw[NW][34][kMaxGroupPerCta];           // per-warp merge scratch
  __shared__ int s_msl[NW][32];
  __shared__ long long s_pend[NW][2][4];                    // per-warp deferred merges
  __shared__ unsigned long long s_ropeF[ROPE ? rope_slots(D) : 1];  // frequencies (fixed point)
  __shared__ __align__(16) float2 s_rot8[KROT ? rope_slots(D) : 2];  // e^(i * 8 * omega_f)
  __shared__ WorkerStart s_start[NW];

  // Q and the page table are small and needed right after the start-up scan, when the
  // first tiles of every worker flood HBM: each block prefetches its share into L2 now
  if (threadIdx.x == 0) {
    prefetch_l2_share(p.Q, (size_t)p.B * p.q_len * p.H_qo * D * sizeof(QT), blockIdx.x, gridDim.x);
    if (p.values) prefetch_l2_share(p.values, (size_t)p.nnz_pages * sizeof(int32_t), blockIdx.x, gridDim.x);
  }
  if (ROPE) {
    for (int i = threadIdx.x; i < D / 2; i += NT) {
      const unsigned long long F = p.rope_F[i];
      s_ropeF[rope_slot(i)] = F;
      if (KROT) {
        float c8, s8;
        rope_cos_sin(8, F, c8, s8);
        s_rot8[rope_slot(i)] = make_float2(c8, s8);
      }
    }
  }
  // By default nothing of the caller's is read before the kernel launched before this
  // one on the stream has completed; with early_inputs the scan, the page table and Q
  // are read while it finishes, and only the first page read (or write) waits.
  if (!p.early_inputs) {
    pdl_wait();
    pdl_release();
  }
  worker_starts<NT, NW>(p, s_start, s_units);  // the last block-wide barrier of the kernel

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g_id = lane >> 2, q4 = lane & 3;
  const WorkerStart ws = s_start[warp];
  if (ws.b < 0) return;  // no units for this worker

  const int P = p.P;
  const uint8_t* kv_base = reinterpret_cast<const uint8_t*>(p.pages);
  const size_t block_bytes = (size_t)P * RB;          // one (page, K|V, head) block
  const size_t v_off = (size_t)p.H_kv * block_bytes;  // K block -> V block
  // line workers (grouped slices: zg adjacent warps share one) and this warp's slice
  const int zg = p.mode == kSchedBalanced ? p.zg : 1;
  const long long Wn = (long long)gridDim.x * NW / zg;
  const long long wid = (long long)blockIdx.x * NW + warp;

  Segment sg;
  sg.b = ws.b;
  sg.hz = ws.hz;
  sg.off = ws.off;
  sg.seq = load_seq(p, sg.b);
  sg.n = units_of(sg.seq, P);
  // cost-line positions: a segment spans [off, off + C + n), its units from off + C
  const int C = p.mode == kSchedBalanced ? p.seg_cost : 0;
  const long long cx1 = p.mode == kSchedBalanced ? ws.x1 : sg.off + sg.n;

  int npend = 0;  // next free entry of s_pend[warp] (entries with b < 0 are unused)
  if (lane < 2) s_pend[warp][lane][0] = -1;
  __syncwarp();

  // The worker walks the segments (sequence, head slice) its range [x0, x1) touches.
  for (;;) {
  const int ua = (int)min(max(ws.x0 - sg.off - C, 0ll), (long long)sg.n);
  const int ub = (int)min(max(cx1 - sg.off - C, 0ll), (long long)sg.n);
  if (ua < ub) {  // else only the segment's set-up positions fall in this range
  const int hk = sg.hz / p.n_z, z = sg.hz - (sg.hz / p.n_z) * p.n_z;
  const Pieces pcs = make_pieces(0, sg.seq.L, sg.seq, P);
  const int pend = min(ub, sg.seq.L > 0 ? pcs.count() : 0);  // pieces [ua, pend) here
  const int c0 = z * kMaxGroupPerCta;                      // first query column of the slice
  const int hcount = min(kMaxGroupPerCta, p.ncol - c0);  // its columns (heads x tokens)

  // Raw Q of this lane's B-fragment elements (pairs of adjacent dims), loaded first:
  // they are tiny and needed before anything else.
  // Split-operand slices of at most 4 columns pack Q's lo part into the unused MMA
  // columns 4..7 (lane group g_id >= 4 builds column g_id - 4's lo fragment): K Q^T then
  // takes one MMA per k-tile instead of two, and column h + 4 is folded into column h.
  const bool pack4 = Tr::kQSplit && hcount <= 4;
  const int qh = pack4 ? (g_id & 3) : g_id;  // the column this lane's B fragment holds
  const bool have_q = qh < hcount;
  // The lane's Q elements (dims frag_dim(kt, h, e, q4)) form KT/2 contiguous 16-byte
  // chunks, loaded with one vector load each: chunk c starts at element 8 (4c + q4)
  // (16-bit KV) or 16 (4 (c >> 1) + q4) + 8 (c & 1) (FP8 KV).
  constexpr int QCH = KT / 2;
  uint4 qchunk[QCH];
  {
    const QT* qrow = reinterpret_cast<const QT*>(p.Q) + col_row<MQ>(p, sg.b, hk, c0 + (have_q ? qh : 0)) * D;
#pragma unroll
    for (int c = 0; c < QCH; ++c) {
      const int e0 = FP8 ? 16 * (4 * (c >> 1) + q4) + 8 * (c & 1) : 8 * (4 * c + q4);
      qchunk[c] = have_q ? __ldg(reinterpret_cast<const uint4*>(qrow + e0)) : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  // the pair of Q elements (kt, h, e = 0..1) of this lane's B fragment
  auto qraw = [&](int kt, int h) -> uint32_t {
    return FP8 ? comp(qchunk[2 * (kt >> 2) + ((kt & 3) >> 1)], 2 * (kt & 1) + h)
               : comp(qchunk[kt >> 1], 2 * (kt & 1) + h);
  };
  // query position: q_rope_position[b], plus the token index of this lane's column
  const int qpos = ROPE ? __ldg(p.q_rope_position + sg.b) + (MQ ? (c0 + qh) / p.group : 0) : 0;
  // multi-query: attended-row limits of this lane's two score columns (token t sees rows
  // r < L - q_len + 1 + t; packed slices keep columns 0..3, folded into lanes q4 and q4^2)
  int lim0 = 0, lim1 = 0;
  if constexpr (MQ) {
    const int cc = c0 + (pack4 ? 2 * (q4 & 1) : 2 * q4);
    lim0 = sg.seq.L - p.q_len + 1 + cc / p.group;
    lim1 = sg.seq.L - p.q_len + 1 + (cc + 1) / p.group;
  }
  const int kpos0 = KROT ? __ldg(p.k_rope_pos_offset + sg.b) : 0;

  // ---------------------------------------------------------------- tile stream
  // Pieces [ua, pend) in order.  Entering a piece, the warp prefetches the K and V
  // blocks of the piece kPrefetchPieces ahead into L2, so that the register loads of a
  // tile mostly hit L2 and each warp keeps more than one page in flight without
  // spending registers on it.
  struct Tile {
    int piece, t, s_lo, s_hi, r_lo;
    const uint8_t* kblk;  // K block of (page, hk); nullptr = no more tiles
    // PAIR: the second page's K block (rows 8-15; nullptr: none) and its slot range
    const uint8_t* kblk2;
    int s_lo2, s_hi2;
  };
  // This warp's pieces come 32 at a time: lane i holds piece base + i (its physical
  // page or -1, its slot range, its first row), handed out with shuffles, so moving to
  // the next piece costs a few shuffles and one (warp-uniform) branch.
  int pb_base = -64, pb_page = -1, pb_slots = 0, pb_row = 0;
  auto load_batch = [&](int j) {
    pb_base = j;
    const int jj = j + lane;
    pb_page = -1;
    if (jj < pend) {
      const Piece pc = get_piece(pcs, jj, P);
      pb_page = lookup_page(p, sg.seq, pc.page_idx);  // -1 (error recorded) if out of range
      pb_slots = pc.s_lo | (pc.s_hi << 16);            // s_hi <= P <= 256
      pb_row = pc.r_lo;
    }
  };
  auto kblock = [&](int pg) { return kv_base + (((size_t)pg * 2) * p.H_kv + hk) * block_bytes; };
  auto prefetch_piece = [&](int j) {  // K and V blocks of piece j into L2 (if in this batch)
    if (j < pend && j < pb_base + 32) {
      const int pg = __shfl_sync(0xffffffffu, pb_page, j - pb_base);
      if (pg >= 0 && lane == 0) {
        prefetch_l2_bulk(kblock(pg), (uint32_t)block_bytes);
        prefetch_l2_bulk(kblock(pg) + v_off, (uint32_t)block_bytes);
      }
    }
  };
  auto first_tile_from = [&](int j) -> Tile {  // first tile of piece j or later
    Tile tl;
    tl.kblk = nullptr;  // no more tiles (the other fields stay defined)
    tl.kblk2 = nullptr;
    tl.piece = pend;
    tl.t = tl.s_lo = tl.s_hi = tl.r_lo = tl.s_lo2 = tl.s_hi2 = 0;
    for (; j < pend; ++j) {
      if (j >= pb_base + 32) load_batch(j);
      const int src = j - pb_base;
      const int pg = __shfl_sync(0xffffffffu, pb_page, src);
      if (pg < 0) continue;  // bad page id: its rows are skipped (error already recorded)
      const int sl = __shfl_sync(0xffffffffu, pb_slots, src);
      tl.piece = j;
      tl.s_lo = sl & 0xffff;
      tl.s_hi = sl >> 16;
      tl.t = tl.s_lo >> 4;
      tl.r_lo = __shfl_sync(0xffffffffu, pb_row, src);
      tl.kblk = kblock(pg);
      if constexpr (PAIR) {
        // the next piece joins as rows 8-15 when it is in this batch, has a valid page
        // and its attended rows continue this page's (row 8 + s of the tile = its slot s)
        const int j2 = j + 1, src2 = min(j2 - pb_base, 31);
        const int pg2 = __shfl_sync(0xffffffffu, pb_page, src2);
        const int sl2 = __shfl_sync(0xffffffffu, pb_slots, src2);
        const int rl2 = __shfl_sync(0xffffffffu, pb_row, src2);
        if (j2 < pend && j2 - pb_base < 32 && pg2 >= 0 &&
            rl2 - (sl2 & 0xffff) == tl.r_lo - tl.s_lo + 8) {
          tl.kblk2 = kblock(pg2);
          tl.s_lo2 = sl2 & 0xffff;
          tl.s_hi2 = sl2 >> 16;
          tl.piece = j2;  // the tile ends with piece j2
        }
      }
      break;
    }
    return tl;
  };
  // Common cases without a branch: the next tile of the same piece, or the first tile of
  // the next piece when it is in the current batch and has a valid page; anything else
  // (a batch reload, a bad page id, the end) takes the slow path.
  auto next_tile = [&](const Tile& c) -> Tile {
    if constexpr (PAIR) return first_tile_from(c.piece + 1);
    const bool same = (c.t + 1) * 16 < c.s_hi;
    const int j = c.piece + 1;
    const int src = min(max(j - pb_base, 0), 31);
    const int pg = __shfl_sync(0xffffffffu, pb_page, src);
    const int sl = __shfl_sync(0xffffffffu, pb_slots, src);
    const int rl = __shfl_sync(0xffffffffu, pb_row, src);
    const bool fast = same || (j < pend && j - pb_base < 32 && pg >= 0);
    if (!fast) return first_tile_from(j);
    Tile n;
    n.piece = same ? c.piece : j;
    n.s_lo = same ? c.s_lo : (sl & 0xffff);
    n.s_hi = same ? c.s_hi : (sl >> 16);
    n.t = same ? c.t + 1 : ((sl & 0xffff) >> 4);
    n.r_lo = same ? c.r_lo : rl;
    n.kblk = same ? c.kblk : kblock(pg);
    n.kblk2 = nullptr;
    n.s_lo2 = n.s_hi2 = 0;
    return n;
  };
  uint4 kr[2][KCH];      // K rows t*16 + g_id (+8): chunks 4c + q4
  uint4 vr[4][VCH];      // V rows t*16 + 2q4, +1, +8, +9: chunks g_id + 8j
  // PAIR: rows 8-15 come from the tile's second page, at slots 0-7, or are zero (no second
  // page); the softmax and P.V masks drop them then.
  auto load_k = [&](const Tile& c) {
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int row_in_page = PAIR ? g_id : c.t * 16 + g_id + 8 * rr;
      const uint8_t* blk = PAIR && rr ? c.kblk2 : c.kblk;
      const bool ok = !PAIR || rr == 0 || c.kblk2 != nullptr;
      const uint8_t* row = blk + (size_t)row_in_page * RB;
#pragma unroll
      for (int ch = 0; ch < KCH; ++ch)
        kr[rr][ch] = ok ? ldg_stream(row + (4 * ch + q4) * 16) : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  auto load_v = [&](const Tile& c) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row_in_page = PAIR ? 2 * q4 + (i & 1) : c.t * 16 + 2 * q4 + (i & 1) + 8 * (i >> 1);
      const uint8_t* blk = PAIR && (i >> 1) ? c.kblk2 : c.kblk;
      const bool ok = !PAIR || (i >> 1) == 0 || c.kblk2 != nullptr;
      const uint8_t* row = blk + v_off + (size_t)row_in_page * RB;
#pragma unroll
      for (int j = 0; j < VCH; ++j)
        vr[i][j] = ok ? ldg_stream(row + (g_id + 8 * j) * 16) : make_uint4(0u, 0u, 0u, 0u);
    }
  };

  // first tile's loads go out before the Q set-up, which then overlaps their latency
  Tile cur = first_tile_from(ua);
  if (p.early_inputs) {  // pages may still be written by the previous kernel until here
    // the first tile's blocks can come into L2 meanwhile: L2 is where the previous
    // kernel's writes land, so a line fetched now still sees them
    if (cur.kblk && lane == 0) {
      prefetch_l2_bulk(cur.kblk, (uint32_t)block_bytes);
      prefetch_l2_bulk(cur.kblk + v_off, (uint32_t)block_bytes);
    }
    pdl_wait();
    pdl_release();
  }
  if (cur.kblk) {
    load_k(cur);
    load_v(cur);
  }

  // ---------------------------------------------------------------- Q^T B fragments
  // Per k-tile and lane: {hi b0, hi b1, lo b0, lo b1} with b0 = (k 2q..2q+1, head g_id),
  // b1 = (k 2q+8..2q+9, head g_id) in the permuted dim order, in this warp's shared
  // memory (k-tile pairs kt / kt + KT/2 together, for RoPE).
  {
#pragma unroll
    for (int kt = 0; kt < KT / 2; ++kt) {
      float qv[2][2][2];  // [pair member u: kt, kt + KT/2][half][e]
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float2 f = unpack2<QT>(qraw(kt + u * (KT / 2), h));
          qv[u][h][0] = f.x;
          qv[u][h][1] = f.y;
        }
      if (ROPE && !IL) {  // rotate-half: dims d (k-tile kt) and d + D/2 (kt + KT/2)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float c, sn;
            rope_cos_sin(qpos, s_ropeF[rope_slot(frag_dim<FP8>(kt, h, e, q4))], c, sn);
            const float x = qv[0][h][e], y = qv[1][h][e];
            qv[0][h][e] = x * c - y * sn;
            qv[1][h][e] = y * c + x * sn;
          }
      }
      if (IL) {  // interleaved: the element pair (2i, 2i + 1) of a fragment, frequency i
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float c, sn;
            rope_cos_sin(qpos, s_ropeF[rope_slot(frag_dim<FP8>(kt + u * (KT / 2), h, 0, q4) >> 1)], c, sn);
            const float x = qv[u][h][0], y = qv[u][h][1];
            qv[u][h][0] = x * c - y * sn;
            qv[u][h][1] = y * c + x * sn;
          }
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        uint32_t hi[2], lo[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (Tr::kQSplit) {
            split2<QKT>(qv[u][h][0] * p.q_prescale, qv[u][h][1] * p.q_prescale, hi[h], lo[h]);
          } else {
            hi[h] = pack2<QKT>(qv[u][h][0], qv[u][h][1]);
            lo[h] = 0u;
          }
        }
        s_qf[warp][kt + u * (KT / 2)][lane] =
            !pack4 ? make_uint4(hi[0], hi[1], lo[0], lo[1])
                   : (g_id < 4 ? make_uint4(hi[0], hi[1], 0u, 0u) : make_uint4(lo[0], lo[1], 0u, 0u));
      }
    }
  }
  __syncwarp();
  // The next page's L2 prefetch goes out only now: issued with the first tile's loads,
  // at the start of a segment, it crowded them and the Q loads (the RoPE Q build
  // waited longer; llama3 68.0 -> 64.6 us).
  if (cur.kblk) prefetch_piece(cur.piece + kPrefetchPieces);
  const float post_scale = Tr::kQSplit ? 1.f : p.score_scale;

  float st_m[2] = {kEmptyM, kEmptyM}, st_d[2] = {0.f, 0.f};
  float oacc[KT][4];
#pragma unroll
  for (int i = 0; i < KT; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;

  // The tile loop, instantiated with the Q packing decided at compile time (it is
  // fixed for a segment; a runtime test inside the unrolled QK costs branches per tile).
  auto tile_loop = [&](auto pack_tag) {
    constexpr bool PK = decltype(pack_tag)::value;
  while (cur.kblk) {
      const Tile nxt = next_tile(cur);
      const int slot0 = cur.t * 16 + g_id, slot1 = slot0 + 8;
      const bool v0 = slot0 >= cur.s_lo && slot0 < cur.s_hi;
      const bool v1 = PAIR ? (cur.kblk2 != nullptr && g_id >= cur.s_lo2 && g_id < cur.s_hi2)
                           : (slot1 >= cur.s_lo && slot1 < cur.s_hi);
      // ------------------------------------------------------------ S^T = K Q^T
      // independent accumulators shorten the dependent MMA chain; summed after
      // spread over kQChains independent accumulators: the products of one tile would
      // otherwise form long chains of dependent MMAs (mma.sync latency, not throughput,
      // bounds the tile loop)
      float qacc[kQChains][4];
#pragma unroll
      for (int c = 0; c < kQChains; ++c) qacc[c][0] = qacc[c][1] = qacc[c][2] = qacc[c][3] = 0.f;
      if constexpr (!KROT) {
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
          const uint4 qf = s_qf[warp][kt][lane];
          Mma<MT>::run(qacc[(2 * kt) % kQChains], a, qf.x, qf.y);
          if (Tr::kQSplit && !PK) Mma<MT>::run(qacc[(2 * kt + 1) % kQChains], a, qf.z, qf.w);
        }
      } else if constexpr (IL) {
        // interleaved RoPE on K in registers: each A-fragment register holds the pair
        // (2i, 2i + 1) of one row, rotated by frequency i; rows g_id and g_id + 8 (8
        // positions further) go through the rotation together as an fp32x2 pair
        const int pos0 = kpos0 + cur.r_lo + (slot0 - cur.s_lo);
#pragma unroll
        for (int kt = 0; kt < KT; ++kt) {
          uint32_t araw[4];
          if constexpr (FP8) {
            const uint32_t r0w = comp(kr[0][kt >> 2], kt & 3), r1w = comp(kr[1][kt >> 2], kt & 3);
            araw[0] = e4m3x2_to_f16x2((uint16_t)(r0w & 0xffff));
            araw[2] = e4m3x2_to_f16x2((uint16_t)(r0w >> 16));
            araw[1] = e4m3x2_to_f16x2((uint16_t)(r1w & 0xffff));
            araw[3] = e4m3x2_to_f16x2((uint16_t)(r1w >> 16));
          } else {
            araw[0] = comp(kr[0][kt >> 1], 2 * (kt & 1));
            araw[2] = comp(kr[0][kt >> 1], 2 * (kt & 1) + 1);
            araw[1] = comp(kr[1][kt >> 1], 2 * (kt & 1));
            araw[3] = comp(kr[1][kt >> 1], 2 * (kt & 1) + 1);
          }
          uint32_t ar[4];
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int f = frag_dim<FP8>(kt, half, 0, q4) >> 1;
            float c0, s0;
            rope_cos_sin(pos0, s_ropeF[rope_slot(f)], c0, s0);
            const float2 r8 = s_rot8[rope_slot(f)];  // (cos, sin) of 8 positions
            const float2 cc = make_float2(c0, c0 * r8.x - s0 * r8.y);
            const float2 ss = make_float2(s0, s0 * r8.x + c0 * r8.y);
            const float2 a0 = unpack2<MT>(araw[2 * half]);      // row g_id: (2i, 2i + 1)
            const float2 a1 = unpack2<MT>(araw[2 * half + 1]);  // row g_id + 8
            const float2 x = make_float2(a0.x, a1.x), y = make_float2(a0.y, a1.y);
            const float2 xr = sub_f2(mul_f2(x, cc), mul_f2(y, ss));
            const float2 yr = fma_f2(y, cc, mul_f2(x, ss));
            ar[2 * half] = pack2<QKT>(xr.x, yr.x);
            ar[2 * half + 1] = pack2<QKT>(xr.y, yr.y);
          }
          const uint4 qf = s_qf[warp][kt][lane];
          Mma<QKT>::run(qacc[kt % kQChains], ar, qf.x, qf.y);
          if (!PK) Mma<QKT>::run(qacc[(kt + 1) % kQChains], ar, qf.z, qf.w);
        }
      } else {
        // RoPE on K in registers: k-tiles kt and kt + KT/2 hold dims d and d + D/2
        const int pos0 = kpos0 + cur.r_lo + (slot0 - cur.s_lo);  // row g_id; row g_id + 8 is pos0 + 8
        // rotate, round and multiply the k-tile pair (kt, kt + KT/2) given its raw fragments
        auto rope_pair = [&](int kt, const uint32_t (&araw)[2][4]) {
          uint32_t ar[2][4];  // rotated K of k-tiles kt, kt + KT/2 (f16)
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            // (cos, sin) of this half's two frequencies f, f + 1 (packed fp32 pairs) at
            // rows g_id (direct) and g_id + 8 (rotated by 8 positions)
            const int f = frag_dim<FP8>(kt, half, 0, q4);
            float2 cs_c[2], cs_s[2];  // [row] (cos f, cos f+1), (sin f, sin f+1)
            rope_cos_sin(pos0, s_ropeF[rope_slot(f)], cs_c[0].x, cs_s[0].x);
            rope_cos_sin(pos0, s_ropeF[rope_slot(f) + 1], cs_c[0].y, cs_s[0].y);
            const float4 r8 = *reinterpret_cast<const float4*>(&s_rot8[rope_slot(f)]);  // (c8, s8) of f, f+1
            const float2 r8c = make_float2(r8.x, r8.z), r8s = make_float2(r8.y, r8.w);
            cs_c[1] = sub_f2(mul_f2(cs_c[0], r8c), mul_f2(cs_s[0], r8s));
            cs_s[1] = fma_f2(cs_s[0], r8c, mul_f2(cs_c[0], r8s));
#pragma unroll
            for (int row = 0; row < 2; ++row) {
              const int ai = 2 * half + row;
              const float2 x = unpack2<MT>(araw[0][ai]);
              const float2 y = unpack2<MT>(araw[1][ai]);
              const float2 xr = sub_f2(mul_f2(x, cs_c[row]), mul_f2(y, cs_s[row]));
              const float2 yr = fma_f2(y, cs_c[row], mul_f2(x, cs_s[row]));
              ar[0][ai] = pack2<QKT>(xr.x, xr.y);
              ar[1][ai] = pack2<QKT>(yr.x, yr.y);
            }
          }
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const uint4 qf = s_qf[warp][kt + u * (KT / 2)][lane];
            Mma<QKT>::run(qacc[(2 * u + kt) % kQChains], ar[u], qf.x, qf.y);
            if (!PK) Mma<QKT>::run(qacc[(2 * u + kt + 1) % kQChains], ar[u], qf.z, qf.w);
          }
        };
        {
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
            rope_pair(kt, araw);
          }
        }
      }
      float acc[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[i] = qacc[0][i];
#pragma unroll
        for (int c = 1; c < kQChains; ++c) acc[i] += qacc[c][i];
      }
      if (PK) {  // score(h) = column h + column h + 4 (held two lanes over)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], 2);
      }
      // K registers are free: start the next tile's K loads (after the last tile: this
      // tile's block again, never used)
      const Tile& ntile = nxt.kblk ? nxt : cur;
      load_k(ntile);
      // ------------------------------------------------------------ online softmax (log2)
      float sc[4];
      sc[0] = v0 ? acc[0] * post_scale : -INFINITY;  // row g_id, heads 2q, 2q+1
      sc[1] = v0 ? acc[1] * post_scale : -INFINITY;
      sc[2] = v1 ? acc[2] * post_scale : -INFINITY;  // row g_id + 8
      sc[3] = v1 ? acc[3] * post_scale : -INFINITY;
      if constexpr (MQ) {  // causal among the new tokens
        const int r0 = cur.r_lo + (slot0 - cur.s_lo);  // attended index of row g_id
        if (r0 >= lim0) sc[0] = -INFINITY;
        if (r0 >= lim1) sc[1] = -INFINITY;
        if (r0 + 8 >= lim0) sc[2] = -INFINITY;
        if (r0 + 8 >= lim1) sc[3] = -INFINITY;
      }
      // Lazy running max: the reference max m moves only when some score exceeds it by
      // more than kLazyMax (log2 units; a warp vote), so the tile max reduction and the
      // rescale of O and d run on the first tile and then rarely.  Probabilities stay
      // <= 2^kLazyMax, and out = O/d, lse = m + log2 d are exact for any reference m.
      {
        const float over = fmaxf(fmaxf(sc[0], sc[2]) - st_m[0], fmaxf(sc[1], sc[3]) - st_m[1]);
        if (__any_sync(0xffffffffu, over > kLazyMax)) {
          const float tm0 = max_over_groups(fmaxf(sc[0], sc[2]));
          const float tm1 = max_over_groups(fmaxf(sc[1], sc[3]));
          const float mn0 = fmaxf(st_m[0], tm0), mn1 = fmaxf(st_m[1], tm1);
          const float al0 = fast_exp2(st_m[0] - mn0), al1 = fast_exp2(st_m[1] - mn1);
          st_d[0] *= al0;
          st_d[1] *= al1;
          st_m[0] = mn0;
          st_m[1] = mn1;
#pragma unroll
          for (int mt = 0; mt < KT; ++mt) {
            oacc[mt][0] *= al0;
            oacc[mt][1] *= al1;
            oacc[mt][2] *= al0;
            oacc[mt][3] *= al1;
          }
        }
      }
      float pr[4];
      pr[0] = fast_exp2(sc[0] - st_m[0]);
      pr[1] = fast_exp2(sc[1] - st_m[1]);
      pr[2] = fast_exp2(sc[2] - st_m[0]);
      pr[3] = fast_exp2(sc[3] - st_m[1]);
      st_d[0] += pr[0] + pr[2];
      st_d[1] += pr[1] + pr[3];
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
      // rows outside the piece may hold anything (even NaN): in a partial tile (the first
      // or last of a piece; warp-uniform test) this thread's V rows 2q, 2q+1, 2q+8, 2q+9
      // that fall outside are zeroed in the registers, so full tiles need no masking
      if constexpr (PAIR) {  // rows 0-7: the first page's slots; rows 8-15: the second's
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = 2 * q4 + (i & 1);
          const bool ok = (i >> 1) ? (cur.kblk2 != nullptr && r >= cur.s_lo2 && r < cur.s_hi2)
                                   : (r >= cur.s_lo && r < cur.s_hi);
          if (!ok) {
#pragma unroll
            for (int j = 0; j < VCH; ++j) vr[i][j] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
      } else if (cur.t * 16 < cur.s_lo || cur.t * 16 + 16 > cur.s_hi) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = cur.t * 16 + 2 * q4 + (i & 1) + 8 * (i >> 1);
          if (r < cur.s_lo || r >= cur.s_hi) {
#pragma unroll
            for (int j = 0; j < VCH; ++j) vr[i][j] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
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
          a[0] = e4m3x2_to_f16x2((uint16_t)(xy01 & 0xffff));
          a[1] = e4m3x2_to_f16x2((uint16_t)(xy01 >> 16));
          a[2] = e4m3x2_to_f16x2((uint16_t)(xy23 & 0xffff));
          a[3] = e4m3x2_to_f16x2((uint16_t)(xy23 >> 16));
        } else {
          const int j = mt >> 2, ci = mt & 3;
          const uint32_t x0 = comp(vr[0][j], ci), x1 = comp(vr[1][j], ci);
          const uint32_t y0 = comp(vr[2][j], ci), y1 = comp(vr[3][j], ci);
          a[0] = __byte_perm(x0, x1, 0x5410);
          a[1] = __byte_perm(x0, x1, 0x7632);
          a[2] = __byte_perm(y0, y1, 0x5410);
          a[3] = __byte_perm(y0, y1, 0x7632);
        }
        Mma<MT>::run(oacc[mt], a, pb0, pb1);
      }
      load_v(ntile);
      // The L2 prefetch of the page kPrefetchPieces ahead goes out when a new piece starts,
      // behind the next tile's K and V loads so that it does not delay them
      // (llama3 decode 65.4 -> 63.7 us, window 108.9 -> 106.7 us, alternating replicas).
      {
        const int jpf = nxt.piece + kPrefetchPieces;
        const bool pf = nxt.kblk && nxt.piece != cur.piece && jpf < pend && jpf < pb_base + 32;
        const int pg = __shfl_sync(0xffffffffu, pb_page, min(max(jpf - pb_base, 0), 31));
        if (pf && pg >= 0 && lane == 0) {
          prefetch_l2_bulk(kblock(pg), (uint32_t)block_bytes);
          prefetch_l2_bulk(kblock(pg) + v_off, (uint32_t)block_bytes);
        }
        if constexpr (PAIR) {  // a tile spans two pages: the one after jpf as well
          const int j2 = jpf + 1;
          const int pg2 = __shfl_sync(0xffffffffu, pb_page, min(max(j2 - pb_base, 0), 31));
          if (pf && j2 < pend && j2 < pb_base + 32 && pg2 >= 0 && lane == 0) {
            prefetch_l2_bulk(kblock(pg2), (uint32_t)block_bytes);
            prefetch_l2_bulk(kblock(pg2) + v_off, (uint32_t)block_bytes);
          }
        }
      }
      cur = nxt;
    }
  };
  if constexpr (Tr::kQSplit) {
    if (pack4) tile_loop(std::true_type{});
    else tile_loop(std::false_type{});
  } else {
    tile_loop(std::false_type{});
  }
  st_d[0] = sum_over_groups(st_d[0]);
  st_d[1] = sum_over_groups(st_d[1]);

  // ---------------------------------------------------------------- finish the segment
  // This thread holds heads 2q4 (c0, c2) and 2q4 + 1 (c1, c3); per head NR runs of RL
  // consecutive dims: run r starts at dim 16 g_id (FP8) or 8 (g_id + 8 r).
  const bool whole = (ua == 0 && ub == sg.n);
  const size_t slot = (size_t)(2 * wid + (sg.off <= ws.x0 ? 0 : 1)) * kMaxGroupPerCta;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int j = 2 * q4 + hh;
    if (j < hcount) {
      const bool empty = !(st_d[hh] > 0.f);
      float inv = empty ? 0.f : 1.f / st_d[hh];
      float l = empty ? kEmptyM : st_m[hh] + log2f(st_d[hh]);
      const size_t row = col_row<MQ>(p, sg.b, hk, c0 + j);
      if (whole && p.sink) {  // a final output: the head's sink joins here (a partial leaves it to the merge)
        const SinkAdj sa = apply_sink(p, col_head<MQ>(p, hk, c0 + j), l);
        inv *= sa.scale;
        l = sa.lse;
      }
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        const int d0 = FP8 ? 16 * g_id : 8 * (g_id + 8 * r);
        float v[RL];
#pragma unroll
        for (int o = 0; o < RL; ++o) v[o] = oacc[r * (RL / 2) + (o >> 1)][hh + 2 * (o & 1)] * inv;
        if (whole) {
#pragma unroll
          for (int o = 0; o < RL; ++o) v[o] *= p.out_scale;
          store_run<RL>(p, row * D + d0, v);
        } else {
          float4* po = reinterpret_cast<float4*>(p.part_o + (slot + j) * D + d0);
#pragma unroll
          for (int i = 0; i < RL / 4; ++i) po[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        }
      }
      if (g_id == 0) {
        if (whole) p.lse[row] = l;
        else p.part_lse[slot + j] = l;
      }
    }
  }
  if (!whole) {
    // publish the partial, count this worker's units; the worker completing the count
    // merges every partial of the segment and resets the counter for the next call
    fence_acq_rel_gpu();
    __syncwarp();
    int last = 0;
    if (lane == 0) {
      int* cnt = p.counters + (size_t)sg.b * p.H_kv * p.n_z + sg.hz;
      const int mine = ub - ua;
      const int prev = atomicAdd(cnt, mine);
      last = (prev + mine == sg.n);
      if (last) *cnt = 0;
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (last) {
      // the merge runs after this worker's last segment (only a worker's first and last
      // segments can be partial, so there are at most two), keeping the tile loop's
      // register budget free of it
      fence_acq_rel_gpu();
      if (lane == 0) {
        s_pend[warp][npend][0] = sg.b;
        s_pend[warp][npend][1] = sg.hz;
        s_pend[warp][npend][2] = sg.off;
        s_pend[warp][npend][3] = sg.n;
      }
      npend = 1;  // at most two entries: indices 0 and 1
    }
  }
  }  // ua < ub
  if (sg.off + C + sg.n >= cx1 || !next_segment(p, sg, C)) break;
  }  // segments

  // ---------------------------------------------------------------- deferred merges
  __syncwarp();
  for (int i = 0; i < 2; ++i) {
    const long long b = s_pend[warp][i][0];
    if (b < 0) continue;
    const int hz = (int)s_pend[warp][i][1];
    const long long off = s_pend[warp][i][2];
    const int n = (int)s_pend[warp][i][3];
    const int hk = hz / p.n_z, z = hz - hk * p.n_z;
    const int c0 = z * kMaxGroupPerCta;
    const int hcount = min(kMaxGroupPerCta, p.ncol - c0);
    // slot rows in flight together: about 16 float4 per lane (4 where registers are
    // tight), for the slice's head count
    constexpr int kBudget = MinBlocks<KROT, FP8>::v >= 3 ? 4 : 16;
    constexpr int kV4 = (4 * (D / 4) + 31) / 32, kV8 = (8 * (D / 4) + 31) / 32;
    if (hcount <= 4)
      warp_merge<D, 4, (kBudget / kV4 > 1 ? kBudget / kV4 : 1), MQ>(p, (int)b, off, C, n, ws.U, Wn, hk, c0, hcount, s_mw[warp], s_msl[warp], zg, (int)(wid % zg));
    else
      warp_merge<D, 8, (kBudget / kV8 > 1 ? kBudget / kV8 : 1), MQ>(p, (int)b, off, C, n, ws.U, Wn, hk, c0, hcount, s_mw[warp], s_msl[warp], zg, (int)(wid % zg));
  }
}

template <typename KVT, typename QT, int D, int RM, bool MQ, bool PAIR = false>
static cudaError_t launch_mma_t(const DecodeParams& p, dim3 grid, cudaStream_t st, MmaConfig* cfg) {
  constexpr int NW = kMmaWarps;
  constexpr int dyn = 0;
  auto kern = decode_mma_kernel<KVT, QT, D, RM, NW, MQ, PAIR>;
  if (cfg) {
    cfg->threads = NW * 32;
    cfg->smem_bytes = dyn;
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, NW * 32, dyn);
    if (e != cudaSuccess) return e;
    cfg->ctas_per_sm = n;
    return cudaSuccess;
  }
  return launch_pdl(kern, grid, dim3(NW * 32), dyn, st, p);
}

// MQ: the multi-query form (query columns = tokens x heads, causal among the tokens);
// a separate instantiation, so the single-token kernel carries none of it.
template <typename KVT, typename QT, int D, bool MQ, bool PAIR = false>
static cudaError_t launch_mma_r(const DecodeParams& p, dim3 grid, cudaStream_t st, MmaConfig* cfg) {
  const int rm = p.rotary ? p.rotary + (p.k_rotated ? 2 : 0) : 0;
  if (rm == 1) return launch_mma_t<KVT, QT, D, 1, MQ, PAIR>(p, grid, st, cfg);
  if (rm == 2) return launch_mma_t<KVT, QT, D, 2, MQ, PAIR>(p, grid, st, cfg);
  if (rm == 3) return launch_mma_t<KVT, QT, D, 3, MQ, PAIR>(p, grid, st, cfg);
  if (rm == 4) return launch_mma_t<KVT, QT, D, 4, MQ, PAIR>(p, grid, st, cfg);
  return launch_mma_t<KVT, QT, D, 0, MQ, PAIR>(p, grid, st, cfg);
}

}  // namespace pd
