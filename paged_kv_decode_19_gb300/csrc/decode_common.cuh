// Pieces shared by the decode kernels: parameters, work-item location (length
// decode + split plan), the row -> page mapping, and the per-block finish (merge
// of the warps' softmax states, then either the final output or a partial state
// plus an on-device merge of the sequence's partials by its last-finishing block).
//
// Source of the operation: Apache TVM `_decode_kernels.py`, `batch_decode_paged_kv`
// (length_info, page-table addressing, base-2 online softmax, lse in log2 units)
// and `merge_state_inplace` (the state-merge formula, used here for the split-KV
// combine and for the in-block combine of the warps' states).
#pragma once

#include "common.cuh"

namespace pd {

constexpr int kMaxGroupPerCta = 8;  // query heads one block serves (a grid z-slice)
constexpr int kMaxHalfDim = 128;    // D <= 256

struct DecodeParams {
  const void* Q;
  const void* pages;
  const int32_t* indptr;
  const int32_t* values;
  const int32_t* length_info;
  const int32_t* k_rope_pos_offset;
  const int32_t* q_rope_position;
  void* out;
  float* lse;
  float* part_o;    // [grid_items, H_qo, D] fp32 partial outputs (normalised)
  float* part_lse;  // [grid_items, H_qo] fp32 partial lse (log2)
  int* counters;    // [B, H_kv, n_z] arrivals per (sequence, KV head, head slice)
  unsigned* err;    // device error word
  long long max_pages;
  int B, H_qo, H_kv, D, P, group, n_z;
  int window, rotary;
  int precise;        // fp32 path: softmax weights via double-precision exp2
  int chunk_rows;     // attended rows per work item (INT_MAX: no split)
  int out_dtype;
  float score_scale;  // raw q.k -> log2 units (sm_scale * log2 e [* k_scale])
  float q_prescale;   // split-operand MMA path: Q is pre-multiplied by this
  float out_scale;    // applied to the final output (v_scale for e4m3 KV)
  unsigned long long rope_F[kMaxHalfDim];  // fixed-point turns/position per frequency
};

// Attended length and row mapping of one sequence (length_info reading: no window
// -> L = (npages-1)P + last, rows at offsets 0..L-1; window -> L = (npages-1)P + last
// - win_off + sink, row r at r (r < sink) or r - sink + win_off).
struct SeqInfo {
  int L, sink, win_off, page_begin, npages;
};

__device__ __forceinline__ SeqInfo load_seq(const DecodeParams& p, int b) {
  SeqInfo s;
  s.page_begin = p.indptr[b];
  s.npages = p.indptr[b + 1] - s.page_begin;
  s.L = 0;
  s.sink = 0;
  s.win_off = 0;
  if (s.npages <= 0) {
    if (s.npages < 0) set_error(p.err, kErrBadLength);
    s.npages = 0;
    return s;
  }
  long long last = p.length_info[b];
  long long L;
  if (!p.window) {
    L = (long long)(s.npages - 1) * p.P + last;
    s.sink = (int)min(max(L, 0ll), (long long)INT32_MAX);
  } else {
    long long off = p.length_info[p.B + b], sk = p.length_info[2 * p.B + b];
    L = (long long)(s.npages - 1) * p.P + last - off + sk;
    if (sk < 0 || off < sk) {  // inconsistent window: sequence treated as empty
      set_error(p.err, kErrBadLength);
      L = 0;
    }
    s.sink = (int)sk;
    s.win_off = (int)off;
  }
  if (L < 0 || L > (long long)INT32_MAX) {
    set_error(p.err, kErrBadLength);
    L = 0;
  }
  s.L = (int)L;
  return s;
}

// Work items of a sequence: ceil(L / chunk_rows), and one (empty) item for L = 0 so
// that an empty sequence still gets its output written (out = 0, lse = -5e4).
__device__ __forceinline__ int chunks_of(int L, int chunk_rows) {
  return L > 0 ? 1 + (L - 1) / chunk_rows : 1;
}

struct Work {
  int b, chunk, nchunks, first_item;
  SeqInfo seq;
};

// Finds which (sequence, chunk) the work item `item` is: a block-wide exclusive scan
// of the per-sequence chunk counts.  Returns false if `item` is past the last chunk.
// Block 0 flags a plan overflow (more chunks than grid items).
template <int NT>
__device__ bool locate_item(const DecodeParams& p, int item, Work& w) {
  __shared__ int s_warp[NT / 32];
  __shared__ int s_hit[3];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  if (tid == 0) s_hit[0] = -1;
  int base = 0;
  for (int start = 0; start < p.B; start += NT) {
    const int b = start + tid;
    int n = 0, L = 0;
    if (b < p.B) {
      SeqInfo s = load_seq(p, b);
      L = s.L;
      n = chunks_of(L, p.chunk_rows);
    }
    int incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) s_warp[wid] = incl;
    __syncthreads();
    int warp_base = 0, total = 0;
#pragma unroll
    for (int i = 0; i < NT / 32; ++i) {
      int v = s_warp[i];
      if (i < wid) warp_base += v;
      total += v;
    }
    incl += warp_base;
    const int excl = incl - n;
    if (b < p.B && item >= base + excl && item < base + incl) {
      s_hit[0] = b;
      s_hit[1] = item - base - excl;
      s_hit[2] = n;
    }
    base += total;
    __syncthreads();
  }
  __syncthreads();
  if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && tid == 0 && base > (int)gridDim.x)
    set_error(p.err, kErrBadLength);
  if (s_hit[0] < 0) return false;
  w.b = s_hit[0];
  w.chunk = s_hit[1];
  w.nchunks = s_hit[2];
  w.first_item = item - w.chunk;
  w.seq = load_seq(p, w.b);
  return true;
}

// ---------------------------------------------------------------------------- pieces
// A chunk's attended rows [r0, r1) cover at most two contiguous runs of sequence
// offsets (the sink run and the window run); each run is cut at page boundaries into
// "pieces": one page, a slot range [s_lo, s_hi), first attended row r_lo.
struct Pieces {
  int ra0, ra1, ob0, ob1, shift;  // run A rows [ra0,ra1) (offset = row); run B offsets [ob0,ob1)
  int pa, na, pb, nb;             // first page and count of each run
  __device__ __forceinline__ int count() const { return na + nb; }
};

__device__ __forceinline__ Pieces make_pieces(int r0, int r1, const SeqInfo& s, int P) {
  Pieces c;
  c.ra0 = r0;
  c.ra1 = max(r0, min(r1, s.sink));
  const int rb0 = max(r0, s.sink), rb1 = max(rb0, r1);
  c.shift = s.win_off - s.sink;
  c.ob0 = rb0 + c.shift;
  c.ob1 = rb1 + c.shift;
  c.pa = c.ra0 / P;
  c.na = c.ra1 > c.ra0 ? (c.ra1 - 1) / P - c.pa + 1 : 0;
  c.pb = c.ob0 / P;
  c.nb = c.ob1 > c.ob0 ? (c.ob1 - 1) / P - c.pb + 1 : 0;
  return c;
}

struct Piece {
  int page_idx, s_lo, s_hi, r_lo;
};

__device__ __forceinline__ Piece get_piece(const Pieces& c, int i, int P) {
  Piece q;
  int lo, hi, shift;
  if (i < c.na) {
    q.page_idx = c.pa + i;
    lo = c.ra0;
    hi = c.ra1;
    shift = 0;
  } else {
    q.page_idx = c.pb + (i - c.na);
    lo = c.ob0;
    hi = c.ob1;
    shift = c.shift;
  }
  const int pbase = q.page_idx * P;
  const int o_lo = max(lo, pbase), o_hi = min(hi, pbase + P);
  q.s_lo = o_lo - pbase;
  q.s_hi = o_hi - pbase;
  q.r_lo = o_lo - shift;
  return q;
}

// Physical page of piece page index `pidx` (or -1 when out of range -> error bit).
__device__ __forceinline__ int lookup_page(const DecodeParams& p, const SeqInfo& s, int pidx) {
  if (pidx < 0 || pidx >= s.npages) {
    set_error(p.err, kErrBadPage);
    return -1;
  }
  const int page = __ldg(p.values + s.page_begin + pidx);
  if (page < 0 || (long long)page >= p.max_pages) {
    set_error(p.err, kErrBadPage);
    return -1;
  }
  return page;
}

// ---------------------------------------------------------------------------- finish
// 2^x for the merge weights: fp32-accurate on the fp32 path, hardware ex2 otherwise.
__device__ __forceinline__ float merge_exp2(const DecodeParams& p, float x) {
  return p.precise ? (float)exp2((double)x) : fast_exp2(x);
}

__device__ __forceinline__ void store_out(const DecodeParams& p, size_t idx, float v) {
  if (p.out_dtype == kF32) reinterpret_cast<float*>(p.out)[idx] = v;
  else if (p.out_dtype == kBF16) reinterpret_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16_rn(v);
  else reinterpret_cast<__half*>(p.out)[idx] = __float2half_rn(v);
}

// Merge the NWS warp states held in shared memory (sm_m/sm_d [NWS][8], sm_o
// [NWS][8][D], unnormalised O, log2-unit m) and write the block's result for heads
// [hq0, hq0+hcount).  A single-chunk sequence writes out/lse directly; otherwise the
// block writes its partial (O/d, lse), and the last block of the sequence to finish
// merges all partials of the sequence (S-way form of merge_state).
template <int NT, int NWS>
__device__ void finish_block(const DecodeParams& p, const Work& w, int item, int hk, int z,
                             int hq0, int hcount, const float* sm_m, const float* sm_d,
                             const float* sm_o) {
  __shared__ int s_last;
  const int D = p.D;
  const int tid = threadIdx.x;
  const bool split = w.nchunks > 1;
  for (int idx = tid; idx < hcount * D; idx += NT) {
    const int j = idx / D, d = idx - j * D;
    float M = kEmptyM;
#pragma unroll
    for (int s = 0; s < NWS; ++s) M = fmaxf(M, sm_m[s * 8 + j]);
    float den = 0.f, num = 0.f;
#pragma unroll
    for (int s = 0; s < NWS; ++s) {
      const float a = merge_exp2(p, sm_m[s * 8 + j] - M);
      den += sm_d[s * 8 + j] * a;
      num += sm_o[(s * 8 + j) * D + d] * a;
    }
    const bool empty = !(den > 0.f);
    const float o = empty ? 0.f : num / den;
    const float l = empty ? kEmptyM : M + log2f(den);
    const int hq = hq0 + j;
    if (!split) {
      store_out(p, ((size_t)w.b * p.H_qo + hq) * D + d, o * p.out_scale);
      if (d == 0) p.lse[(size_t)w.b * p.H_qo + hq] = l;
    } else {
      p.part_o[((size_t)item * p.H_qo + hq) * D + d] = o;
      if (d == 0) p.part_lse[(size_t)item * p.H_qo + hq] = l;
    }
  }
  if (!split) return;
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    int* cnt = p.counters + ((size_t)w.b * p.H_kv + hk) * p.n_z + z;
    const int prev = atomicAdd(cnt, 1);
    s_last = (prev == w.nchunks - 1);
    if (s_last) *cnt = 0;  // every other block of this sequence has arrived: reset for reuse
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int idx = tid; idx < hcount * D; idx += NT) {
    const int j = idx / D, d = idx - j * D;
    const int hq = hq0 + j;
    float M = kEmptyM;
    for (int c = 0; c < w.nchunks; ++c)
      M = fmaxf(M, __ldcg(p.part_lse + (size_t)(w.first_item + c) * p.H_qo + hq));
    float den = 0.f, num = 0.f;
    for (int c = 0; c < w.nchunks; ++c) {
      const size_t it = (size_t)(w.first_item + c);
      const float a = merge_exp2(p, __ldcg(p.part_lse + it * p.H_qo + hq) - M);
      den += a;
      num += a * __ldcg(p.part_o + (it * p.H_qo + hq) * D + d);
    }
    const bool empty = !(M > kEmptyM);
    store_out(p, ((size_t)w.b * p.H_qo + hq) * D + d, empty ? 0.f : num / den * p.out_scale);
    if (d == 0) p.lse[(size_t)w.b * p.H_qo + hq] = empty ? kEmptyM : M + log2f(den);
  }
}

}  // namespace pd
