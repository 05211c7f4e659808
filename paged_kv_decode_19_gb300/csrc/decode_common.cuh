// Pieces shared by the decode kernels: parameters, length decode, the row -> page
// mapping, the block schedule (which pages of which (sequence, KV head) a block
// processes) and the finish of a block's share of a sequence (merge of the warps'
// softmax states, then the final output, or a partial state that the last block of
// the sequence to finish merges with the others).
//
// Source of the operation: Apache TVM `_decode_kernels.py`, `batch_decode_paged_kv`
// (length_info, page-table addressing, base-2 online softmax, lse in log2 units)
// and `merge_state_inplace` (the state-merge formula, used here for the split-KV
// combine and for the in-block combine of the warps' states).
#pragma once

#include "common.cuh"

namespace pd {

constexpr int kMaxGroupPerCta = 8;  // query heads one block serves at a time (a z-slice)
constexpr int kMaxHalfDim = 128;    // D <= 256
constexpr int kMmaWarps = 4;        // warps (independent workers) per tensor-core block
constexpr int kStartCacheB = 1024;  // batch sizes whose start-up scan runs in shared memory
// Host plan: ints of sequence metadata the launch itself may carry (see DecodeParams::hp)
constexpr int kHostPlanInts = 1024;

// Block schedules (DecodeParams::mode)
enum : int {
  kSchedBalanced = 0,   // all pages of all (sequence, head-slice) segments, cut into G equal shares
  kSchedPerSegment = 1  // one block per (sequence, head-slice) segment: no split
};

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
  float* part_o;    // [2G][8][D] fp32 partial outputs (normalised): slot 2c + side
  float* part_lse;  // [2G][8] fp32 partial lse (log2)
  int* counters;    // [B * H_kv * n_z] pages merged so far per segment (reset by the last)
  unsigned* err;    // device error word
  long long max_pages;
  long long nnz_pages;  // entries of the page table (page_table_values)
  int B, H_qo, H_kv, D, P, group, n_z;
  int zg;             // 1, or n_z (2 or 4): the n_z slices of a (sequence, KV head) run on
                      // n_z adjacent warps of one block, which walk the same pages together
                      // (the cost line then holds (sequence, KV head) groups, one position per
                      // page, and every group of n_z warps takes one share of it)
  int q_len;          // query tokens per sequence (multi-query decode; 1 = plain decode)
  int ncol;           // query columns per KV head: q_len * group, in slices of <= 8
  int window, rotary;
  int precise;        // fp32 path: merge weights via the accurate exp2f
  int mode;           // kSchedBalanced / kSchedPerSegment
  int seg_cost;       // worker schedule: extra cost units charged per segment (its set-up
                      // and finish), so ranges that cross segment boundaries get fewer pages
  int out_dtype;
  int out_vec16;      // out is 16-byte aligned (vector stores of whole runs)
  int early_inputs;   // Q, page table, lengths and positions may be read before pdl_wait()
  const float* sink;  // [H_qo] learned logit per query head (natural units), or nullptr
  int k_rotated;      // the cache holds K rotated at append time: only Q is rotated here
  float score_scale;  // raw q.k -> log2 units (sm_scale * log2 e [* k_scale])
  float q_prescale;   // split-operand MMA path: Q is pre-multiplied by this
  float out_scale;    // applied to the final output (v_scale for e4m3 KV)
  unsigned long long rope_F[kMaxHalfDim];  // fixed-point turns/position per frequency
  // Host plan: when hp_B > 0 the caller gave host copies of page_table_indptr and
  // length_info, and the launch carries them: hp[0 .. B] = prefix sums over the
  // sequences of (work units + seg_cost), hp[hp_ptr ..] = indptr [B+1],
  // hp[hp_li ..] = length_info [B] or [3,B].  The kernels then read a sequence's
  // lengths and page-table offset from here, and each worker finds its first segment
  // by a binary search over the prefix, without the start-up scan of device memory.
  // (The launch's parameters grow with hp: measured, a 16 KB plan made every launch about
  // 1.5 us slower than a 4 KB one, while 0.6 KB and 4 KB cost the same.)
  int hp_B, hp_ptr, hp_li;
  int32_t hp[kHostPlanInts];
};

// Attended length and row mapping of one sequence (length_info reading: no window
// -> L = (npages-1)P + last, rows at offsets 0..L-1; window -> L = (npages-1)P + last
// - win_off + sink, row r at r (r < sink) or r - sink + win_off).
struct SeqInfo {
  int L, sink, win_off, page_begin, npages;
};

// Row of (sequence b, query column c of KV head hk) in Q, out and lse: column c is query
// token c / group and head hk * group + c % group (with one token per sequence, c is
// the head's index within the group).
// MQ = false: one token per sequence (no division).
template <bool MQ>
__device__ __forceinline__ size_t col_row(const DecodeParams& p, int b, int hk, int c) {
  if (!MQ) return (size_t)b * p.H_qo + hk * p.group + c;
  const int t = c / p.group;
  return ((size_t)b * p.q_len + t) * p.H_qo + hk * p.group + (c - t * p.group);
}

// Query head of column c of KV head hk.
template <bool MQ>
__device__ __forceinline__ int col_head(const DecodeParams& p, int hk, int c) {
  return hk * p.group + (MQ ? c % p.group : c);
}

// A learned sink logit of query head h joins the softmax as one more score with a zero
// value row.  Given a final, sink-free output (o, lse = l; l = kEmptyM when no row was
// attended), the result is o * scale with lse: the merge of (o, l) with (0, sink log2 e).
struct SinkAdj {
  float scale, lse;
};
__device__ __forceinline__ SinkAdj apply_sink(const DecodeParams& p, int h, float l) {
  if (!p.sink) return {1.f, l};
  const float ls = __ldg(p.sink + h) * 1.4426950408889634f;
  const float m = fmaxf(l, ls);
  const float a = l > kEmptyM ? exp2f(l - m) : 0.f;  // weight of the attended rows
  const float den = a + exp2f(ls - m);
  return {a / den, m + log2f(den)};
}

// SeqInfo from a sequence's raw fields (page-table offsets i0, i1; last page length;
// window start and sink length); an inconsistent sequence is treated as empty and sets
// `bad`.  Shared by the kernels and the host planner, so both count the same work.
__host__ __device__ __forceinline__ SeqInfo seq_from(long long i0, long long i1, long long last,
                                                     long long off, long long sk, int P,
                                                     bool window, bool& bad) {
  SeqInfo s;
  s.page_begin = (int)i0;
  s.npages = (int)(i1 - i0);
  s.L = 0;
  s.sink = 0;
  s.win_off = 0;
  if (s.npages <= 0) {
    if (s.npages < 0) bad = true;
    s.npages = 0;
    return s;
  }
  long long L;
  if (!window) {
    L = (long long)(s.npages - 1) * P + last;
    s.sink = (int)(L < 0 ? 0 : L > (long long)INT32_MAX ? (long long)INT32_MAX : L);
  } else {
    L = (long long)(s.npages - 1) * P + last - off + sk;
    if (sk < 0 || off < sk) {  // inconsistent window: sequence treated as empty
      bad = true;
      L = 0;
    }
    s.sink = (int)sk;
    s.win_off = (int)off;
  }
  if (L < 0 || L > (long long)INT32_MAX) {
    bad = true;
    L = 0;
  }
  s.L = (int)L;
  return s;
}

__device__ __forceinline__ SeqInfo load_seq(const DecodeParams& p, int b) {
  long long i0, i1, last, off = 0, sk = 0;
  if (p.hp_B) {  // the launch carries the host copies
    i0 = p.hp[p.hp_ptr + b];
    i1 = p.hp[p.hp_ptr + b + 1];
    last = p.hp[p.hp_li + b];
    if (p.window) {
      off = p.hp[p.hp_li + p.B + b];
      sk = p.hp[p.hp_li + 2 * p.B + b];
    }
  } else {
    // every load is issued up front (one round trip), then the fields are checked
    i0 = __ldg(p.indptr + b);
    i1 = __ldg(p.indptr + b + 1);
    last = __ldg(p.length_info + b);
    if (p.window) {
      off = __ldg(p.length_info + p.B + b);
      sk = __ldg(p.length_info + 2 * p.B + b);
    }
  }
  bool bad = false;
  const SeqInfo s = seq_from(i0, i1, last, off, sk, p.P, p.window != 0, bad);
  if (bad) set_error(p.err, kErrBadLength);
  return s;
}

// ---------------------------------------------------------------------------- pieces
// A sequence's attended rows [0, L) cover at most two contiguous runs of sequence
// offsets (the sink run and the window run); each run is cut at page boundaries into
// "pieces": one page, a slot range [s_lo, s_hi), first attended row r_lo.
struct Pieces {
  int ra0, ra1, ob0, ob1, shift;  // run A rows [ra0,ra1) (offset = row); run B offsets [ob0,ob1)
  int pa, na, pb, nb;             // first page and count of each run
  __host__ __device__ __forceinline__ int count() const { return na + nb; }
};

__host__ __device__ __forceinline__ int imin(int a, int b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int imax(int a, int b) { return a > b ? a : b; }

__host__ __device__ __forceinline__ Pieces make_pieces(int r0, int r1, const SeqInfo& s, int P) {
  Pieces c;
  c.ra0 = r0;
  c.ra1 = imax(r0, imin(r1, s.sink));
  const int rb0 = imax(r0, s.sink), rb1 = imax(rb0, r1);
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

__host__ __device__ __forceinline__ Piece get_piece(const Pieces& c, int i, int P) {
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

// Work units of a sequence: its pieces, or one (empty) unit when it has none, so that
// an empty sequence still gets its output written (out = 0, lse = -5e4).
__host__ __device__ __forceinline__ int units_of(const SeqInfo& s, int P) {
  return s.L > 0 ? make_pieces(0, s.L, s, P).count() : 1;
}

// Physical page of piece page index `pidx` (or -1 when out of range -> error bit).
__device__ __forceinline__ int lookup_page(const DecodeParams& p, const SeqInfo& s, int pidx) {
  if (pidx < 0 || pidx >= s.npages || (long long)s.page_begin + pidx >= p.nnz_pages) {
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

// ---------------------------------------------------------------------------- schedule
// Segments are (sequence b, head slice hz = hk * n_z + z) in the order b-major; segment
// (b, hz) owns units [HZ * pre_b + hz * n_b, ... + n_b) of the global unit range [0, U),
// with n_b = units_of(b), pre_b = sum of n_b' for b' < b, HZ = H_kv * n_z.
// Balanced schedule: block c takes units [floor(c U / G), floor((c+1) U / G)).
// Per-segment schedule: block c takes exactly segment c.
struct Segment {
  int b, hz, n;       // sequence, head slice, its units
  long long off;      // first global unit of the segment
  SeqInfo seq;
};

struct BlockRange {
  long long x0, x1, U;
  Segment seg;        // segment containing x0 (valid when x0 < x1)
};

// Block-wide: total units U, this block's range, and the segment holding its first unit.
template <int NT>
__device__ BlockRange block_range(const DecodeParams& p) {
  __shared__ long long s_warp[NT / 32];
  __shared__ long long s_hit[2];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int HZ = p.H_kv * p.n_z;
  const long long G = gridDim.x;
  BlockRange r;
  if (p.mode != kSchedBalanced) {
    // per-segment: block c takes segment c = (sequence c / HZ, slice c % HZ) whole, on a
    // private range; no scan (the barrier publishes what the block wrote before the call)
    __syncthreads();
    const long long c = blockIdx.x;
    r.U = (long long)p.B * HZ;
    r.x0 = r.x1 = 0;
    if (c >= r.U) return r;
    Segment& sg = r.seg;
    sg.b = (int)(c / HZ);
    sg.hz = (int)(c - (long long)sg.b * HZ);
    sg.seq = load_seq(p, sg.b);
    sg.n = units_of(sg.seq, p.P);
    sg.off = 0;
    r.x1 = sg.n;
    return r;
  }
  // pass 1: U
  long long total = 0;
  for (int start = 0; start < p.B; start += NT) {
    const int b = start + tid;
    long long n = b < p.B ? units_of(load_seq(p, b), p.P) : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
    if (lane == 0) s_warp[wid] = n;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < NT / 32; ++i) total += s_warp[i];
    __syncthreads();
  }
  r.U = total * HZ;
  const long long c = blockIdx.x;
  long long target;
  if (p.mode == kSchedBalanced) {
    r.x0 = c * r.U / G;
    r.x1 = (c + 1) * r.U / G;
    target = r.x0;
  } else {
    r.x0 = r.x1 = -1;  // set below from the segment
    target = c;        // segment index
  }
  // pass 2: the sequence holding `target` (a unit, or a segment index)
  if (tid == 0) s_hit[0] = -1;
  long long base = 0;
  for (int start = 0; start < p.B; start += NT) {
    const int b = start + tid;
    const long long n = b < p.B ? (p.mode == kSchedBalanced ? (long long)units_of(load_seq(p, b), p.P) * HZ : HZ) : 0;
    long long incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) s_warp[wid] = incl;
    __syncthreads();
    long long wbase = 0, tot = 0;
#pragma unroll
    for (int i = 0; i < NT / 32; ++i) {
      const long long v = s_warp[i];
      if (i < wid) wbase += v;
      tot += v;
    }
    incl += wbase;
    if (b < p.B && target >= base + incl - n && target < base + incl) {
      s_hit[0] = b;
      s_hit[1] = base + incl - n;  // balanced: first unit of b; per-segment: first segment of b
    }
    base += tot;
    __syncthreads();
  }
  __syncthreads();
  const int b = (int)s_hit[0];
  if (b < 0) {
    r.x0 = r.x1 = 0;
    return r;
  }
  Segment& sg = r.seg;
  sg.b = b;
  sg.seq = load_seq(p, b);
  sg.n = units_of(sg.seq, p.P);
  if (p.mode == kSchedBalanced) {
    const long long first = s_hit[1];  // = HZ * pre_b
    sg.hz = (int)((target - first) / sg.n);
    sg.off = first + (long long)sg.hz * sg.n;
  } else {
    // per-segment: units of earlier sequences are needed for the global offset, but
    // only the segment's own range matters here; give it a private range
    sg.hz = (int)(target - s_hit[1]);
    sg.off = 0;
    r.x0 = 0;
    r.x1 = sg.n;
  }
  return r;
}

// Next segment after `s` (same sequence next head slice, or the next sequence); each
// segment spans its n units plus `extra` cost units on the schedule's line.
__device__ __forceinline__ bool next_segment(const DecodeParams& p, Segment& s, int extra = 0) {
  const int HZ = p.H_kv * p.n_z;
  s.off += s.n + extra;
  if (s.hz + p.zg < HZ) {  // the next KV head's slice of this warp (zg = 1: next slice)
    s.hz += p.zg;
    return true;
  }
  if (s.b + 1 >= p.B) return false;
  ++s.b;
  s.hz = s.hz % p.zg;
  s.seq = load_seq(p, s.b);
  s.n = units_of(s.seq, p.P);
  return true;
}

// floor(a / b) for 0 <= a, 0 < b: the hardware-friendly 32-bit division when both fit in
// 32 bits (the usual case: cost-line positions times worker counts), else the 64-bit one.
__device__ __forceinline__ long long div_floor(long long a, long long b) {
  if (((unsigned long long)a | (unsigned long long)b) < (1ull << 32))
    return (long long)((unsigned)a / (unsigned)b);
  return a / b;
}

// Share (block or worker) whose balanced range holds global unit x, with G shares:
// floor(((x+1) G - 1) / U).
__device__ __forceinline__ long long share_of(long long x, long long U, long long G) {
  return div_floor((x + 1) * G - 1, U);
}

// ---------------------------------------------------------------------------- workers
// Independent workers (warps of the tensor-core kernel): worker w = block * WPB + i.
// Balanced schedule: every segment occupies n + C positions of a cost line (C =
// p.seg_cost positions for its set-up and finish, then its n units); worker w takes
// positions [floor(w U / W), floor((w+1) U / W)) of the line's U positions, with
// W = gridDim.x * WPB, i.e. the units of each segment whose positions fall in its range.
// Per-segment schedule: worker w takes segment w whole.
struct WorkerStart {
  long long x0, x1, U;  // cost-line range (per-segment: [0, huge)), line length
  long long off;        // line position where the segment holding x0 starts
  int b, hz;            // that segment; b < 0: this worker has no work
};

// Block-wide (ends with a block barrier): the start of each of the block's WPB workers.
// s_units: shared scratch of kStartCacheB ints.
template <int NT, int WPB>
__device__ void worker_starts(const DecodeParams& p, WorkerStart* s_ws, int* s_units) {
  __shared__ long long s_warp[NT / 32];
  __shared__ long long s_hit[WPB][2];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int C = p.seg_cost;
  // grouped slices (zg > 1): the line holds (sequence, KV head) groups and each group of
  // zg adjacent workers takes one share of it; worker i of the block is line worker
  // (w_first + i) / zg, slice (w_first + i) % zg of each group
  const int zg = p.mode == kSchedBalanced ? p.zg : 1;
  const int HZ = p.H_kv * p.n_z / zg;
  const long long W = (long long)gridDim.x * WPB / zg;
  const long long w_first = (long long)blockIdx.x * WPB;
  if (p.hp_B && p.mode == kSchedBalanced) {
    // host plan: the sequences' cost-line prefix is in the launch; each worker finds the
    // sequence holding its first position by a binary search over it
    if (tid < WPB) {
      const int32_t* pre = p.hp;  // [B+1], strictly increasing (every sequence >= 1 unit)
      const long long U = (long long)pre[p.B] * HZ;
      const long long w = (w_first + tid) / zg;
      WorkerStart s;
      s.U = U;
      s.x0 = div_floor(w * U, W);
      s.x1 = div_floor((w + 1) * U, W);
      s.b = -1;
      s.hz = 0;
      s.off = 0;
      if (s.x0 < s.x1) {
        int lo = 0, hi = p.B - 1;  // last b with pre[b] * HZ <= x0
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if ((long long)pre[mid] * HZ <= s.x0) lo = mid;
          else hi = mid - 1;
        }
        const long long first = (long long)pre[lo] * HZ;
        const int n = pre[lo + 1] - pre[lo];
        s.b = lo;
        s.hz = (int)((s.x0 - first) / n);
        s.off = first + (long long)s.hz * n;
        s.hz = s.hz * zg + (int)((w_first + tid) % zg);
      } else {
        s.x1 = s.x0;
      }
      s_ws[tid] = s;
    }
    __syncthreads();
    return;
  }
  if (p.mode != kSchedBalanced) {
    if (tid < WPB) {
      const long long w = w_first + tid;
      WorkerStart s;
      s.U = (long long)p.B * HZ;
      s.off = 0;
      s.x0 = 0;
      s.hz = 0;
      s.b = -1;
      s.x1 = 0;
      if (w < s.U) {
        s.b = (int)(w / HZ);
        s.hz = (int)(w - (long long)s.b * HZ);
        s.x1 = LLONG_MAX;
      }
      s_ws[tid] = s;
    }
    __syncthreads();
    return;
  }
  long long U;
  if (p.B <= kStartCacheB) {
    // one pass over the sequences: unit counts into shared memory, then a block-wide
    // scan in which each thread owns `per` consecutive sequences
    for (int b = tid; b < p.B; b += NT) s_units[b] = units_of(load_seq(p, b), p.P);
    if (tid < WPB) s_hit[tid][0] = -1;
    __syncthreads();
    const int per = (p.B + NT - 1) / NT;
    const int b0 = min(tid * per, p.B), b1 = min(b0 + per, p.B);
    long long mine = 0;
    for (int b = b0; b < b1; ++b) mine += s_units[b] + C;
    long long incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) s_warp[wid] = incl;
    __syncthreads();
    long long wbase = 0, total = 0;
#pragma unroll
    for (int i = 0; i < NT / 32; ++i) {
      const long long v = s_warp[i];
      if (i < wid) wbase += v;
      total += v;
    }
    U = total * HZ;
    long long lo = (wbase + incl - mine) * HZ;
    for (int b = b0; b < b1; ++b) {
      const long long hi = lo + (long long)(s_units[b] + C) * HZ;
#pragma unroll
      for (int i = 0; i < WPB; ++i) {
        const long long t = ((w_first + i) / zg) * U / W;
        if (t >= lo && t < hi) {
          s_hit[i][0] = b;
          s_hit[i][1] = lo;  // = HZ * (units of the sequences before b)
        }
      }
      lo = hi;
    }
    __syncthreads();
  } else {
    // pass 1: total units
    long long total = 0;
    for (int start = 0; start < p.B; start += NT) {
      const int b = start + tid;
      long long n = b < p.B ? units_of(load_seq(p, b), p.P) + C : 0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
      if (lane == 0) s_warp[wid] = n;
      __syncthreads();
#pragma unroll
      for (int i = 0; i < NT / 32; ++i) total += s_warp[i];
      __syncthreads();
    }
    U = total * HZ;
    if (tid < WPB) s_hit[tid][0] = -1;
    __syncthreads();
    // pass 2: the sequence holding each worker's first unit
    long long base = 0;
    for (int start = 0; start < p.B; start += NT) {
      const int b = start + tid;
      const long long n = b < p.B ? (long long)(units_of(load_seq(p, b), p.P) + C) * HZ : 0;
      long long incl = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      if (lane == 31) s_warp[wid] = incl;
      __syncthreads();
      long long wbase = 0, tot = 0;
#pragma unroll
      for (int i = 0; i < NT / 32; ++i) {
        const long long v = s_warp[i];
        if (i < wid) wbase += v;
        tot += v;
      }
      incl += wbase;
      const long long lo = base + incl - n, hi = base + incl;
#pragma unroll
      for (int i = 0; i < WPB; ++i) {
        const long long t = ((w_first + i) / zg) * U / W;
        if (b < p.B && t >= lo && t < hi) {
          s_hit[i][0] = b;
          s_hit[i][1] = lo;
        }
      }
      base += tot;
      __syncthreads();
    }
  }
  if (tid < WPB) {
    const long long w = (w_first + tid) / zg;
    WorkerStart s;
    s.U = U;
    s.x0 = w * U / W;
    s.x1 = (w + 1) * U / W;
    s.b = (int)s_hit[tid][0];
    s.hz = 0;
    s.off = 0;
    if (s.x0 >= s.x1 || s.b < 0) {
      s.b = -1;
      s.x1 = s.x0;
    } else {
      const int n = C + (s.b < kStartCacheB && p.B <= kStartCacheB ? s_units[s.b] : units_of(load_seq(p, s.b), p.P));
      s.hz = (int)((s.x0 - s_hit[tid][1]) / n);
      s.off = s_hit[tid][1] + (long long)s.hz * n;
      s.hz = s.hz * zg + (int)((w_first + tid) % zg);
    }
    s_ws[tid] = s;
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------- finish
// 2^x for the merge weights: the accurate exp2f on the fp32 path, hardware ex2 otherwise.
__device__ __forceinline__ float merge_exp2(const DecodeParams& p, float x) {
  return p.precise ? exp2f(x) : fast_exp2(x);
}

__device__ __forceinline__ void store_out(const DecodeParams& p, size_t idx, float v) {
  if (p.out_dtype == kF32) reinterpret_cast<float*>(p.out)[idx] = v;
  else if (p.out_dtype == kBF16) reinterpret_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16_rn(v);
  else reinterpret_cast<__half*>(p.out)[idx] = __float2half_rn(v);
}

// Partial slot written by block cc for a segment whose first global unit is `off`,
// or -1 when block cc's range is empty (it wrote nothing).
__device__ __forceinline__ long long share_slot(long long cc, long long off, long long U,
                                                long long G) {
  const long long x0 = div_floor(cc * U, G);
  if (div_floor((cc + 1) * U, G) <= x0) return -1;
  return (2 * cc + (off <= x0 ? 0 : 1)) * kMaxGroupPerCta;
}
// The same for line worker cc of a grouped schedule: its slice-z worker is cc * zg + z.
__device__ __forceinline__ long long share_slot_z(long long cc, long long off, long long U,
                                                  long long G, int zg, int z) {
  const long long x0 = div_floor(cc * U, G);
  if (div_floor((cc + 1) * U, G) <= x0) return -1;
  return (2 * (cc * zg + z) + (off <= x0 ? 0 : 1)) * kMaxGroupPerCta;
}

// Combine the partial states of every block holding units of segment `sg` into the
// final out/lse (merge_state over S partials: lse = M + log2 sum_s 2^(lse_s - M),
// out = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M)).  Called by the block that
// completed the segment's count.  All slots' lse are read in parallel (one slot per
// thread), the weights go to shared memory, and each thread then sums its float4 of
// (head, dims) over a chunk of slots with independent loads, so the merge costs a few
// L2 round trips rather than one per slot.
template <int NT>
__device__ void merge_segment(const DecodeParams& p, const BlockRange& br, const Segment& sg,
                              int hq0, int hcount) {
  constexpr int G8 = kMaxGroupPerCta;
  constexpr int kVec = G8 * 2 * kMaxHalfDim / 4 / NT;  // float4s per thread, at most
  __shared__ float s_w[NT][G8];
  __shared__ long long s_sl[NT];
  __shared__ float s_red[NT / 32][G8];
  __shared__ float s_M[G8], s_den[G8];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int D = p.D, D4 = D / 4;
  const long long G = gridDim.x;
  const long long c0 = share_of(sg.off, br.U, G);
  const int ns = (int)(share_of(sg.off + sg.n - 1, br.U, G) - c0 + 1);
  const long long sl0 = share_slot(c0, sg.off, br.U, G);  // block c0 always holds units
  // pass 1: per-head maximum of the partial lse
  float m[G8];
#pragma unroll
  for (int j = 0; j < G8; ++j) m[j] = kEmptyM;
  for (int s = tid; s < ns; s += NT) {
    const long long sl = share_slot(c0 + s, sg.off, br.U, G);
    if (sl < 0) continue;
    const float4 a = __ldcg(reinterpret_cast<const float4*>(p.part_lse + sl));
    const float4 b = __ldcg(reinterpret_cast<const float4*>(p.part_lse + sl) + 1);
    const float v[G8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int j = 0; j < G8; ++j) m[j] = fmaxf(m[j], j < hcount ? v[j] : kEmptyM);
  }
#pragma unroll
  for (int j = 0; j < G8; ++j) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m[j] = fmaxf(m[j], __shfl_xor_sync(0xffffffffu, m[j], o));
    if (lane == 0) s_red[wid][j] = m[j];
  }
  __syncthreads();
  if (tid < G8) {
    float M = kEmptyM;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) M = fmaxf(M, s_red[w][tid]);
    s_M[tid] = M;
  }
  __syncthreads();
  float M[G8], den[G8];
#pragma unroll
  for (int j = 0; j < G8; ++j) {
    M[j] = s_M[j];
    den[j] = 0.f;
  }
  float4 acc[kVec > 0 ? kVec : 1];
#pragma unroll
  for (int e = 0; e < kVec; ++e) acc[e] = make_float4(0.f, 0.f, 0.f, 0.f);
  // pass 2: weights of a chunk of NT slots, then the weighted sum of their outputs
  for (int base = 0; base < ns; base += NT) {
    const int s = base + tid;
    if (s < ns) {
      const long long sl = share_slot(c0 + s, sg.off, br.U, G);
      float v[G8];
      if (sl >= 0) {
        const float4 a = __ldcg(reinterpret_cast<const float4*>(p.part_lse + sl));
        const float4 b = __ldcg(reinterpret_cast<const float4*>(p.part_lse + sl) + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
      }
#pragma unroll
      for (int j = 0; j < G8; ++j) {
        const float w = (sl >= 0 && j < hcount) ? merge_exp2(p, v[j] - M[j]) : 0.f;
        den[j] += w;
        s_w[tid][j] = w;
      }
      s_sl[tid] = sl >= 0 ? sl : sl0;  // an empty block: weight 0 on a written slot
    }
    __syncthreads();
    const int cnt = min(NT, ns - base);
#pragma unroll
    for (int e = 0; e < kVec; ++e) {
      const int v = tid + e * NT;
      if (v < hcount * D4) {
        const int j = v / D4, d4 = v - j * D4;
        float4 a = acc[e];
#pragma unroll 8
        for (int i = 0; i < cnt; ++i) {
          const float w = s_w[i][j];
          const float4 o = __ldcg(reinterpret_cast<const float4*>(p.part_o + (s_sl[i] + j) * D) + d4);
          a.x += w * o.x;
          a.y += w * o.y;
          a.z += w * o.z;
          a.w += w * o.w;
        }
        acc[e] = a;
      }
    }
    __syncthreads();
  }
  // per-head sum of the weights
#pragma unroll
  for (int j = 0; j < G8; ++j) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den[j] += __shfl_xor_sync(0xffffffffu, den[j], o);
    if (lane == 0) s_red[wid][j] = den[j];
  }
  __syncthreads();
  if (tid < G8) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) t += s_red[w][tid];
    s_den[tid] = t;
  }
  __syncthreads();
#pragma unroll
  for (int e = 0; e < kVec; ++e) {
    const int v = tid + e * NT;
    if (v < hcount * D4) {
      const int j = v / D4, d4 = v - j * D4;
      const int hq = hq0 + j;
      const bool empty = !(s_M[j] > kEmptyM);
      const SinkAdj sa = p.sink ? apply_sink(p, hq, empty ? kEmptyM : s_M[j] + log2f(s_den[j]))
                                : SinkAdj{1.f, empty ? kEmptyM : s_M[j] + log2f(s_den[j])};
      const float sc = empty ? 0.f : p.out_scale / s_den[j] * sa.scale;
      const size_t o = ((size_t)sg.b * p.H_qo + hq) * D + 4 * d4;
      store_out(p, o + 0, acc[e].x * sc);
      store_out(p, o + 1, acc[e].y * sc);
      store_out(p, o + 2, acc[e].z * sc);
      store_out(p, o + 3, acc[e].w * sc);
      if (d4 == 0) p.lse[(size_t)sg.b * p.H_qo + hq] = sa.lse;
    }
  }
}

// Finish this block's share [ua, ub) of segment `sg` (heads [hq0, hq0 + hcount)):
// merge the NWS warp states in shared memory (sm_m/sm_d [NWS][8], sm_o [NWS][8][D],
// unnormalised O, log2 m).  A whole segment writes out/lse; otherwise the block
// writes its partial (O/d, lse) into slot 2c + side (side 0: the segment is this
// block's first, 1: its last), adds its units to the segment's counter, and the block
// that completes the count merges every partial of the segment (S-way merge_state).
// Ends with a block barrier (shared memory is reusable afterwards).
template <int NT, int NWS>
__device__ void finish_share(const DecodeParams& p, const BlockRange& br, const Segment& sg,
                             int ua, int ub, int hq0, int hcount, const float* sm_m,
                             const float* sm_d, const float* sm_o) {
  __shared__ int s_last;
  const int D = p.D;
  const int tid = threadIdx.x;
  const bool whole = (ua == 0 && ub == sg.n);
  const long long c = blockIdx.x;
  const int side = (sg.off <= br.x0) ? 0 : 1;
  const size_t slot = (size_t)(2 * c + side) * kMaxGroupPerCta;
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
    if (whole) {
      const SinkAdj sa = p.sink ? apply_sink(p, hq, l) : SinkAdj{1.f, l};
      store_out(p, ((size_t)sg.b * p.H_qo + hq) * D + d, o * p.out_scale * sa.scale);
      if (d == 0) p.lse[(size_t)sg.b * p.H_qo + hq] = sa.lse;
    } else {
      p.part_o[(slot + j) * D + d] = o;
      if (d == 0) p.part_lse[slot + j] = l;
    }
  }
  if (whole) {
    __syncthreads();
    return;
  }
  fence_acq_rel_gpu();
  __syncthreads();
  if (tid == 0) {
    int* cnt = p.counters + (size_t)sg.b * p.H_kv * p.n_z + sg.hz;
    const int mine = ub - ua;
    const int prev = atomicAdd(cnt, mine);
    s_last = (prev + mine == sg.n);
    if (s_last) *cnt = 0;  // every other share of this segment has arrived: reset for reuse
  }
  __syncthreads();
  if (s_last) {
    fence_acq_rel_gpu();
    merge_segment<NT>(p, br, sg, hq0, hcount);
  }
  __syncthreads();
}

}  // namespace pd
