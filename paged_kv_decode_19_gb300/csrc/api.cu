// Host side of libpageddecode: argument validation, the split planner, workspace
// and error-word management and kernel dispatch.  Every entry point of
// include/pageddecode.h is defined here, except pd_batch_decode_paged_kv_noalloc
// (decode_noalloc.cu), which calls pd_batch_decode_paged_kv.
#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "arena.h"
#include "kernels.h"
#include "pageddecode.h"

namespace pd {

// Split planner: the balanced schedule runs one resident wave of blocks (SMs x blocks
// per SM); an explicit split count n > 1 asks for about n blocks per (sequence, head
// slice) segment, capped at kMaxWaves resident waves.
constexpr int kMaxWaves = 8;
#ifndef PD_SEG_COST_TILES
#define PD_SEG_COST_TILES 4
#endif
// Cost of a segment's set-up and finish in the tensor-core schedule, in 16-row tiles
// (measured: a warp crossing a segment boundary loses about 4-6 tiles' time).
constexpr int kSegCostTiles = PD_SEG_COST_TILES;
constexpr size_t kWsAlign = 256;

static thread_local std::string t_last_error;
static thread_local const char* t_last_variant = "none";

static pd_status fail(pd_status st, const std::string& msg) {
  t_last_error = msg;
  return st;
}
// Lets the library's other translation units set the message of a failure they return.
void record_error(const char* msg) { t_last_error = msg; }

static pd_status cuda_fail(cudaError_t e, const char* what) {
  return fail(PD_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

// Device error word: one per device that loads the library.
static __device__ unsigned g_error_word;

struct DeviceState {
  bool ready = false;
  int num_sms = 0;
  unsigned* err = nullptr;
  // library-managed workspace: one arena per stream (arena.h); ws_mu is held from an
  // arena's hand-out until the kernel that uses it is enqueued
  std::mutex ws_mu;
  ArenaTable arenas;
  // resident blocks per SM of each kernel variant, queried once:
  // [mma][q_dtype][kv_dtype][D 64/128/256][kernel RoPE mode 0..4][single / multi-query /
  // pages of 8 rows]; 0 = not yet known
  int occupancy[2][4][4][3][5][3] = {};
};
constexpr int kMaxDevices = 64;
static DeviceState g_dev[kMaxDevices];
static std::mutex g_mu;

static pd_status device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(PD_ERR_CUDA, "device index out of range");
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& s = g_dev[dev];
  if (!s.ready) {
    e = cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    e = cudaGetSymbolAddress((void**)&s.err, g_error_word);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
    s.ready = true;
  }
  *out = &s;
  return PD_OK;
}

static int elem_bytes(int dt) {
  switch (dt) {
    case kF32: return 4;
    case kF16: return 2;
    case kBF16: return 2;
    case kE4M3: return 1;
  }
  return 0;
}

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Stream-ordered allocator operations of the per-stream workspace arenas.
static int arena_alloc(void*, void** p, size_t bytes, void* st) {
  return (int)cudaMallocAsync(p, bytes, (cudaStream_t)st);
}
static int arena_release(void*, void* p, void* st) { return (int)cudaFreeAsync(p, (cudaStream_t)st); }
static int arena_zero(void*, void* p, size_t bytes, void* st) {
  return (int)cudaMemsetAsync(p, 0, bytes, (cudaStream_t)st);
}
static const ArenaOps kCudaArenaOps = {nullptr, arena_alloc, arena_release, arena_zero};

// ---------------------------------------------------------------------------- validation
static pd_status validate_desc(const pd_decode_desc* d) {
  if (!d) return fail(PD_ERR_INVALID_ARG, "desc is NULL");
  if (d->B < 0) return fail(PD_ERR_INVALID_ARG, "B < 0");
  if (d->H_kv <= 0 || d->H_qo <= 0 || d->H_qo % d->H_kv != 0)
    return fail(PD_ERR_INVALID_ARG, "H_qo must be a positive multiple of H_kv");
  if (d->D != 64 && d->D != 128 && d->D != 256)
    return fail(PD_ERR_UNSUPPORTED, "head dim must be 64, 128 or 256");
  if (d->page_size <= 0 || d->page_size > 256) return fail(PD_ERR_INVALID_ARG, "page_size must be in [1, 256]");
  if (d->q_dtype != kF32 && d->q_dtype != kF16 && d->q_dtype != kBF16)
    return fail(PD_ERR_INVALID_ARG, "q_dtype must be F32, F16 or BF16");
  if (d->kv_dtype < kF32 || d->kv_dtype > kE4M3) return fail(PD_ERR_INVALID_ARG, "bad kv_dtype");
  if (d->out_dtype != kF32 && d->out_dtype != kF16 && d->out_dtype != kBF16)
    return fail(PD_ERR_INVALID_ARG, "out_dtype must be F32, F16 or BF16");
  if (d->max_pages <= 0 && d->B > 0) return fail(PD_ERR_INVALID_ARG, "max_pages must be positive");
  if (d->nnz_pages < 0) return fail(PD_ERR_INVALID_ARG, "nnz_pages < 0");
  if ((long long)d->max_pages * 2 * d->H_kv > INT_MAX)
    return fail(PD_ERR_UNSUPPORTED, "max_pages * 2 * H_kv exceeds 2^31");
  if (d->num_splits < 0) return fail(PD_ERR_INVALID_ARG, "num_splits < 0");
  if (d->flags & ~(PD_DECODE_EARLY_INPUTS | PD_DECODE_K_ROTATED))
    return fail(PD_ERR_INVALID_ARG, "unknown bits in flags");
  if (d->kv_dtype == kE4M3 && !(d->k_scale > 0.f && d->v_scale > 0.f && std::isfinite(d->k_scale) &&
                                std::isfinite(d->v_scale)))
    return fail(PD_ERR_INVALID_ARG, "E4M3 KV needs finite positive k_scale and v_scale");
  if (d->kv_dtype != d->q_dtype && d->kv_dtype != kE4M3)
    return fail(PD_ERR_UNSUPPORTED, "q_dtype must equal kv_dtype unless the cache is E4M3");
  return PD_OK;
}

// ---------------------------------------------------------------------------- planner
// Schedule, grid and workspace for `desc` with `wpb` independent workers per block
// (the tensor-core kernel's warps, or 1 for the SIMT kernel's blocks).  *mode:
// kSchedBalanced or kSchedPerSegment; *grid: blocks; workspace = per-segment arrival
// counters + two partial (lse, out) slots per worker.
// q_len: query tokens per sequence (multi-query decode); a segment's query columns
// (q_len x group per KV head) come in slices of at most kMaxGroupPerCta.
static void plan_impl(const pd_decode_desc* d, int num_sms, int ctas_per_sm, int wpb, int* mode,
                      int* grid, size_t* ws_bytes, int q_len = 1) {
  const int ncol = (d->H_qo / d->H_kv) * q_len;
  const int n_z = (ncol + kMaxGroupPerCta - 1) / kMaxGroupPerCta;
  const long long segments = (long long)d->B * d->H_kv * n_z;
  const long long wave = (long long)std::max(num_sms, 1) * std::max(ctas_per_sm, 1);
  wpb = std::max(wpb, 1);
  long long g;
  int m;
  if (d->num_splits == 1 || d->B == 0) {
    m = kSchedPerSegment;
    g = (segments + wpb - 1) / wpb;
  } else {
    m = kSchedBalanced;
    // upper bound on work units (pages touched per segment, plus one per sequence)
    const long long units = ((long long)d->nnz_pages + d->B) * d->H_kv * n_z;
    if (d->num_splits > 1) {
      const long long workers = std::min(segments * d->num_splits, wave * kMaxWaves * wpb);
      g = (workers + wpb - 1) / wpb;
    } else {
      g = wave;
    }
    g = std::max(1ll, std::min(g, (units + wpb - 1) / wpb));
  }
  size_t ws = 0;
  if (m == kSchedBalanced) {
    const size_t slots = (size_t)2 * g * wpb;
    ws = align_up((size_t)segments * sizeof(int), kWsAlign) +
         align_up(slots * kMaxGroupPerCta * sizeof(float), kWsAlign) +
         align_up(slots * kMaxGroupPerCta * d->D * sizeof(float), kWsAlign);
  }
  *mode = m;
  *grid = (int)std::min<long long>(g, INT_MAX);
  *ws_bytes = ws;
}

// Tensor-core variant eligibility (pages == nullptr: ignore the pointer's alignment).
static bool mma_path(const pd_decode_desc* d, const void* pages) {
  if ((reinterpret_cast<uintptr_t>(pages) & 15) != 0) return false;
  if (d->page_size % 16 != 0 && d->page_size != 8) return false;
  if (d->kv_dtype == kBF16 || d->kv_dtype == kF16) return d->D == 64 || d->D == 128;
  if (d->kv_dtype == kE4M3) return d->D == 128 && (d->q_dtype == kBF16 || d->q_dtype == kF16);
  return false;
}

static cudaError_t mma_dispatch(const DecodeParams& p, int q_dtype, int kv_dtype, dim3 grid,
                                cudaStream_t st, MmaConfig* cfg) {
  if (p.q_len > 1) {
    if (kv_dtype == kBF16) return launch_mma_mq_bf16(p, q_dtype, grid, st, cfg);
    if (kv_dtype == kF16) return launch_mma_mq_f16(p, q_dtype, grid, st, cfg);
    return launch_mma_mq_fp8(p, q_dtype, grid, st, cfg);
  }
  if (p.P == 8) {  // pages of 8 rows: two pages per 16-row tile
    if (kv_dtype == kBF16) return launch_mma_pair_bf16(p, q_dtype, grid, st, cfg);
    if (kv_dtype == kF16) return launch_mma_pair_f16(p, q_dtype, grid, st, cfg);
    return launch_mma_pair_fp8(p, q_dtype, grid, st, cfg);
  }
  if (kv_dtype == kBF16) return launch_mma_bf16(p, q_dtype, grid, st, cfg);
  if (kv_dtype == kF16) return launch_mma_f16(p, q_dtype, grid, st, cfg);
  return launch_mma_fp8(p, q_dtype, grid, st, cfg);
}

// Host plan: copy the caller's host indptr / length_info into the launch, with the
// prefix over the sequences of (work units + segment cost) that places the workers
// (the device's units_of on the same fields).  False when they do not fit.
static bool fill_host_plan(const pd_decode_desc& d, DecodeParams& p) {
  const int B = d.B;
  const long long li_n = d.sliding_window ? 3ll * B : (long long)B;
  if (2ll * (B + 1) + li_n > kHostPlanInts) return false;
  const int32_t* ip = d.host_indptr;
  const int32_t* li = d.host_length_info;
  p.hp_ptr = B + 1;
  p.hp_li = 2 * (B + 1);
  long long acc = 0;
  p.hp[0] = 0;
  for (int b = 0; b < B; ++b) {
    const long long off = d.sliding_window ? li[B + b] : 0, sk = d.sliding_window ? li[2 * B + b] : 0;
    bool bad = false;
    const SeqInfo s = seq_from(ip[b], ip[b + 1], li[b], off, sk, d.page_size, d.sliding_window != 0, bad);
    acc += units_of(s, d.page_size) + p.seg_cost;
    if (acc > INT_MAX) return false;
    p.hp[b + 1] = (int32_t)acc;
    p.hp[p.hp_ptr + b] = ip[b];
  }
  p.hp[p.hp_ptr + B] = ip[B];
  for (long long i = 0; i < li_n; ++i) p.hp[p.hp_li + i] = li[i];
  p.hp_B = B;
  return true;
}

// Fixed-point RoPE frequencies: F_i = 2^64 * frac(rope_scale / rope_theta^(2i/D) / (2 pi)).
static void rope_table(float rope_scale, float rope_theta, int D, unsigned long long* F) {
  const double two_pi = 6.283185307179586476925286766559;
  for (int i = 0; i < D / 2; ++i) {
    const double x = (double)rope_scale * std::pow((double)rope_theta, -2.0 * i / D) / two_pi;
    const double f = x - std::floor(x);
    double s = std::ldexp(f, 64);
    if (s >= 18446744073709551616.0) s = 0.0;
    F[i] = (unsigned long long)s;
  }
}

}  // namespace pd

using namespace pd;

extern "C" {

int32_t pd_version(void) { return 10100; }

const char* pd_get_last_error_string(void) { return t_last_error.c_str(); }

const char* pd_last_decode_variant(void) { return t_last_variant; }

pd_status pd_plan(const pd_decode_desc* desc, int32_t num_sms, int32_t ctas_per_sm,
                  int32_t* schedule, int32_t* grid_blocks, size_t* workspace_bytes) {
  pd_status st = validate_desc(desc);
  if (st != PD_OK) return st;
  if (!schedule || !grid_blocks || !workspace_bytes) return fail(PD_ERR_INVALID_ARG, "NULL output");
  plan_impl(desc, num_sms, ctas_per_sm, mma_path(desc, nullptr) ? kMmaWarps : 1, schedule,
            grid_blocks, workspace_bytes);
  return PD_OK;
}

// rm: the kernel's RoPE mode: 0 none, 1 / 2 rotate-half / interleaved on Q and K, 3 / 4
// the same on Q only (the cache holds K rotated).
static pd_status occupancy_for(const pd_decode_desc* d, bool use_mma, int rm, int* ctas,
                               DeviceState* ds = nullptr, int q_len = 1) {
  const int di = d->D == 64 ? 0 : d->D == 128 ? 1 : 2;
  const int mq = q_len > 1 ? 1 : (use_mma && d->page_size == 8 ? 2 : 0);
  int* cached = ds ? &ds->occupancy[use_mma ? 1 : 0][d->q_dtype & 3][d->kv_dtype & 3][di][rm][mq]
                   : nullptr;
  if (cached && *cached > 0) {
    *ctas = *cached;
    return PD_OK;
  }
  DecodeParams p{};
  p.D = d->D;
  p.P = d->page_size;
  p.rotary = rm > 2 ? rm - 2 : rm;
  p.k_rotated = rm > 2 ? 1 : 0;
  p.q_len = q_len;
  cudaError_t e;
  int n = 0;
  if (use_mma) {
    MmaConfig cfg{};
    e = mma_dispatch(p, d->q_dtype, d->kv_dtype, dim3(1), nullptr, &cfg);
    n = cfg.ctas_per_sm;
  } else {
    if (!simt_supports(d->q_dtype, d->kv_dtype, d->D)) return fail(PD_ERR_UNSUPPORTED, "dtype / head-dim combination");
    e = launch_decode_simt(p, d->q_dtype, d->kv_dtype, dim3(1), nullptr, &n);
  }
  if (e != cudaSuccess) return cuda_fail(e, "occupancy query");
  *ctas = std::max(n, 1);
  if (cached) *cached = *ctas;
  return PD_OK;
}

static size_t workspace_size_q(const pd_decode_desc* desc, int q_len) {
  if (validate_desc(desc) != PD_OK || q_len < 1) return 0;
  DeviceState* ds = nullptr;
  if (device_state(&ds) != PD_OK) return 0;
  // the largest plan over the variants a call with this desc may take
  size_t best = 0;
  for (int mma = 0; mma < 2; ++mma) {
    if (mma && !mma_path(desc, nullptr)) continue;
    if (!mma && q_len > 1) continue;  // the multi-query form runs on the tensor-core kernel only
    for (int rm = 0; rm < 5; ++rm) {
      int ctas = 1;
      if (occupancy_for(desc, mma != 0, rm, &ctas, ds, q_len) != PD_OK) continue;
      int mode, grid;
      size_t ws;
      plan_impl(desc, ds->num_sms, ctas, mma ? kMmaWarps : 1, &mode, &grid, &ws, q_len);
      best = std::max(best, ws);
    }
  }
  return best;
}

size_t pd_workspace_size(const pd_decode_desc* desc) { return workspace_size_q(desc, 1); }

size_t pd_workspace_size_mq(const pd_decode_desc* desc, int32_t q_len) {
  return workspace_size_q(desc, q_len);
}

pd_status pd_workspace_init(void* workspace, size_t bytes, pd_stream_t stream) {
  if (!workspace && bytes) return fail(PD_ERR_INVALID_ARG, "workspace is NULL");
  cudaError_t e = cudaMemsetAsync(workspace, 0, bytes, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
  return PD_OK;
}

}  // extern "C"

// Both decode entry points: q_len query tokens per sequence (1: batch_decode_paged_kv).
static pd_status decode_call(const void* Q, const void* pages, const int32_t* page_table_indptr,
                             const int32_t* page_table_values, const int32_t* length_info,
                             const int32_t* k_rope_pos_offset, const int32_t* q_rope_position,
                             void* output, float* lse, int q_len, int32_t rotary_mode,
                             float rope_scale, float rope_theta, float sm_scale,
                             const pd_decode_desc* desc, pd_stream_t stream) {
  pd_status st = validate_desc(desc);
  if (st != PD_OK) return st;
  const pd_decode_desc& d = *desc;
  if (rotary_mode < 0 || rotary_mode > 2) return fail(PD_ERR_INVALID_ARG, "rotary_mode must be 0, 1 or 2");
  if (rotary_mode != 0 && (!q_rope_position ||
                           (!k_rope_pos_offset && !(desc->flags & PD_DECODE_K_ROTATED))))
    return fail(PD_ERR_INVALID_ARG, "RoPE needs q_rope_position (and k_rope_pos_offset unless K is rotated)");
  if (rotary_mode != 0 && !(rope_theta > 0.f && std::isfinite(rope_theta) && std::isfinite(rope_scale)))
    return fail(PD_ERR_INVALID_ARG, "rope_theta must be finite and positive");
  if (!std::isfinite(sm_scale)) return fail(PD_ERR_INVALID_ARG, "sm_scale must be finite");
  if (d.B == 0) return PD_OK;
  if (!Q || !pages || !page_table_indptr || !length_info || !output || !lse)
    return fail(PD_ERR_INVALID_ARG, "NULL device pointer");
  if (d.nnz_pages > 0 && !page_table_values) return fail(PD_ERR_INVALID_ARG, "page_table_values is NULL");
  if (!d.host_indptr != !d.host_length_info)
    return fail(PD_ERR_INVALID_ARG, "host_indptr and host_length_info go together");
  if (d.host_indptr) {
    if (d.host_indptr[0] < 0 || d.host_indptr[d.B] > d.nnz_pages)
      return fail(PD_ERR_INVALID_ARG, "host_indptr outside [0, nnz_pages]");
    for (int b = 0; b < d.B; ++b)
      if (d.host_indptr[b + 1] < d.host_indptr[b]) return fail(PD_ERR_INVALID_ARG, "host_indptr decreases");
  }
  // both kernels read Q and K/V rows with vector accesses of up to 16 bytes
  if ((reinterpret_cast<uintptr_t>(pages) % 16) != 0 || (reinterpret_cast<uintptr_t>(Q) % 16) != 0)
    return fail(PD_ERR_INVALID_ARG, "Q and pages must be 16-byte aligned");

  DeviceState* ds = nullptr;
  st = device_state(&ds);
  if (st != PD_OK) return st;
  const bool use_mma = mma_path(desc, pages);
  if (q_len > 1 && (!use_mma || d.page_size % 16 != 0))
    return fail(PD_ERR_UNSUPPORTED, "multi-query decode runs on the tensor-core kernel only: "
                                    "f16/bf16 (D 64 or 128) or E4M3 (D 128) KV, page size a multiple of 16");
  int ctas = 1;
  const bool k_rotated = rotary_mode != 0 && (d.flags & PD_DECODE_K_ROTATED);
  st = occupancy_for(desc, use_mma, rotary_mode + (k_rotated ? 2 : 0), &ctas, ds, q_len);
  if (st != PD_OK) return st;
  int mode = 0, grid_blocks = 0;
  size_t ws_need = 0;
  const int wpb = use_mma ? kMmaWarps : 1;
  plan_impl(desc, ds->num_sms, ctas, wpb, &mode, &grid_blocks, &ws_need, q_len);
  if (grid_blocks == 0) return PD_OK;

  cudaStream_t s = (cudaStream_t)stream;
  const int group = d.H_qo / d.H_kv;
  const int ncol = group * q_len;
  const int n_z = (ncol + kMaxGroupPerCta - 1) / kMaxGroupPerCta;
  const size_t cnt_bytes = align_up((size_t)d.B * d.H_kv * n_z * sizeof(int), kWsAlign);
  const size_t lse_bytes = align_up((size_t)2 * grid_blocks * wpb * kMaxGroupPerCta * sizeof(float), kWsAlign);
  int* counters = nullptr;
  char* partials = nullptr;
  std::unique_lock<std::mutex> ws_lock;  // library workspace: held until the launch
  if (ws_need) {
    if (d.workspace) {
      // caller workspace: [counters][partial lse][partial out]; the counter prefix is
      // cleared on the stream every call, since a previous call with another layout
      // may have left partial results there.
      if (d.workspace_bytes < ws_need || (reinterpret_cast<uintptr_t>(d.workspace) % kWsAlign) != 0)
        return fail(PD_ERR_WORKSPACE, "caller workspace smaller than pd_workspace_size() or not 256-byte aligned");
      counters = (int*)d.workspace;
      partials = (char*)d.workspace + cnt_bytes;
      cudaError_t e = cudaMemsetAsync(counters, 0, cnt_bytes, s);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(counters)");
    } else {
      // library workspace: the arena of this stream (counters in one buffer, zero
      // between calls; partial results in another), grown stream-ordered; the device's
      // workspace lock stays held until the kernel is enqueued.  While the stream is
      // being captured into a graph its arena must already be large enough (nothing is
      // allocated behind the graph's back; a capturing stream's id cannot be queried).
      cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
      cudaError_t e = cudaStreamIsCapturing(s, &cap);
      if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
      unsigned long long sid = 0;
      if (cap == cudaStreamCaptureStatusNone) {
        e = cudaStreamGetId(s, &sid);
        if (e != cudaSuccess) return cuda_fail(e, "cudaStreamGetId");
      }
      ws_lock = std::unique_lock<std::mutex>(ds->ws_mu);
      void* cnt = nullptr;
      void* part = nullptr;
      if (cap != cudaStreamCaptureStatusNone) {
        if (ds->arenas.acquire_captured((void*)s, cnt_bytes, ws_need - cnt_bytes, &cnt, &part))
          return fail(PD_ERR_WORKSPACE,
                      "stream capture: the stream's library workspace is missing or too small; "
                      "make the same call on the stream once before capturing, or pass "
                      "desc->workspace");
      } else {
        const int rc = ds->arenas.acquire(sid, (void*)s, cnt_bytes, ws_need - cnt_bytes,
                                          kCudaArenaOps, &cnt, &part);
        if (rc) return cuda_fail((cudaError_t)rc, "library workspace (stream-ordered allocation)");
      }
      counters = (int*)cnt;
      partials = (char*)part;
    }
  }

  DecodeParams p{};
  p.Q = Q;
  p.pages = pages;
  p.indptr = page_table_indptr;
  p.values = page_table_values;
  p.length_info = length_info;
  p.k_rope_pos_offset = k_rope_pos_offset;
  p.q_rope_position = q_rope_position;
  p.out = output;
  p.lse = lse;
  if (ws_need) {
    p.counters = counters;
    p.part_lse = (float*)partials;
    p.part_o = (float*)(partials + lse_bytes);
  }
  p.err = ds->err;
  p.max_pages = d.max_pages;
  p.nnz_pages = d.nnz_pages;
  p.B = d.B;
  p.H_qo = d.H_qo;
  p.H_kv = d.H_kv;
  p.D = d.D;
  p.P = d.page_size;
  p.group = group;
  p.n_z = n_z;
  // two or four slices of a KV head's query columns: their warps walk the same pages
  // side by side in one block, so the pages come from HBM once
  p.zg = use_mma && mode == kSchedBalanced && (n_z == 2 || n_z == 4) ? n_z : 1;
  p.q_len = q_len;
  p.ncol = ncol;
  p.precise = d.kv_dtype == kF32 ? 1 : 0;
  p.window = d.sliding_window ? 1 : 0;
  p.rotary = rotary_mode;
  p.mode = mode;
  // tensor-core schedule: a segment's set-up and finish cost about kSegCostTiles tiles
  p.seg_cost = use_mma && mode == kSchedBalanced && kSegCostTiles > 0
                   ? std::max(1, kSegCostTiles * 16 / d.page_size) : 0;
  p.out_dtype = d.out_dtype;
  p.out_vec16 = (reinterpret_cast<uintptr_t>(output) % 16) == 0 ? 1 : 0;
  p.early_inputs = (d.flags & PD_DECODE_EARLY_INPUTS) ? 1 : 0;
  p.k_rotated = k_rotated ? 1 : 0;
  p.sink = d.sink;
  const double log2e = 1.4426950408889634073599246810019;
  const double kdeq = d.kv_dtype == kE4M3 ? (double)d.k_scale : 1.0;
  p.score_scale = (float)((double)sm_scale * log2e * kdeq);
  p.q_prescale = p.score_scale;
  p.out_scale = d.kv_dtype == kE4M3 ? d.v_scale : 1.f;
  if (rotary_mode) rope_table(rope_scale, rope_theta, d.D, p.rope_F);
  if (d.host_indptr && d.host_length_info) fill_host_plan(d, p);

  const dim3 grid((unsigned)grid_blocks);
  cudaError_t e;
  if (use_mma) {
    e = mma_dispatch(p, d.q_dtype, d.kv_dtype, grid, s, nullptr);
    t_last_variant = "mma";
  } else {
    if (!simt_supports(d.q_dtype, d.kv_dtype, d.D)) return fail(PD_ERR_UNSUPPORTED, "dtype / head-dim combination");
    e = launch_decode_simt(p, d.q_dtype, d.kv_dtype, grid, s);
    t_last_variant = "simt";
  }
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return PD_OK;
}

extern "C" {

pd_status pd_batch_decode_paged_kv(const void* Q, const void* pages,
                                   const int32_t* page_table_indptr,
                                   const int32_t* page_table_values, const int32_t* length_info,
                                   const int32_t* k_rope_pos_offset,
                                   const int32_t* q_rope_position, void* output, float* lse,
                                   int32_t rotary_mode, float rope_scale, float rope_theta,
                                   float sm_scale, const pd_decode_desc* desc,
                                   pd_stream_t stream) {
  return decode_call(Q, pages, page_table_indptr, page_table_values, length_info,
                     k_rope_pos_offset, q_rope_position, output, lse, 1, rotary_mode, rope_scale,
                     rope_theta, sm_scale, desc, stream);
}

pd_status pd_batch_decode_paged_kv_mq(const void* Q, const void* pages,
                                      const int32_t* page_table_indptr,
                                      const int32_t* page_table_values,
                                      const int32_t* length_info,
                                      const int32_t* k_rope_pos_offset,
                                      const int32_t* q_rope_position, void* output, float* lse,
                                      int32_t q_len, int32_t rotary_mode, float rope_scale,
                                      float rope_theta, float sm_scale,
                                      const pd_decode_desc* desc, pd_stream_t stream) {
  if (q_len < 1) return fail(PD_ERR_INVALID_ARG, "q_len must be >= 1");
  if (desc && desc->sliding_window)
    return fail(PD_ERR_UNSUPPORTED, "multi-query decode has no sliding-window form");
  if (desc && (long long)desc->B * q_len > INT_MAX) return fail(PD_ERR_UNSUPPORTED, "B * q_len exceeds 2^31");
  return decode_call(Q, pages, page_table_indptr, page_table_values, length_info,
                     k_rope_pos_offset, q_rope_position, output, lse, q_len, rotary_mode,
                     rope_scale, rope_theta, sm_scale, desc, stream);
}

pd_status pd_merge_state_inplace(void* V, float* S, const void* V_other, const float* S_other,
                                 int32_t N, int32_t H, int32_t D, int32_t v_dtype,
                                 pd_stream_t stream) {
  if (N < 0 || H < 0 || D <= 0) return fail(PD_ERR_INVALID_ARG, "bad N/H/D");
  if (v_dtype != kF32 && v_dtype != kF16 && v_dtype != kBF16)
    return fail(PD_ERR_INVALID_ARG, "v_dtype must be F32, F16 or BF16");
  if ((long long)N * H == 0) return PD_OK;
  if (!V || !S || !V_other || !S_other) return fail(PD_ERR_INVALID_ARG, "NULL device pointer");
  cudaError_t e = launch_merge_state(V, S, V_other, S_other, N, H, D, v_dtype, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  return PD_OK;
}

pd_status pd_merge_states(void* V_out, float* S_out, const float* V_parts, const float* S_parts,
                          int64_t v_rank_stride, int64_t s_rank_stride, int32_t R, int32_t N,
                          int32_t H, int32_t D, int32_t out_dtype, pd_stream_t stream) {
  if (R < 1 || N < 0 || H < 0 || D <= 0) return fail(PD_ERR_INVALID_ARG, "bad R/N/H/D");
  if (out_dtype != kF32 && out_dtype != kF16 && out_dtype != kBF16)
    return fail(PD_ERR_INVALID_ARG, "out_dtype must be F32, F16 or BF16");
  const long long rows = (long long)N * H;
  if (rows == 0) return PD_OK;
  if (rows > INT_MAX || (long long)R * rows > INT_MAX) return fail(PD_ERR_UNSUPPORTED, "R * N * H exceeds 2^31");
  if (!V_out || !S_out || !V_parts || !S_parts) return fail(PD_ERR_INVALID_ARG, "NULL device pointer");
  if (v_rank_stride != rows * D || s_rank_stride != rows) {
    // strided partners (one packed buffer per rank): the kernel reads partner r at
    // V_parts + r * v_rank_stride; it is given contiguous strides below, so only the
    // packed layout [R][N*H*D + N*H] of the exchange and the plain [R,N,H,D] are taken
    if (!(v_rank_stride == s_rank_stride && v_rank_stride == rows * D + rows &&
          S_parts == V_parts + rows * D))
      return fail(PD_ERR_INVALID_ARG,
                  "partner strides must be [R,N,H,D] / [R,N,H], or one packed [out | lse] block per partner");
  }
  cudaError_t e = launch_merge_states(V_out, S_out, V_parts, S_parts, R, (int)N, H, D, out_dtype,
                                      v_rank_stride, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "merge_states launch");
  return PD_OK;
}

pd_status pd_cp_shard_plan(const int32_t* indptr, const int32_t* values, const int32_t* length_info,
                           const int32_t* k_rope_pos_offset, int32_t B, int32_t page_size,
                           int32_t world, int32_t rank, int32_t* shard_indptr,
                           int32_t* shard_values, int64_t shard_values_capacity,
                           int32_t* shard_length_info, int32_t* shard_k_rope_pos_offset) {
  if (B < 0 || page_size <= 0 || world < 1 || rank < 0 || rank >= world)
    return fail(PD_ERR_INVALID_ARG, "bad B / page_size / world / rank");
  if (!shard_indptr || (B > 0 && (!indptr || !length_info || !shard_length_info || !shard_k_rope_pos_offset)))
    return fail(PD_ERR_INVALID_ARG, "NULL host pointer");
  shard_indptr[0] = 0;
  long long n = 0;
  for (int b = 0; b < B; ++b) {
    const long long npg = (long long)indptr[b + 1] - indptr[b];
    if (npg < 0) return fail(PD_ERR_INVALID_ARG, "page_table_indptr decreases");
    const long long per = npg > 0 ? (npg + world - 1) / world : 1;
    const long long p0 = std::min(npg, rank * per), p1 = std::min(npg, (rank + 1) * per);
    const long long L = npg > 0 ? (npg - 1) * page_size + length_info[b] : 0;
    if (npg > 0 && (length_info[b] < 1 || length_info[b] > page_size))
      return fail(PD_ERR_INVALID_ARG, "last_page_len outside [1, page_size]");
    if (p1 > p0) {
      if (!values || !shard_values) return fail(PD_ERR_INVALID_ARG, "NULL page table");
      if (n + (p1 - p0) > shard_values_capacity)
        return fail(PD_ERR_INVALID_ARG, "shard_values_capacity too small");
      for (long long j = p0; j < p1; ++j) shard_values[n++] = values[indptr[b] + j];
      const long long rows = std::min(L, p1 * page_size) - p0 * page_size;
      shard_length_info[b] = (int32_t)(rows - (p1 - p0 - 1) * page_size);
    } else {
      shard_length_info[b] = 0;
    }
    if (n > INT_MAX) return fail(PD_ERR_UNSUPPORTED, "shard page table exceeds 2^31 entries");
    shard_indptr[b + 1] = (int32_t)n;
    shard_k_rope_pos_offset[b] =
        (int32_t)((k_rope_pos_offset ? (long long)k_rope_pos_offset[b] : 0) + p0 * page_size);
  }
  return PD_OK;
}

}  // extern "C"

static pd_status append_call(void* pages, const void* k_new, const void* v_new,
                             const int64_t* slot_mapping, int32_t T, int32_t H_kv, int32_t D,
                             int32_t page_size, int64_t max_pages, int32_t in_dtype,
                             int32_t kv_dtype, float k_scale, float v_scale,
                             const int32_t* positions, int32_t rotary_mode, float rope_scale,
                             float rope_theta, pd_stream_t stream) {
  if (rotary_mode < 0 || rotary_mode > 2) return fail(PD_ERR_INVALID_ARG, "rotary_mode must be 0, 1 or 2");
  if (rotary_mode && (D % 2 || D / 2 > kMaxHalfDim))
    return fail(PD_ERR_UNSUPPORTED, "RoPE append needs an even head dim of at most 256");
  if (rotary_mode && !(rope_theta > 0.f && std::isfinite(rope_theta) && std::isfinite(rope_scale)))
    return fail(PD_ERR_INVALID_ARG, "rope_theta must be finite and positive");
  if (rotary_mode && T > 0 && !positions) return fail(PD_ERR_INVALID_ARG, "RoPE append needs positions");
  if (T < 0 || H_kv <= 0 || D <= 0 || page_size <= 0 || max_pages <= 0)
    return fail(PD_ERR_INVALID_ARG, "bad T/H_kv/D/page_size/max_pages");
  if (in_dtype != kF32 && in_dtype != kF16 && in_dtype != kBF16)
    return fail(PD_ERR_INVALID_ARG, "in_dtype must be F32, F16 or BF16");
  if (kv_dtype < kF32 || kv_dtype > kE4M3) return fail(PD_ERR_INVALID_ARG, "bad kv_dtype");
  if (kv_dtype == kE4M3 && !(k_scale > 0.f && v_scale > 0.f && std::isfinite(k_scale) && std::isfinite(v_scale)))
    return fail(PD_ERR_INVALID_ARG, "E4M3 cache needs finite positive k_scale and v_scale");
  if ((long long)T * H_kv > INT_MAX) return fail(PD_ERR_UNSUPPORTED, "T * H_kv too large");
  if (T == 0) return PD_OK;
  if (!pages || !k_new || !v_new || !slot_mapping) return fail(PD_ERR_INVALID_ARG, "NULL device pointer");
  DeviceState* ds = nullptr;
  pd_status st = device_state(&ds);
  if (st != PD_OK) return st;
  AppendRope rope{};
  rope.positions = positions;
  rope.mode = rotary_mode;
  if (rotary_mode) rope_table(rope_scale, rope_theta, D, rope.F);
  cudaError_t e = launch_append(pages, k_new, v_new, slot_mapping, T, H_kv, D, page_size, max_pages,
                                in_dtype, kv_dtype, k_scale, v_scale, ds->err, rope, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "append launch");
  return PD_OK;
}

extern "C" {

pd_status pd_append_paged_kv(void* pages, const void* k_new, const void* v_new,
                             const int64_t* slot_mapping, int32_t T, int32_t H_kv, int32_t D,
                             int32_t page_size, int64_t max_pages, int32_t in_dtype,
                             int32_t kv_dtype, float k_scale, float v_scale, pd_stream_t stream) {
  return append_call(pages, k_new, v_new, slot_mapping, T, H_kv, D, page_size, max_pages, in_dtype,
                     kv_dtype, k_scale, v_scale, nullptr, 0, 1.f, 1e4f, stream);
}

pd_status pd_append_paged_kv_rope(void* pages, const void* k_new, const void* v_new,
                                  const int64_t* slot_mapping, const int32_t* positions,
                                  int32_t T, int32_t H_kv, int32_t D, int32_t page_size,
                                  int64_t max_pages, int32_t in_dtype, int32_t kv_dtype,
                                  float k_scale, float v_scale, int32_t rotary_mode,
                                  float rope_scale, float rope_theta, pd_stream_t stream) {
  if (rotary_mode != 1 && rotary_mode != 2) return fail(PD_ERR_INVALID_ARG, "rotary_mode must be 1 or 2");
  return append_call(pages, k_new, v_new, slot_mapping, T, H_kv, D, page_size, max_pages, in_dtype,
                     kv_dtype, k_scale, v_scale, positions, rotary_mode, rope_scale, rope_theta,
                     stream);
}

pd_status pd_release_stream_workspace(pd_stream_t stream) {
  DeviceState* ds = nullptr;
  pd_status st = device_state(&ds);
  if (st != PD_OK) return st;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing((cudaStream_t)stream, &cap);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
  if (cap != cudaStreamCaptureStatusNone)
    return fail(PD_ERR_INVALID_ARG, "the workspace of a stream is not released while it is being captured");
  unsigned long long sid = 0;
  e = cudaStreamGetId((cudaStream_t)stream, &sid);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamGetId");
  std::lock_guard<std::mutex> lk(ds->ws_mu);
  const int rc = ds->arenas.release(sid, (void*)stream, kCudaArenaOps);
  if (rc) return cuda_fail((cudaError_t)rc, "cudaFreeAsync (stream workspace)");
  return PD_OK;
}

pd_status pd_check_device_errors(pd_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  DeviceState* ds = nullptr;
  pd_status st = device_state(&ds);
  if (st != PD_OK) return st;
  unsigned word = 0;
  e = cudaMemcpy(&word, ds->err, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read error word");
  if (word) {
    const unsigned zero = 0;
    e = cudaMemcpy(ds->err, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "clear error word");
  }
  if (word & kErrBadPage) return fail(PD_ERR_BAD_PAGE, "a page id or sequence offset was out of range");
  if (word & kErrBadLength) return fail(PD_ERR_BAD_LENGTH, "inconsistent length_info or split-plan overflow");
  if (word & kErrBadSlot) return fail(PD_ERR_BAD_SLOT, "an append slot was beyond the cache");
  if (word & kErrTimeout) return fail(PD_ERR_TIMEOUT, "a pipeline wait timed out");
  return PD_OK;
}

}  // extern "C"
