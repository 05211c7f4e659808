/*
 * libpageddecode — single-token (decode) attention over a paged KV cache, for
 * NVIDIA GB300 (sm_103a).  Plain C ABI: device pointers, sizes and a CUDA stream.
 *
 * The operations follow three published descriptions of the problem:
 *   [TVM]  Apache TVM, python/tvm/relax/frontend/nn/llm/_decode_kernels.py —
 *          `batch_decode_paged_kv` (argument list, page layout, length_info,
 *          RoPE arguments, base-2 log-sum-exp) and `merge_state_inplace`.
 *   [VLLM] vllm-cpu 0.8.5, vllm/attention/ops/nki_flash_attn.py — `reshape_and_cache`
 *          (writing new tokens' K/V into their cache slots).
 *   [NKI]  NKI Attention Block TKG Kernel API Reference — FP8 KV cache with
 *          per-tensor `k_scale` / `v_scale`, OCP e4m3fn (max 448), and the
 *          sentinel slot that skips a cache write.
 *
 * Conventions shared by every entry point:
 *   - Every pointer argument is a DEVICE pointer owned by the caller unless noted;
 *     the library never frees or retains it beyond the call.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream) and
 *     return a status; no exception or abort crosses the ABI.
 *   - Host-side argument errors return PD_ERR_INVALID_ARG / PD_ERR_UNSUPPORTED
 *     before anything is launched.  Problems only visible on the device (a page id
 *     outside [0, max_pages), inconsistent lengths, a slot beyond the cache) never
 *     trap: the offending rows/tokens are skipped and a device error word records
 *     them; `pd_check_device_errors` reports and clears it.
 *   - `lse` is always float32 in log2 units: lse = log2(sum_r 2^(s_r)), where
 *     s_r = sm_scale * log2(e) * q.k_r.
 */
#ifndef PAGEDDECODE_H_
#define PAGEDDECODE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque CUDA stream (binary-compatible with cudaStream_t / CUstream). */
typedef struct CUstream_st* pd_stream_t;

typedef enum {
  PD_OK = 0,
  PD_ERR_INVALID_ARG = 1,   /* bad pointer / shape / dtype combination (host check) */
  PD_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. odd head dim) */
  PD_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed */
  PD_ERR_BAD_PAGE = 4,      /* device: a page id or sequence offset was out of range */
  PD_ERR_BAD_LENGTH = 5,    /* device: length_info inconsistent, or more KV chunks than planned */
  PD_ERR_BAD_SLOT = 6,      /* device: an append slot lay beyond max_pages*page_size */
  PD_ERR_TIMEOUT = 7,       /* device: reserved (the current kernels have no waits) */
  PD_ERR_WORKSPACE = 8      /* caller workspace too small or misaligned */
} pd_status;

/* Element types.  PD_E4M3 = OCP float8 e4m3fn (bias 7, max 448, no inf); KV only. */
typedef enum { PD_F32 = 0, PD_F16 = 1, PD_BF16 = 2, PD_E4M3 = 3 } pd_dtype;

/*
 * What [TVM] fixes when it builds a decode kernel (head counts, head dim, page
 * size, dtype, sliding-window variant), plus the FP8 scales of [NKI] and the
 * split controls of this library.
 */
typedef struct {
  int32_t B;                 /* number of sequences (one query token each) */
  int32_t H_qo;              /* query heads; must be a multiple of H_kv */
  int32_t H_kv;              /* KV heads; Q head h reads KV head h / (H_qo/H_kv) */
  int32_t D;                 /* head dim: 64, 128 or 256 */
  int32_t page_size;         /* rows per page, P: 1 to 256.  The tensor-core kernel runs
                                P = 8 or a multiple of 16 with F16/BF16 KV (D 64 or 128) or
                                E4M3 KV (D 128, 16-bit Q); every other accepted shape
                                runs on the SIMT kernel (pd_last_decode_variant) */
  int32_t q_dtype;           /* pd_dtype of Q: F32, F16 or BF16 */
  int32_t kv_dtype;          /* pd_dtype of pages: F32, F16, BF16 or E4M3 */
  int32_t out_dtype;         /* pd_dtype of output: F32, F16 or BF16 */
  int32_t sliding_window;    /* 0: length_info is [B] = last_page_len.
                                1: length_info is [3,B] = (last_page_len,
                                   window start offset, attention-sink length). */
  int32_t num_splits;        /* work split: 0 = balanced (one resident wave of blocks;
                                each worker -- a warp of the tensor-core kernel, a block
                                of the SIMT kernel -- takes an equal share of all pages
                                of all sequences and heads); 1 = one worker per
                                (sequence, <=8-head slice), never split; n > 1 =
                                balanced over about n workers per (sequence, head slice) */
  int64_t max_pages;         /* pages buffer holds [max_pages,2,H_kv,P,D] */
  int64_t nnz_pages;         /* entries in page_table_values (= indptr[B]) */
  int32_t max_kv_len_hint;   /* reserved (ignored); set to 0 */
  float k_scale;             /* E4M3 KV only: K = code * k_scale (else ignored) */
  float v_scale;             /* E4M3 KV only: V = code * v_scale (else ignored) */
  int32_t flags;             /* 0, or PD_DECODE_EARLY_INPUTS | PD_DECODE_K_ROTATED (below) */
  void* workspace;           /* optional caller workspace (device, 256-byte aligned);
                                NULL = library-managed */
  size_t workspace_bytes;    /* size of `workspace` */
  const float* sink;         /* optional device array [H_qo] float32, or NULL: a learned
                                logit per query head ([NKI] `sink`), in natural units,
                                that joins the softmax as one more score with a zero value
                                row -- out = sum_r e^(t_r) v_r / (e^sink + sum_r e^(t_r)),
                                t_r = sm_scale q.k_r, and lse includes it (an empty
                                sequence gives out = 0, lse = sink * log2(e)) */
  const int32_t* host_indptr;       /* optional HOST copy of page_table_indptr [B+1], or NULL */
  const int32_t* host_length_info;  /* optional HOST copy of length_info ([B] or [3,B]), or NULL.
                                 Both or neither.  When given (and 2(B+1) plus the length_info
                                 entries fit in 1024 ints), the decode uses these instead of
                                 the device arrays: the split is planned on the host and the
                                 sequences' lengths and page-table offsets travel inside the
                                 kernel launch, so no kernel reads page_table_indptr or
                                 length_info and the start-up scan of them is skipped (the
                                 serving scheduler that builds these arrays holds them on the
                                 host anyway).  Read during the call only.  Page-table reads
                                 stay bounds-checked against nnz_pages. */
} pd_decode_desc;

/*
 * Launch order.  Every kernel of this library is launched with programmatic stream
 * serialisation (CUDA programmatic dependent launch): it may be scheduled while the
 * kernel before it on the stream is finishing, and it waits for that kernel to complete
 * before it reads any caller memory or writes anything.  Results are the same as with
 * plain stream order.
 * PD_DECODE_EARLY_INPUTS in desc->flags lets the decode read Q, page_table_indptr,
 * page_table_values, length_info and the RoPE positions while the previous kernel on
 * the stream still runs; only its page reads and its writes wait for that kernel.
 * The caller asserts that the kernel enqueued just before the decode writes none of
 * those inputs, and that everything enqueued before that kernel is complete once it
 * starts: both hold when it is pd_append_paged_kv (which writes only the pages and,
 * itself, waits for its predecessor before it lets the decode start).  The decode then
 * runs its start-up (work split scan, page-table and Q loads) under the append.
 */
#define PD_DECODE_EARLY_INPUTS 1

/*
 * PD_DECODE_K_ROTATED in desc->flags (with rotary_mode 1 or 2): the cache holds every
 * K row already rotated at its position, as pd_append_paged_kv_rope writes it ([NKI]
 * TKG: RoPE, then the KV cache update).  The decode then rotates only Q (at
 * q_rope_position, per rotary_mode) and uses K as stored: each row is read once
 * without the per-row rotation, so the RoPE path costs what the plain one does.
 * k_rope_pos_offset is not read.  Ignored when rotary_mode is 0.
 */
#define PD_DECODE_K_ROTATED 2

/*
 * batch_decode_paged_kv — [TVM] `batch_decode_paged_kv`.
 * For each sequence b and query head h (KV head hk = h / (H_qo/H_kv)):
 *   rows  r = 0 .. L_b-1, L_b from page_table_indptr and length_info:
 *         no window: L = (npages-1)*P + last_page_len, row r at sequence offset r;
 *         window:    L = (npages-1)*P + last_page_len - win_off + sink, row r at
 *                    offset r (r < sink) or r - sink + win_off.
 *   page  page_table_values[indptr[b] + off / P], slot off % P;
 *         K row = pages[page, 0, hk, slot, :], V row = pages[page, 1, hk, slot, :].
 *   RoPE  (rotary_mode == 1) rotate-half over the full head dim: frequency i
 *         rotates the pair (i, i + D/2) by the angle pos * rope_scale /
 *         rope_theta^(2i/D); Q at q_rope_position[b], K row r at
 *         k_rope_pos_offset[b] + r.  rotary_mode == 2: the interleaved layout of
 *         [NKI] (`rope_contiguous_layout` = False), frequency i rotating the pair
 *         (2i, 2i + 1) by the same angle.
 *   s_r = sm_scale * log2(e) * q.k_r;  out = sum_r 2^(s_r) v_r / sum_r 2^(s_r);
 *   lse = log2(sum_r 2^(s_r)).  An empty sequence gives out = 0, lse = -5e4.
 * Arguments (all device pointers):
 *   Q           [B, H_qo, D] desc->q_dtype, contiguous, 16-byte aligned.
 *   pages       [max_pages, 2, H_kv, P, D] desc->kv_dtype, contiguous, 16-byte aligned.
 *   page_table_indptr [B+1] int32, non-decreasing, indptr[0] = 0.
 *   page_table_values [nnz_pages] int32 physical page ids.
 *   length_info [B] or [3,B] int32 (see desc->sliding_window).
 *   k_rope_pos_offset, q_rope_position [B] int32; may be NULL when rotary_mode == 0.
 *   output      [B, H_qo, D] desc->out_dtype.   lse [B, H_qo] float32 (log2 units).
 * Scalars: rotary_mode (0 none, 1 RoPE rotate-half, 2 RoPE interleaved), rope_scale,
 * rope_theta, sm_scale.
 * Work is split by pages (see desc->num_splits); a (sequence, head slice) that
 * several workers share is merged on the device from their partial (out, lse) pairs
 * by the worker that completes its page count.  The grid uses only host-known sizes;
 * each block finds its workers' shares with a scan of indptr/length_info.
 * Q or pages not 16-byte aligned: PD_ERR_INVALID_ARG (both kernels read rows with
 * 16-byte vector loads).
 * Arithmetic: f16, bf16 and E4M3 caches run on tensor cores (fp32 accumulation, Q
 * split into hi + lo 16-bit parts where it is not already of the cache's type, P
 * rounded to the cache's 16-bit type for P.V); with RoPE the rotated K is rounded
 * once to f16, so a bf16 cache must keep |k| below 46000.  f32 caches run an fp32
 * kernel without tensor cores.
 * Workspace: desc->workspace if non-NULL (at least pd_workspace_size(desc) bytes,
 * 256-byte aligned, zero-filled before its first use — see pd_workspace_init; the
 * caller must not let two calls that share it overlap on the GPU), otherwise the
 * library's workspace for `stream`: one arena per stream (per process-unique stream
 * id) on the current device, allocated stream-ordered (cudaMallocAsync) on the first
 * split call on that stream and grown stream-ordered when a larger batch needs more
 * (the new buffer is allocated first, the old one released with cudaFreeAsync on the
 * stream, after the work already enqueued there).  So decodes in flight on different
 * streams never share split scratch, and any host threads may call concurrently; a
 * per-device lock is held from the arena's hand-out until the kernel is enqueued.
 * CUDA-graph capture: while `stream` is being captured the library allocates nothing;
 * it hands out the arena that the same stream handle last used outside capture, which
 * must already be large enough (make the same call, or a larger one, on the stream once
 * before capturing), else the call returns PD_ERR_WORKSPACE without enqueuing anything.
 * The graph keeps those buffers: replay it only while the stream's arena is neither
 * released nor grown, and replays must not overlap one another or other split decodes
 * on that stream's arena.  A caller workspace (desc->workspace) has no such conditions
 * beyond its own.  The split is planned on the device unless the host copies of the
 * page table are given, in which case the plan (and the lengths) are fixed in the
 * captured launch.  An arena lives until pd_release_stream_workspace(stream) or
 * process exit.
 * Returns PD_OK once the work is enqueued.
 */
pd_status pd_batch_decode_paged_kv(const void* Q, const void* pages,
                                   const int32_t* page_table_indptr,
                                   const int32_t* page_table_values, const int32_t* length_info,
                                   const int32_t* k_rope_pos_offset,
                                   const int32_t* q_rope_position, void* output, float* lse,
                                   int32_t rotary_mode, float rope_scale, float rope_theta,
                                   float sm_scale, const pd_decode_desc* desc,
                                   pd_stream_t stream);

/*
 * pd_batch_decode_paged_kv_noalloc — no counterpart in the source papers; an addition
 * of this library for callers that cannot allocate device memory.  Some programs may
 * not call cudaMalloc at all once they are running: a serving process that reserved
 * all free HBM for its KV-cache pool at start-up (a later allocation would fail), a
 * plug-in that lives inside a host framework that owns every device allocation, or a
 * latency-critical loop that cannot afford the allocator's implicit synchronisation.
 * This entry point computes exactly what pd_batch_decode_paged_kv computes, with the
 * same arguments, but it never allocates: the split scratch (arrival counters and
 * partial out/lse) is one static 16 MiB device array inside the library, present on
 * every GPU that loads it until the process exits.
 *   - desc->workspace must be NULL.
 *   - If the batch would need more than 16 MiB of split scratch (about
 *     64 * grid_blocks * (D + 1) bytes plus 4 bytes per (sequence, head slice), see
 *     pd_workspace_size), the call returns PD_ERR_WORKSPACE without launching; lower
 *     desc->num_splits or use pd_batch_decode_paged_kv.
 *   - The first call on a device looks up the array's device address (a
 *     cudaGetSymbolAddress, once per device, with that device current); make that
 *     first call before any CUDA-graph stream capture.
 *   - All calls share the one array: the counters are cleared on `stream` at the start
 *     of every call, and the array keeps the last call's partials.  Two calls whose
 *     work overlaps on the GPU (different streams, or different host threads without
 *     ordering) race on it and give undefined results; serialise them.
 * Returns the same statuses as pd_batch_decode_paged_kv.
 */
pd_status pd_batch_decode_paged_kv_noalloc(const void* Q, const void* pages,
                                           const int32_t* page_table_indptr,
                                           const int32_t* page_table_values,
                                           const int32_t* length_info,
                                           const int32_t* k_rope_pos_offset,
                                           const int32_t* q_rope_position, void* output,
                                           float* lse, int32_t rotary_mode, float rope_scale,
                                           float rope_theta, float sm_scale,
                                           const pd_decode_desc* desc, pd_stream_t stream);

/*
 * pd_batch_decode_paged_kv_mq — multi-query decode: q_len query tokens per sequence
 * (speculative decoding, small chunks of prefill), causal among the new tokens.  The
 * new tokens' K/V are already in the cache (pd_append_paged_kv): they are the last
 * q_len attended rows of each sequence.  Token t (0-based) of sequence b sees the
 * attended rows r < L_b - q_len + 1 + t: the cached context in full and the new tokens
 * up to itself, as the active part of the mask of [VLLM] `flash_paged_attention`
 * (context open, active tokens causal); a token with no row gives out = 0,
 * lse = -5e4.  Its RoPE position is q_rope_position[b] + t.  q_len = 1 computes
 * exactly pd_batch_decode_paged_kv.
 * Arguments as pd_batch_decode_paged_kv, except:
 *   Q      [B, q_len, H_qo, D] desc->q_dtype;  output [B, q_len, H_qo, D];
 *   lse    [B, q_len, H_qo] float32 (log2 units);  q_len >= 1.
 * The work unit is (sequence, KV head, slice of <= 8 query columns), a column being
 * one (token, head) of the KV head's group, so each KV page is read once for all
 * tokens and heads of a slice.  Runs on the tensor-core kernel only: f16/bf16 KV
 * (D 64 or 128) or E4M3 KV (D 128), page size a multiple of 16; otherwise
 * PD_ERR_UNSUPPORTED, as is desc->sliding_window != 0.  A caller workspace must hold
 * pd_workspace_size_mq(desc, q_len) bytes.
 */
pd_status pd_batch_decode_paged_kv_mq(const void* Q, const void* pages,
                                      const int32_t* page_table_indptr,
                                      const int32_t* page_table_values,
                                      const int32_t* length_info,
                                      const int32_t* k_rope_pos_offset,
                                      const int32_t* q_rope_position, void* output, float* lse,
                                      int32_t q_len, int32_t rotary_mode, float rope_scale,
                                      float rope_theta, float sm_scale,
                                      const pd_decode_desc* desc, pd_stream_t stream);

/*
 * merge_state_inplace — [TVM] `merge_state_inplace`.
 * For every (n, h):  m = max(S, S_o);  w = 2^(S - m);  w_o = 2^(S_o - m);
 *   V[n,h,:] <- V * w/(w+w_o) + V_other * w_o/(w+w_o);  S[n,h] <- log2(w + w_o) + m.
 * V, V_other [N, H, D] of v_dtype (F32, F16 or BF16), contiguous; S, S_other
 * [N, H] float32 (log2 units).  V and S are updated in place; arithmetic in fp32.
 * A partner with S_other = -5e4 and V_other = 0 leaves (V, S) unchanged.
 */
pd_status pd_merge_state_inplace(void* V, float* S, const void* V_other, const float* S_other,
                                 int32_t N, int32_t H, int32_t D, int32_t v_dtype,
                                 pd_stream_t stream);

/*
 * merge_states — the [TVM] `merge_state_inplace` formula over R partners at once, the
 * combine step of a decode split across R ranks (context parallelism, [NKI] `CP`: each
 * rank decodes its slice of the context to a partial (out, lse), the partials are
 * exchanged and combined) or across R chunks of one GPU's multi-stage decode.
 * For every (n, h):  M = max_r S_r;  w_r = 2^(S_r - M);
 *   V_out[n,h,:] = sum_r w_r V_r[n,h,:] / sum_r w_r;  S_out[n,h] = log2(sum_r w_r) + M.
 * If every partner is empty (S_r <= -5e4, the decode's empty-sequence state), V_out = 0
 * and S_out = -5e4.  Arithmetic in fp32.
 * Arguments (device pointers):
 *   V_parts  float32 partner outputs; partner r's [N, H, D] rows at V_parts + r * v_rank_stride.
 *   S_parts  float32 partner lse (log2); partner r's [N, H] at S_parts + r * s_rank_stride.
 *   Two layouts are accepted: separate arrays [R,N,H,D] / [R,N,H] (v_rank_stride = N*H*D,
 *   s_rank_stride = N*H), or one packed block [N*H*D outputs | N*H lse] per partner, as an
 *   all-gather of each rank's packed partial delivers it (v_rank_stride = s_rank_stride =
 *   N*H*(D+1), S_parts = V_parts + N*H*D); anything else is PD_ERR_INVALID_ARG.
 *   V_out    [N, H, D] of out_dtype (F32, F16 or BF16);  S_out [N, H] float32.
 * The outputs must not overlap the partners.
 */
pd_status pd_merge_states(void* V_out, float* S_out, const float* V_parts, const float* S_parts,
                          int64_t v_rank_stride, int64_t s_rank_stride, int32_t R, int32_t N,
                          int32_t H, int32_t D, int32_t out_dtype, pd_stream_t stream);

/*
 * cp_shard_plan — host-only (no CUDA call): the page table of one rank's slice of the
 * context for a decode split across `world` ranks ([NKI] `CP`: each rank holds an
 * S_ctx/CP slice of the prior KV cache), cut at page boundaries (TVM multi-stage
 * decoding's chunks are valid pseudo-sequences): sequence b's npages pages are cut
 * into `world` chunks of per = ceil(npages / world) pages, and rank `rank` takes pages
 * [rank * per, min((rank + 1) * per, npages)); a rank past the end of the list gets an
 * empty chunk (no pages, its decode gives the empty state, which the merge ignores).
 * The chunk is a sequence of its own: rows = min(L, p1 P) - p0 P, last page length
 * rows - (p1 - p0 - 1) P, and RoPE positions that start at k_rope_pos_offset[b] + p0 P,
 * so that every K row keeps its position.  Decode the rank's chunk with
 * pd_batch_decode_paged_kv (fp32 output) into a partial (out, lse), exchange the
 * partials, and combine them with pd_merge_states: the result equals the unsplit decode.
 * No sliding window (length_info is [B] last_page_len).
 * Arguments (HOST pointers): indptr [B+1], values [indptr[B]], length_info [B],
 * k_rope_pos_offset [B] or NULL (0); outputs shard_indptr [B+1], shard_values (room for
 * shard_values_capacity entries; at most ceil(npages/world) per sequence),
 * shard_length_info [B], shard_k_rope_pos_offset [B].  The page ids are the global
 * table's; a deployment whose ranks hold only their own slice maps them to its pool.
 */
pd_status pd_cp_shard_plan(const int32_t* indptr, const int32_t* values, const int32_t* length_info,
                           const int32_t* k_rope_pos_offset, int32_t B, int32_t page_size,
                           int32_t world, int32_t rank, int32_t* shard_indptr,
                           int32_t* shard_values, int64_t shard_values_capacity,
                           int32_t* shard_length_info, int32_t* shard_k_rope_pos_offset);

/*
 * append_paged_kv — [VLLM] `reshape_and_cache`, on the [TVM] page layout.
 * For token t with slot_mapping[t] = s >= 0:  page = s / P, off = s % P;
 *   pages[page, 0, h, off, :] = conv(k_new[t, h, :]);  pages[page, 1, h, off, :] = conv(v_new[t, h, :]).
 * conv: same dtype -> bit copy; E4M3 cache -> e4m3(x / scale) with an IEEE fp32
 * division (scale = k_scale for K, v_scale for V), round-to-nearest-even,
 * saturating to +-448; other conversions round to nearest even.
 * A negative slot skips the token ([NKI] sentinel).  A slot >= max_pages*P is
 * skipped and recorded as PD_ERR_BAD_SLOT in the device error word.
 * k_new, v_new [T, H_kv, D] of in_dtype (F32, F16, BF16); slot_mapping [T] int64;
 * pages [max_pages, 2, H_kv, P, D] of kv_dtype.  Two tokens with the same slot
 * race (last writer unspecified), as in the source.
 */
pd_status pd_append_paged_kv(void* pages, const void* k_new, const void* v_new,
                             const int64_t* slot_mapping, int32_t T, int32_t H_kv, int32_t D,
                             int32_t page_size, int64_t max_pages, int32_t in_dtype,
                             int32_t kv_dtype, float k_scale, float v_scale, pd_stream_t stream);

/*
 * append_paged_kv_rope — pd_append_paged_kv with each new K row rotated first, at
 * positions[t] (int32 [T], device), by rotary_mode 1 (rotate-half) or 2 (interleaved)
 * with the angles of pd_batch_decode_paged_kv's RoPE: the order of [NKI] TKG (RoPE,
 * then the KV cache update).  The rotation runs in fp32 with angles to fp32 accuracy;
 * the rotated values are then converted as in pd_append_paged_kv (E4M3: divided by
 * k_scale, RNE, saturating).  V rows are stored unrotated.  Decode such a cache with
 * PD_DECODE_K_ROTATED: only Q is rotated then.
 */
pd_status pd_append_paged_kv_rope(void* pages, const void* k_new, const void* v_new,
                                  const int64_t* slot_mapping, const int32_t* positions,
                                  int32_t T, int32_t H_kv, int32_t D, int32_t page_size,
                                  int64_t max_pages, int32_t in_dtype, int32_t kv_dtype,
                                  float k_scale, float v_scale, int32_t rotary_mode,
                                  float rope_scale, float rope_theta, pd_stream_t stream);

/*
 * Releases the library-managed decode workspace of `stream` on the current device
 * (stream-ordered: cudaFreeAsync on `stream`, after the work already enqueued there).
 * A later split decode on the stream allocates a new one.  Call it before destroying a
 * stream that ran split decodes with desc->workspace == NULL, if the process keeps
 * creating streams.  No arena for the stream: PD_OK, nothing is done.  A stream being
 * captured into a CUDA graph: PD_ERR_INVALID_ARG, nothing is done.
 */
pd_status pd_release_stream_workspace(pd_stream_t stream);

/* Bytes of workspace pd_batch_decode_paged_kv needs for `desc` on the current device
 * (0 on invalid desc).  Host-only apart from reading the device's SM count. */
size_t pd_workspace_size(const pd_decode_desc* desc);

/* The same for pd_batch_decode_paged_kv_mq with q_len query tokens per sequence. */
size_t pd_workspace_size_mq(const pd_decode_desc* desc, int32_t q_len);

/* Zero-fill a caller-provided workspace before its first use (enqueued on stream). */
pd_status pd_workspace_init(void* workspace, size_t bytes, pd_stream_t stream);

/*
 * Host-only split planner (no CUDA calls): for `desc` on a GPU with `num_sms`
 * multiprocessors and `ctas_per_sm` resident decode blocks, returns the schedule
 * (*schedule: 0 = balanced shares of all pages, 1 = one worker per (sequence, head
 * slice)), the number of blocks (*grid_blocks) and the workspace bytes (per-segment
 * arrival counters plus two partial (out, lse) slots per worker; 0 when nothing is
 * split).  Workers per block: 4 (warps) when desc selects the tensor-core kernel
 * (16-bit or E4M3 KV, page_size 8 or % 16 == 0, D = 64/128, D = 128 for E4M3), else 1.
 * Used by the library and exposed for tests.
 */
pd_status pd_plan(const pd_decode_desc* desc, int32_t num_sms, int32_t ctas_per_sm,
                  int32_t* schedule, int32_t* grid_blocks, size_t* workspace_bytes);

/* Synchronises `stream`, then reads and clears the current device's error word.
 * Returns PD_OK, PD_ERR_BAD_PAGE, PD_ERR_BAD_LENGTH, PD_ERR_BAD_SLOT or
 * PD_ERR_TIMEOUT (the first that is set, in that order), or PD_ERR_CUDA. */
pd_status pd_check_device_errors(pd_stream_t stream);

/* Name of the decode kernel variant the last pd_batch_decode_paged_kv call on this
 * thread launched ("mma" or "simt"), for tests and benchmarks. */
const char* pd_last_decode_variant(void);

/* Human-readable message for the last non-OK status returned on this thread. */
const char* pd_get_last_error_string(void);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int32_t pd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDDECODE_H_ */
