/*
 * Reference oracle for paged-KV decode attention — TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, fp64 CPU restatement of what the decode path computes.  Only the
 * test-suite, the smoke check and the benchmark's CPU-baseline leg may load this
 * library; the product path never calls it.  It shares no code, header, table or
 * constant with the CUDA library.
 *
 * Sources (cited by page title and section):
 *   [TVM]  Apache TVM, python/tvm/relax/frontend/nn/llm/_decode_kernels.py:
 *          `_attention_decode_cpu` (the scalar definition of batch_decode_paged_kv:
 *          length decode, page-table addressing, base-2 score, output and lse) and
 *          `_merge_state_inplace_cpu` (the state-merge formula).
 *   [VLLM] vllm-cpu 0.8.5, vllm/attention/ops/nki_flash_attn.py: `reshape_and_cache`
 *          (slot -> (block, offset) scatter of new K/V into the cache).
 *   [NKI]  NKI Attention Block TKG Kernel API Reference: parameters `k_scale`,
 *          `v_scale` (per-tensor FP8 KV scales), `dtype_mode` (OCP e4m3fn, max 448),
 *          `kv_cache_update_idx` (a sentinel slot means "skip"), `rope_contiguous_layout`.
 *
 * Readings where the sources are silent (the helper module that defines them is
 * not shown on the TVM page):
 *   R1 length/offset:  no window: L = (npages-1)*P + last_page_len, row r -> seq offset r.
 *                      window:    L = (npages-1)*P + last_page_len - win_off + sink,
 *                                 row r -> r if r < sink else r - sink + win_off.
 *   R2 RoPE:           rotate-half ("contiguous halves") over the full head dim,
 *                      theta_i = pos*rope_scale / rope_theta^(2i/D), K row r at
 *                      position k_rope_pos_offset[b] + r (attended-row index).
 *   R4 empty sequence: out = 0, lse = -5e4 (the TVM initial state m=-5e4, d=1).
 *   R5 lse in log2 units: lse = log2(sum_r exp(sm_scale * q.k_r)).
 *   R7 FP8:            K = code*k_scale, V = code*v_scale (the oracle works on the
 *                      dequantised cache; OCP e4m3fn).
 *   R8 append:         slot s -> page s / P, offset s % P; negative slot = skip;
 *                      FP8 code = e4m3_rn_satfinite(fl32(x) / fl32(scale)).
 *
 * Parity pins for every function here live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* dtype codes of this oracle (independent of the CUDA library's enum) */
enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2, OR_E4M3 = 3, OR_F64 = 4 };

static int elem_size(int dt) {
  switch (dt) {
    case OR_F32: return 4;
    case OR_F16: return 2;
    case OR_BF16: return 2;
    case OR_E4M3: return 1;
    case OR_F64: return 8;
  }
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Number formats, from their bit-level definitions.                         */
/* ------------------------------------------------------------------------- */

/* IEEE binary32 bits -> value (memcpy reinterpretation). */
static double f32_bits_to_double(uint32_t u) {
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* bfloat16 = the upper 16 bits of a binary32. */
double oracle_bf16_to_double(uint16_t h) { return f32_bits_to_double((uint32_t)h << 16); }

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 mantissa bits. */
double oracle_f16_to_double(uint16_t h) {
  int s = (h >> 15) & 1, e = (h >> 10) & 0x1f, m = h & 0x3ff;
  double v;
  if (e == 0) v = ldexp((double)m, -24);                 /* subnormal: m * 2^-14 / 2^10 */
  else if (e == 31) v = m ? NAN : INFINITY;
  else v = ldexp(1.0 + m / 1024.0, e - 15);
  return s ? -v : v;
}

/* OCP FP8 E4M3 ("e4m3fn"): 1 sign, 4 exponent (bias 7), 3 mantissa bits; no
 * infinities; S.1111.111 is NaN; largest finite magnitude 1.75 * 2^8 = 448. */
double oracle_e4m3_to_double(uint8_t c) {
  int s = (c >> 7) & 1, e = (c >> 3) & 0xf, m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m, -9);                  /* subnormal: m/8 * 2^-6 */
  else v = ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

/* Round a finite double to the nearest value of a format with `mbits` explicit
 * mantissa bits, minimum normal exponent `emin` (subnormals below it), ties to
 * even.  Returns the rounded value (may exceed the format's finite range; the
 * caller handles overflow). */
static double round_to_format(double x, int mbits, int emin) {
  if (x == 0.0 || !isfinite(x)) return x;
  double ax = fabs(x);
  int e;
  frexp(ax, &e);           /* ax = f * 2^e, f in [0.5, 1) -> unbiased exponent e-1 */
  int ue = e - 1;
  if (ue < emin) ue = emin; /* subnormal region: fixed quantum */
  double quantum = ldexp(1.0, ue - mbits);
  double q = ax / quantum; /* exact: power-of-two scaling */
  double fl = floor(q);
  double rem = q - fl;
  double r;
  if (rem > 0.5) r = fl + 1.0;
  else if (rem < 0.5) r = fl;
  else r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
  double v = r * quantum;
  return x < 0 ? -v : v;
}

/* value -> e4m3 code, round-to-nearest-even, saturating to +-448 (satfinite);
 * NaN -> 0x7f. */
uint8_t oracle_e4m3_encode(double x) {
  if (isnan(x)) return 0x7f;
  uint8_t sign = (x < 0 || (x == 0 && signbit(x))) ? 0x80 : 0;
  double r = round_to_format(x, 3, -6);
  double ar = fabs(r);
  if (ar > 448.0) ar = 448.0;
  if (ar == 0.0) return sign;
  int e;
  frexp(ar, &e);
  int ue = e - 1;
  uint8_t code;
  if (ue < -6) {                         /* subnormal: ar = m * 2^-9 */
    code = (uint8_t)(int)(ar / ldexp(1.0, -9));
  } else {
    int m = (int)((ar / ldexp(1.0, ue) - 1.0) * 8.0);
    code = (uint8_t)(((ue + 7) << 3) | m);
  }
  return sign | code;
}

/* value -> bfloat16 bits, RNE; overflow -> inf. */
uint16_t oracle_bf16_encode(double x) {
  if (isnan(x)) return 0x7fc0;
  double r = round_to_format(x, 7, -126);
  float f = (float)r; /* exact: r is representable in binary32 (or overflows to inf) */
  if (fabs(r) > 3.3895313892515355e38) f = (r < 0) ? -INFINITY : INFINITY;
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

/* value -> binary16 bits, RNE; overflow -> inf. */
uint16_t oracle_f16_encode(double x) {
  if (isnan(x)) return 0x7e00;
  uint16_t sign = (x < 0 || (x == 0 && signbit(x))) ? 0x8000 : 0;
  double r = fabs(round_to_format(x, 10, -14));
  if (r >= 65520.0 || r > 65504.0) return sign | 0x7c00;
  if (r == 0.0) return sign;
  int e;
  frexp(r, &e);
  int ue = e - 1;
  if (ue < -14) return sign | (uint16_t)(int)(r / ldexp(1.0, -24));
  int m = (int)((r / ldexp(1.0, ue) - 1.0) * 1024.0);
  return sign | (uint16_t)(((ue + 15) << 10) | m);
}

/* value -> binary32 bits, RNE (C's double->float conversion). */
static uint32_t f32_encode(double x) {
  float f = (float)x;
  uint32_t u;
  memcpy(&u, &f, 4);
  return u;
}

/* Element i of a typed buffer, as a double. */
static double load_elem(const void* p, int dt, size_t i) {
  switch (dt) {
    case OR_F32: { uint32_t u; memcpy(&u, (const char*)p + 4 * i, 4); return f32_bits_to_double(u); }
    case OR_F16: return oracle_f16_to_double(((const uint16_t*)p)[i]);
    case OR_BF16: return oracle_bf16_to_double(((const uint16_t*)p)[i]);
    case OR_E4M3: return oracle_e4m3_to_double(((const uint8_t*)p)[i]);
    case OR_F64: return ((const double*)p)[i];
  }
  return NAN;
}

/* Decode n elements of a typed buffer into doubles. */
void oracle_decode(const void* src, int dt, double* dst, int64_t n) {
  for (int64_t i = 0; i < n; ++i) dst[i] = load_elem(src, dt, (size_t)i);
}

/* Encode n doubles into a typed buffer (RNE; e4m3 saturating). */
void oracle_encode(const double* src, int dt, void* dst, int64_t n) {
  for (int64_t i = 0; i < n; ++i) {
    switch (dt) {
      case OR_F32: { uint32_t u = f32_encode(src[i]); memcpy((char*)dst + 4 * i, &u, 4); break; }
      case OR_F16: ((uint16_t*)dst)[i] = oracle_f16_encode(src[i]); break;
      case OR_BF16: ((uint16_t*)dst)[i] = oracle_bf16_encode(src[i]); break;
      case OR_E4M3: ((uint8_t*)dst)[i] = oracle_e4m3_encode(src[i]); break;
      case OR_F64: ((double*)dst)[i] = src[i]; break;
    }
  }
}

/* ------------------------------------------------------------------------- */
/* Length decode and row -> sequence offset (reading R1).                    */
/* [TVM] `_attention_decode_cpu`: kv_chunk_len is 0 for an empty page list,  */
/* otherwise derived from the page count, page size and length_info; the     */
/* length_info comment gives its [B] / [3,B] layout.                          */
/* ------------------------------------------------------------------------- */

typedef struct {
  int64_t L;        /* attended rows */
  int64_t sink;     /* rows [0, sink) map to themselves */
  int64_t win_off;  /* rows [sink, L) map to win_off + (r - sink) */
} seq_len_t;

static seq_len_t seq_length(const int32_t* indptr, const int32_t* length_info, int B, int b,
                            int P, int window) {
  seq_len_t s = {0, 0, 0};
  int64_t npages = (int64_t)indptr[b + 1] - indptr[b];
  if (npages == 0) return s;
  int64_t last = length_info[b];
  if (!window) {
    s.L = (npages - 1) * P + last;
    s.sink = s.L;
    s.win_off = 0;
  } else {
    int64_t off = length_info[B + b], sink = length_info[2 * B + b];
    s.L = (npages - 1) * P + last - off + sink;
    s.sink = sink;
    s.win_off = off;
  }
  if (s.L < 0) s.L = 0;
  return s;
}

static int64_t seq_offset(const seq_len_t* s, int64_t r) {
  return r < s->sink ? r : r - s->sink + s->win_off;
}

/* Exposed for the pins: attended seq offsets of sequence b (returns count). */
int64_t oracle_attended_offsets(const int32_t* indptr, const int32_t* length_info, int B, int b,
                                int P, int window, int64_t* out, int64_t cap) {
  seq_len_t s = seq_length(indptr, length_info, B, b, P, window);
  for (int64_t r = 0; r < s.L && r < cap; ++r) out[r] = seq_offset(&s, r);
  return s.L;
}

/* ------------------------------------------------------------------------- */
/* RoPE (reading R2): rotate-half over the full head dim, in fp64.            */
/* [NKI] `rope_contiguous_layout` = contiguous halves; [TVM] passes           */
/* q_rope_position[b] for Q and k_rope_pos_offset[b] + row for K.             */
/* ------------------------------------------------------------------------- */

void oracle_rope(double* x, int D, double pos, double rope_scale, double rope_theta) {
  int half = D / 2;
  for (int i = 0; i < half; ++i) {
    double inv_freq = 1.0 / pow(rope_theta, (2.0 * i) / (double)D);
    double ang = pos * rope_scale * inv_freq;
    double c = cos(ang), s = sin(ang);
    double a = x[i], b = x[i + half];
    x[i] = a * c - b * s;
    x[i + half] = b * c + a * s;
  }
}

/* The interleaved layout ([NKI] `rope_contiguous_layout` = False): frequency i      */
/* rotates the adjacent pair (2i, 2i+1) instead of (i, i + D/2); same angles.        */
void oracle_rope_interleaved(double* x, int D, double pos, double rope_scale,
                             double rope_theta) {
  for (int i = 0; i < D / 2; ++i) {
    double inv_freq = 1.0 / pow(rope_theta, (2.0 * i) / (double)D);
    double ang = pos * rope_scale * inv_freq;
    double c = cos(ang), s = sin(ang);
    double a = x[2 * i], b = x[2 * i + 1];
    x[2 * i] = a * c - b * s;
    x[2 * i + 1] = b * c + a * s;
  }
}

/* rotary_mode: 0 none, 1 rotate-half, 2 interleaved pairs */
static void apply_rope(int rotary_mode, double* x, int D, double pos, double rope_scale,
                       double rope_theta) {
  if (rotary_mode == 1) oracle_rope(x, D, pos, rope_scale, rope_theta);
  if (rotary_mode == 2) oracle_rope_interleaved(x, D, pos, rope_scale, rope_theta);
}

/* ------------------------------------------------------------------------- */
/* batch_decode_paged_kv: [TVM] `_attention_decode_cpu`, restated from the    */
/* plain definition of softmax attention (two passes, fp64):                  */
/*   t_r = sm_scale * q . k_r          (natural units)                        */
/*   lse = log2( sum_r exp(t_r) )      (log2 units, R5)                        */
/*   out = sum_r exp(t_r - M) v_r / sum_r exp(t_r - M)                         */
/* Layouts: Q [B,H_qo,D]; pages [max_pages,2,H_kv,P,D] (0 = K, 1 = V);        */
/* indptr [B+1]; values [nnz]; length_info [B] or [3,B]; out [B,H_qo,D] and   */
/* lse [B,H_qo] as doubles.  KV head of Q head h is h / (H_qo/H_kv).           */
/* `mask` (nullable, [B*H_qo]) selects which (b,h) to compute; others untouched.*/
/* `k_rotated`: the cache holds K already rotated (append with RoPE); only Q is */
/* rotated here.                                                                */
/* `sink` (nullable, [H_qo]): a learned logit per query head, one more softmax  */
/* term exp(sink[h]) with a zero value row (so lse includes it).               */
/* Returns 0, or -1 if a page id or offset is out of range (the row is then   */
/* excluded), -2 on bad arguments.                                            */
/* ------------------------------------------------------------------------- */

/* Multi-query form (q_len >= 1 query tokens per sequence): the last q_len attended  */
/* rows of sequence b are the new tokens' own K/V, already in the cache, and token t  */
/* (0-based) sees rows r < L - q_len + 1 + t: the cached context in full and the new  */
/* tokens causally ([vllm-cpu] nki_flash_attn.py, flash_paged_attention: the context  */
/* part of the mask is open, the active part causal).  Token t's RoPE position is     */
/* q_rope_position[b] + t.  Q, out: rows (b*q_len + t)*H_qo + h; lse likewise; mask   */
/* [B*q_len*H_qo].  q_len = 1 is batch_decode_paged_kv.  No sliding window (-2).      */
static int decode_impl(const void* Q, int q_dtype, const void* pages, int kv_dtype,
                       const int32_t* indptr, const int32_t* values, const int32_t* length_info,
                       const int32_t* k_rope_pos_offset, const int32_t* q_rope_position,
                       double* out, double* lse, int B, int q_len, int H_qo, int H_kv, int D,
                       int P, int64_t max_pages, int window, int rotary_mode, double rope_scale,
                       double rope_theta, double sm_scale, double k_scale, double v_scale,
                       int k_rotated, const double* sink, const uint8_t* mask) {
  if (B < 0 || H_kv <= 0 || H_qo % H_kv != 0 || D <= 0 || D % 2 || P <= 0) return -2;
  if (q_len < 1 || (q_len > 1 && window) || rotary_mode < 0 || rotary_mode > 2) return -2;
  int group = H_qo / H_kv;
  int status = 0;
  double* q = (double*)malloc(sizeof(double) * D);
  double* k = (double*)malloc(sizeof(double) * D);
  for (int b = 0; b < B; ++b) {
    seq_len_t s = seq_length(indptr, length_info, B, b, P, window);
    int64_t L = s.L, npages = (int64_t)indptr[b + 1] - indptr[b];
    size_t cap = (size_t)(L > 0 ? L : 1);
    /* page-table addressing of every attended row: page number and slot */
    int64_t* page_of = (int64_t*)malloc(sizeof(int64_t) * cap);
    int64_t* slot_of = (int64_t*)malloc(sizeof(int64_t) * cap);
    uint8_t* valid = (uint8_t*)malloc(cap);
    double* score = (double*)malloc(sizeof(double) * cap);
    for (int64_t r = 0; r < L; ++r) {
      int64_t so = seq_offset(&s, r);
      valid[r] = 0;
      if (so < 0 || so / P >= npages) { status = -1; continue; }
      int64_t page_no = values[indptr[b] + so / P];
      if (page_no < 0 || page_no >= max_pages) { status = -1; continue; }
      page_of[r] = page_no;
      slot_of[r] = so % P;
      valid[r] = 1;
    }
    for (int t = 0; t < q_len; ++t)
    for (int h = 0; h < H_qo; ++h) {
      const size_t row = ((size_t)b * q_len + t) * H_qo + h; /* (sequence, token, head) */
      if (mask && !mask[row]) continue;
      int hk = h / group;
      /* rows this token sees: all L for a single token, else causal among the new ones */
      int64_t Lt = L - q_len + 1 + t;
      if (Lt > L) Lt = L;
      if (Lt < 0) Lt = 0;
      double* o = out + row * D;
      for (int d = 0; d < D; ++d) q[d] = load_elem(Q, q_dtype, row * D + d);
      apply_rope(rotary_mode, q, D, (double)q_rope_position[b] + (double)t, rope_scale,
                 rope_theta);
      /* pass 1: scores t_r and their maximum */
      double M = -INFINITY;
      int64_t n_valid = 0;
      for (int64_t r = 0; r < Lt; ++r) {
        if (!valid[r]) continue;
        size_t kbase = ((((size_t)page_of[r] * 2 + 0) * H_kv + hk) * P + slot_of[r]) * D;
        for (int d = 0; d < D; ++d) {
          k[d] = load_elem(pages, kv_dtype, kbase + d);
          if (kv_dtype == OR_E4M3) k[d] *= k_scale;
        }
        if (!k_rotated) /* else the cache holds K rotated at append time */
          apply_rope(rotary_mode, k, D, (double)k_rope_pos_offset[b] + (double)r, rope_scale,
                     rope_theta);
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += q[d] * k[d];
        score[r] = sm_scale * dot;
        if (score[r] > M) M = score[r];
        ++n_valid;
      }
      /* a learned sink (NKI TKG `sink`, one logit per query head) is one more score, */
      /* sink[h] in natural units, whose value row is zero                             */
      if (sink && sink[h] > M) M = sink[h];
      if (n_valid == 0 && !sink) { /* R4: empty sequence */
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        lse[row] = -5e4;
        continue;
      }
      /* pass 2: softmax weights, their sum, and the weighted sum of V rows */
      double den = sink ? exp(sink[h] - M) : 0.0;
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      for (int64_t r = 0; r < Lt; ++r) {
        if (!valid[r]) continue;
        double w = exp(score[r] - M);
        den += w;
        size_t vbase = ((((size_t)page_of[r] * 2 + 1) * H_kv + hk) * P + slot_of[r]) * D;
        for (int d = 0; d < D; ++d) {
          double vv = load_elem(pages, kv_dtype, vbase + d);
          if (kv_dtype == OR_E4M3) vv *= v_scale;
          o[d] += w * vv;
        }
      }
      for (int d = 0; d < D; ++d) o[d] /= den;
      lse[row] = (M + log(den)) / log(2.0); /* natural -> log2 units */
    }
    free(page_of);
    free(slot_of);
    free(valid);
    free(score);
  }
  free(q);
  free(k);
  return status;
}

int oracle_batch_decode_paged_kv(const void* Q, int q_dtype, const void* pages, int kv_dtype,
                                 const int32_t* indptr, const int32_t* values,
                                 const int32_t* length_info, const int32_t* k_rope_pos_offset,
                                 const int32_t* q_rope_position, double* out, double* lse, int B,
                                 int H_qo, int H_kv, int D, int P, int64_t max_pages, int window,
                                 int rotary_mode, double rope_scale, double rope_theta,
                                 double sm_scale, double k_scale, double v_scale,
                                 int k_rotated, const double* sink, const uint8_t* mask) {
  return decode_impl(Q, q_dtype, pages, kv_dtype, indptr, values, length_info, k_rope_pos_offset,
                     q_rope_position, out, lse, B, 1, H_qo, H_kv, D, P, max_pages, window,
                     rotary_mode, rope_scale, rope_theta, sm_scale, k_scale, v_scale, k_rotated,
                     sink, mask);
}

int oracle_batch_decode_paged_kv_mq(const void* Q, int q_dtype, const void* pages, int kv_dtype,
                                    const int32_t* indptr, const int32_t* values,
                                    const int32_t* length_info, const int32_t* k_rope_pos_offset,
                                    const int32_t* q_rope_position, double* out, double* lse,
                                    int B, int q_len, int H_qo, int H_kv, int D, int P,
                                    int64_t max_pages, int rotary_mode, double rope_scale,
                                    double rope_theta, double sm_scale, double k_scale,
                                    double v_scale, int k_rotated, const double* sink,
                                    const uint8_t* mask) {
  return decode_impl(Q, q_dtype, pages, kv_dtype, indptr, values, length_info, k_rope_pos_offset,
                     q_rope_position, out, lse, B, q_len, H_qo, H_kv, D, P, max_pages, 0,
                     rotary_mode, rope_scale, rope_theta, sm_scale, k_scale, v_scale, k_rotated,
                     sink, mask);
}

/* ------------------------------------------------------------------------- */
/* merge_state_inplace: [TVM] `_merge_state_inplace_cpu`, in fp64.            */
/*   s_max = max(S, S_o); w = 2^(S - s_max); w_o = 2^(S_o - s_max)             */
/*   V <- V * w/(w+w_o) + V_o * w_o/(w+w_o);  S <- log2(w + w_o) + s_max       */
/* V, V_other [N,H,D]; S, S_other [N,H].                                       */
/* ------------------------------------------------------------------------- */

void oracle_merge_state(double* V, double* S, const double* V_other, const double* S_other,
                        int N, int H, int D) {
  for (int n = 0; n < N; ++n)
    for (int h = 0; h < H; ++h) {
      size_t i = (size_t)n * H + h;
      double s = S[i], so = S_other[i];
      double smax = s > so ? s : so;
      double w = exp2(s - smax), wo = exp2(so - smax);
      double a = w / (w + wo), ao = wo / (w + wo);
      for (int d = 0; d < D; ++d) V[i * D + d] = V[i * D + d] * a + V_other[i * D + d] * ao;
      S[i] = log2(w + wo) + smax;
    }
}

/* ------------------------------------------------------------------------- */
/* merge of R states at once: the [TVM] merge formula over R partners (the     */
/* pairwise form is R = 2; the module docstring's multi-stage decoding and the */
/* distributed KV-transfer path combine the (V, S) states of R partial         */
/* decodes).  For every (n, h):                                                */
/*   M = max_r S_r;  w_r = 2^(S_r - M);  V = sum_r w_r V_r / sum_r w_r;         */
/*   S = log2(sum_r w_r) + M.                                                   */
/* If every partner is the empty state (S_r <= -5e4: the decode's sentinel of  */
/* a sequence with no row), the result is the empty state itself: V = 0,       */
/* S = -5e4 (reading R4 applied to the merged set of rows, which is empty).    */
/* V_parts [R,N,H,D], S_parts [R,N,H]; V_out [N,H,D], S_out [N,H].             */
/* ------------------------------------------------------------------------- */

void oracle_merge_states(const double* V_parts, const double* S_parts, double* V_out,
                         double* S_out, int R, int N, int H, int D) {
  const size_t rows = (size_t)N * H;
  for (size_t i = 0; i < rows; ++i) {
    double M = -INFINITY;
    for (int r = 0; r < R; ++r) {
      double s = S_parts[(size_t)r * rows + i];
      if (s > M) M = s;
    }
    double* v = V_out + i * D;
    for (int d = 0; d < D; ++d) v[d] = 0.0;
    if (!(M > -5e4)) {
      S_out[i] = -5e4;
      continue;
    }
    double den = 0.0;
    for (int r = 0; r < R; ++r) {
      double w = exp2(S_parts[(size_t)r * rows + i] - M);
      den += w;
      const double* vr = V_parts + ((size_t)r * rows + i) * D;
      for (int d = 0; d < D; ++d) v[d] += w * vr[d];
    }
    for (int d = 0; d < D; ++d) v[d] /= den;
    S_out[i] = log2(den) + M;
  }
}

/* ------------------------------------------------------------------------- */
/* append_paged_kv: [VLLM] `reshape_and_cache` on the TVM page layout.         */
/* For token t with slot s >= 0: page = s / P, off = s % P;                    */
/*   pages[page,0,h,off,:] = conv(k[t,h,:]),  pages[page,1,h,off,:] = conv(v). */
/* conv: same dtype -> bit copy; to e4m3 -> e4m3_rn_satfinite(fl32(x)/scale)   */
/* with the division in binary32 ([NKI] k_scale / v_scale); otherwise RNE.     */
/* Negative slots are skipped ([NKI] kv_cache_update_idx sentinel).            */
/* Returns the number of slots that were out of range (skipped), or -2.        */
/* ------------------------------------------------------------------------- */

/* With RoPE (rotary_mode 1 or 2, positions[t]): the K row is first rotated in fp64   */
/* at its token's position ([NKI] TKG: RoPE, then the KV cache update), then stored    */
/* by the same conversion; V is stored as is.                                           */
static int append_impl(void* pages, int kv_dtype, const void* k_new, const void* v_new,
                       int in_dtype, const int64_t* slot_mapping, int T, int H_kv, int D, int P,
                       int64_t max_pages, float k_scale, float v_scale, const int32_t* positions,
                       int rotary_mode, double rope_scale, double rope_theta) {
  if (T < 0 || H_kv <= 0 || D <= 0 || P <= 0 || rotary_mode < 0 || rotary_mode > 2) return -2;
  if (rotary_mode && (!positions || D % 2)) return -2;
  double* row = (double*)malloc(sizeof(double) * (size_t)D);
  int es_in = elem_size(in_dtype), es_kv = elem_size(kv_dtype);
  int bad = 0;
  for (int t = 0; t < T; ++t) {
    int64_t s = slot_mapping[t];
    if (s < 0) continue;
    int64_t page = s / P, off = s % P;
    if (page >= max_pages) { ++bad; continue; }
    for (int kv = 0; kv < 2; ++kv) {
      const void* src = kv == 0 ? k_new : v_new;
      float scale = kv == 0 ? k_scale : v_scale;
      for (int h = 0; h < H_kv; ++h) {
        size_t si = ((size_t)t * H_kv + h) * D;
        size_t di = ((((size_t)page * 2 + kv) * H_kv + h) * P + off) * D;
        const int rot = kv == 0 && rotary_mode;
        if (in_dtype == kv_dtype && !rot) {
          memcpy((char*)pages + di * es_kv, (const char*)src + si * es_in, (size_t)D * es_kv);
          continue;
        }
        for (int d = 0; d < D; ++d) row[d] = load_elem(src, in_dtype, si + d);
        if (rot) apply_rope(rotary_mode, row, D, (double)positions[t], rope_scale, rope_theta);
        for (int d = 0; d < D; ++d) {
          double x = row[d];
          if (kv_dtype == OR_E4M3) {
            float q = (float)x / scale;  /* binary32 division, round-to-nearest */
            ((uint8_t*)pages)[di + d] = oracle_e4m3_encode((double)q);
          } else {
            oracle_encode(&x, kv_dtype, (char*)pages + (di + d) * es_kv, 1);
          }
        }
      }
    }
  }
  free(row);
  return bad;
}

int oracle_append_paged_kv(void* pages, int kv_dtype, const void* k_new, const void* v_new,
                           int in_dtype, const int64_t* slot_mapping, int T, int H_kv, int D,
                           int P, int64_t max_pages, float k_scale, float v_scale) {
  return append_impl(pages, kv_dtype, k_new, v_new, in_dtype, slot_mapping, T, H_kv, D, P,
                     max_pages, k_scale, v_scale, NULL, 0, 1.0, 1e4);
}

int oracle_append_paged_kv_rope(void* pages, int kv_dtype, const void* k_new, const void* v_new,
                                int in_dtype, const int64_t* slot_mapping, int T, int H_kv,
                                int D, int P, int64_t max_pages, float k_scale, float v_scale,
                                const int32_t* positions, int rotary_mode, double rope_scale,
                                double rope_theta) {
  return append_impl(pages, kv_dtype, k_new, v_new, in_dtype, slot_mapping, T, H_kv, D, P,
                     max_pages, k_scale, v_scale, positions, rotary_mode, rope_scale, rope_theta);
}
