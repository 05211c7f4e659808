"""Seeded synthetic workloads for paged-KV decode attention.

This module only *draws inputs*: sequence lengths, shuffled page tables, random
Q/K/V values and RoPE positions.  It holds none of the attention arithmetic and is
the one module shared by the CUDA path's tests/benchmark and the fp64 oracle.
Dtype casts (fp32 -> bf16/f16/e4m3) use torch's own conversions, so neither
side's number-format code produces the other's inputs.

The five named workloads follow the serving loads described for the decode kernel
(Apache TVM ``_decode_kernels.py`` API: ``Q[B,H_qo,D]``, ``pages[max_pages,2,H_kv,P,D]``,
CSR page table, ``length_info`` ``[B]`` or ``[3,B]``):

  tiny_fp32          B=4,   H 8/2,  D=64,  P=16, fp32, len U[1,200], 64-page pool
  llama3_8b_bf16     B=32,  H 32/8, D=128, P=16, bf16, len U[512,4096], RoPE 5e5
  long_ctx_bf16      B=8,   H 32/8, D=128, P=16, bf16, len U[32768,131072]
  window_sink_f16    B=64,  H 32/4, D=128, P=16, f16, len U[4096,16384], window 4096, sink 4, RoPE 1e4
  fp8_kv_highconc    B=256, H 64/8, D=128, P=32, e4m3 KV (+ bf16 Q), lognormal len, + append
  llama3_8b_bf16_krot  llama3_8b_bf16 with the cache holding K rotated at append time
                     (pd_append_paged_kv_rope; the decode rotates only Q)
  spec_decode_bf16   llama3_8b_bf16 with 2 query tokens per sequence (multi-query decode,
                     causal among them: speculative decoding's verification step; the
                     2 x 4 (token, head) columns of a KV head fill one 8-column MMA tile)

Each has a ``reduced`` variant (same structure, fewer/shorter sequences) that the
oracle finishes in seconds.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

TORCH_DTYPES = {
    "f32": torch.float32,
    "f16": torch.float16,
    "bf16": torch.bfloat16,
    "e4m3": torch.float8_e4m3fn,
}
E4M3_MAX = 448.0  # largest finite OCP e4m3fn magnitude


@dataclasses.dataclass
class Spec:
    name: str
    B: int
    H_qo: int
    H_kv: int
    D: int
    page_size: int
    q_dtype: str
    kv_dtype: str
    out_dtype: str
    len_dist: tuple            # ("uniform", lo, hi) | ("lognormal", median, sigma, lo, hi)
    pool: str = "fit"          # "fit": pool = needed pages * slack; or an int page count
    rotary_mode: int = 0
    rope_theta: float = 1e4
    rope_scale: float = 1.0
    window: Optional[int] = None
    sink: int = 0
    append: bool = False       # one new token per sequence, written before attention
    max_splits: int = 0        # external split count (long-context chunking)
    q_len: int = 1             # query tokens per sequence (multi-query decode, causal)
    k_rotated: bool = False    # the cache holds K rotated at append time (decode rotates Q only)
    # Score-shaping stress inputs (both default off): every cached K row at sequence
    # offset o is multiplied by 1 + k_ramp * o / (len - 1), so scores grow along the
    # sequence and the running maximum of an online softmax keeps moving; Q is
    # multiplied by q_gain (a peaked softmax).  Pure input scaling, applied before the
    # cast to the cache / query type.
    k_ramp: float = 0.0
    q_gain: float = 1.0


SPECS = {
    "tiny_fp32": Spec("tiny_fp32", 4, 8, 2, 64, 16, "f32", "f32", "f32",
                      ("uniform", 1, 200), pool=64),
    "llama3_8b_bf16": Spec("llama3_8b_bf16", 32, 32, 8, 128, 16, "bf16", "bf16", "bf16",
                           ("uniform", 512, 4096), pool=16384, rotary_mode=1,
                           rope_theta=500000.0),
    "long_ctx_bf16": Spec("long_ctx_bf16", 8, 32, 8, 128, 16, "bf16", "bf16", "bf16",
                          ("uniform", 32768, 131072), max_splits=32),
    "window_sink_f16": Spec("window_sink_f16", 64, 32, 4, 128, 16, "f16", "f16", "f16",
                            ("uniform", 4096, 16384), rotary_mode=1, rope_theta=10000.0,
                            window=4096, sink=4),
    "fp8_kv_highconc": Spec("fp8_kv_highconc", 256, 64, 8, 128, 32, "bf16", "e4m3", "bf16",
                            ("lognormal", 2048, 0.6, 64, 8192), append=True),
    "llama3_8b_bf16_krot": Spec("llama3_8b_bf16_krot", 32, 32, 8, 128, 16, "bf16", "bf16",
                                "bf16", ("uniform", 512, 4096), pool=16384, rotary_mode=1,
                                rope_theta=500000.0, k_rotated=True),
    "spec_decode_bf16": Spec("spec_decode_bf16", 32, 32, 8, 128, 16, "bf16", "bf16", "bf16",
                             ("uniform", 512, 4096), pool=16384, rotary_mode=1,
                             rope_theta=500000.0, q_len=2),
}

# Reduced variants: same heads/dtypes/page size/features, sizes the oracle handles in
# seconds while still spanning several pages, splits and a ragged last page.
REDUCED = {
    "tiny_fp32": {},
    "llama3_8b_bf16": dict(B=5, len_dist=("uniform", 17, 700), pool=512),
    "long_ctx_bf16": dict(B=2, len_dist=("uniform", 1500, 3000)),
    "window_sink_f16": dict(B=5, len_dist=("uniform", 200, 900), window=300),
    "fp8_kv_highconc": dict(B=6, len_dist=("lognormal", 300, 0.6, 20, 700)),
    "spec_decode_bf16": dict(B=5, len_dist=("uniform", 17, 700), pool=512),
    "llama3_8b_bf16_krot": dict(B=5, len_dist=("uniform", 17, 700), pool=512),
}


def spec(name: str, reduced: bool = False, **overrides) -> Spec:
    s = dataclasses.replace(SPECS[name])
    if reduced:
        s = dataclasses.replace(s, **REDUCED[name])
    if overrides:
        s = dataclasses.replace(s, **overrides)
    return s


@dataclasses.dataclass
class Workload:
    spec: Spec
    Q: torch.Tensor                 # [B,H_qo,D] q_dtype ([B,q_len,H_qo,D] multi-query)
    pages: torch.Tensor             # [max_pages,2,H_kv,P,D] kv_dtype
    indptr: torch.Tensor            # [B+1] int32
    values: torch.Tensor            # [nnz] int32
    length_info: torch.Tensor       # [B] or [3,B] int32
    k_rope_pos_offset: torch.Tensor  # [B] int32
    q_rope_position: torch.Tensor   # [B] int32
    seq_len: np.ndarray             # rows held in the cache per sequence
    attended: np.ndarray            # rows attended per sequence
    sm_scale: float
    k_scale: float = 1.0
    v_scale: float = 1.0
    k_new: Optional[torch.Tensor] = None       # [B,H_kv,D] new-token K (q_dtype)
    v_new: Optional[torch.Tensor] = None
    slot_mapping: Optional[torch.Tensor] = None  # [B] int64

    @property
    def max_pages(self) -> int:
        return int(self.pages.shape[0])

    def kv_bytes_attended(self) -> int:
        """K+V bytes of the attended rows (no padding)."""
        es = torch.empty(0, dtype=self.pages.dtype).element_size()
        s = self.spec
        return int(self.attended.sum()) * 2 * s.H_kv * s.D * es

    def io_bytes(self) -> int:
        s = self.spec
        qes = torch.empty(0, dtype=self.Q.dtype).element_size()
        oes = torch.empty(0, dtype=TORCH_DTYPES[s.out_dtype]).element_size()
        return s.q_len * (s.B * s.H_qo * s.D * (qes + oes) + s.B * s.H_qo * 4)

    def to(self, device) -> "Workload":
        def mv(x):
            return None if x is None else x.to(device)
        return dataclasses.replace(
            self, Q=mv(self.Q), pages=mv(self.pages), indptr=mv(self.indptr),
            values=mv(self.values), length_info=mv(self.length_info),
            k_rope_pos_offset=mv(self.k_rope_pos_offset),
            q_rope_position=mv(self.q_rope_position), k_new=mv(self.k_new),
            v_new=mv(self.v_new), slot_mapping=mv(self.slot_mapping))


def _draw_lengths(rng: np.random.Generator, s: Spec) -> np.ndarray:
    kind = s.len_dist[0]
    if kind == "uniform":
        _, lo, hi = s.len_dist
        return rng.integers(lo, hi + 1, size=s.B).astype(np.int64)
    if kind == "lognormal":
        _, median, sigma, lo, hi = s.len_dist
        x = rng.lognormal(mean=math.log(median), sigma=sigma, size=s.B)
        return np.clip(np.rint(x), lo, hi).astype(np.int64)
    raise ValueError(kind)


def _randn(shape, gen, device, chunk=1 << 26):
    """N(0,1) float32 on `device`, drawn in chunks (bounded temporary memory)."""
    n = int(np.prod(shape))
    out = torch.empty(n, dtype=torch.float32, device=device)
    for i in range(0, n, chunk):
        m = min(chunk, n - i)
        out[i:i + m] = torch.randn(m, generator=gen, device=device, dtype=torch.float32)
    return out.view(*shape)


def _cast_pool(x: torch.Tensor, dtype: str, scale: float) -> torch.Tensor:
    if dtype == "e4m3":
        return (x / scale).to(torch.float8_e4m3fn)
    return x.to(TORCH_DTYPES[dtype])


def _ramp_factors(values, indptr, seq_len, pool, P, ramp) -> torch.Tensor:
    """[pool, P] float32 row factors: 1 + ramp * o / (len - 1) for the row at sequence
    offset o of the sequence owning the page, 1 for rows of unused pages."""
    f = np.ones((pool, P), np.float32)
    for b in range(len(seq_len)):
        n = int(indptr[b + 1] - indptr[b])
        if n == 0:
            continue
        o = np.arange(n * P, dtype=np.float64).reshape(n, P)
        f[values[indptr[b]:indptr[b + 1]]] = 1.0 + ramp * o / max(int(seq_len[b]) - 1, 1)
    return torch.from_numpy(f)


def make(name: str, seed: int = 0, reduced: bool = False, device="cpu", **overrides) -> Workload:
    """Draw the workload `name` with `seed` on `device` (torch generator of that device)."""
    s = spec(name, reduced, **overrides)
    rng = np.random.default_rng(seed)
    P = s.page_size
    seq_len = _draw_lengths(rng, s)
    npages = (seq_len + P - 1) // P
    nnz = int(npages.sum())
    pool = int(math.ceil(nnz * 1.05)) + 1 if s.pool == "fit" else int(s.pool)
    if pool < nnz:
        raise ValueError(f"{name}: pool {pool} < needed pages {nnz}")
    perm = rng.permutation(pool).astype(np.int32)
    values = perm[:nnz].copy()
    indptr = np.zeros(s.B + 1, np.int32)
    indptr[1:] = np.cumsum(npages)
    last = (seq_len - (npages - 1) * P).astype(np.int32)
    last[npages == 0] = 0
    if s.window is None:
        length_info = last
        attended = seq_len.copy()
    else:
        win_off = np.maximum(s.sink, seq_len - s.window).astype(np.int32)
        sink = np.full(s.B, s.sink, np.int32)
        sink = np.minimum(sink, seq_len).astype(np.int32)
        win_off = np.maximum(win_off, sink)
        length_info = np.stack([last, win_off, sink]).astype(np.int32)
        attended = (seq_len - win_off + sink).astype(np.int64)
        attended[npages == 0] = 0
    k_off = np.zeros(s.B, np.int32)
    q_pos = attended.astype(np.int32)  # query sits right after the attended (compacted) rows
    if s.q_len > 1:  # the new tokens are the last q_len cached rows: token t at its own row
        q_pos = np.maximum(attended - s.q_len, 0).astype(np.int32)

    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    x = _randn((pool, 2, s.H_kv, P, s.D), gen, device)
    if s.k_ramp:
        x[:, 0] *= _ramp_factors(values, indptr, seq_len, pool, P, s.k_ramp).to(device)[:, None, :, None]
    k_scale = v_scale = 1.0
    if s.kv_dtype == "e4m3":
        k_scale = float(x[:, 0].abs().max()) / E4M3_MAX
        v_scale = float(x[:, 1].abs().max()) / E4M3_MAX
        pages = torch.empty(x.shape, dtype=torch.float8_e4m3fn, device=device)
        pages[:, 0] = _cast_pool(x[:, 0], "e4m3", k_scale)
        pages[:, 1] = _cast_pool(x[:, 1], "e4m3", v_scale)
    else:
        pages = x.to(TORCH_DTYPES[s.kv_dtype])
    del x
    qshape = (s.B, s.H_qo, s.D) if s.q_len == 1 else (s.B, s.q_len, s.H_qo, s.D)
    Q = _randn(qshape, gen, device)
    if s.q_gain != 1.0:
        Q *= s.q_gain
    Q = Q.to(TORCH_DTYPES[s.q_dtype])
    k_new = v_new = slot_mapping = None
    if s.append:
        in_dt = TORCH_DTYPES[s.q_dtype]
        k_new = _randn((s.B, s.H_kv, s.D), gen, device).to(in_dt)
        v_new = _randn((s.B, s.H_kv, s.D), gen, device).to(in_dt)
        row = seq_len - 1
        slots = np.where(seq_len > 0, values[indptr[:-1] + np.maximum(row, 0) // P].astype(np.int64) * P
                         + np.maximum(row, 0) % P, -1)
        slot_mapping = torch.from_numpy(slots.astype(np.int64)).to(device)

    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
    return Workload(
        spec=s, Q=Q, pages=pages, indptr=t(indptr), values=t(values if nnz else np.zeros(1, np.int32)),
        length_info=t(length_info), k_rope_pos_offset=t(k_off), q_rope_position=t(q_pos),
        seq_len=seq_len, attended=attended, sm_scale=1.0 / math.sqrt(s.D),
        k_scale=k_scale, v_scale=v_scale, k_new=k_new, v_new=v_new, slot_mapping=slot_mapping)


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw bits of a typed tensor as a host numpy array (uint16 for 16-bit floats,
    uint8 for e4m3, uint32 for fp32)."""
    t = t.detach().contiguous().cpu()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    if t.dtype == torch.float32:
        return t.numpy().view(np.uint32)
    return t.numpy()


def split_chunks(indptr: np.ndarray, values: np.ndarray, seq_len: np.ndarray, page_size: int,
                 max_splits: int):
    """External split of each sequence's page list into <= max_splits page-aligned
    chunks (a pure re-indexing of the page table; no attention arithmetic).

    Returns (indptr_c, values_c, last_c, k_off_c, owner) describing the chunks as
    pseudo-sequences: chunk j of sequence b covers rows [start, start+len) and RoPE
    positions start from ``k_off_c``.
    """
    P = page_size
    ip, vals, last, koff, owner = [0], [], [], [], []
    for b in range(len(seq_len)):
        n = int(indptr[b + 1] - indptr[b])
        if n == 0:
            continue
        per = max(1, -(-n // max_splits))
        for p0 in range(0, n, per):
            p1 = min(n, p0 + per)
            vals.extend(values[indptr[b] + p0: indptr[b] + p1].tolist())
            ip.append(len(vals))
            rows = min(int(seq_len[b]), p1 * P) - p0 * P
            last.append(rows - (p1 - p0 - 1) * P)
            koff.append(p0 * P)
            owner.append(b)
    return (np.array(ip, np.int32), np.array(vals, np.int32), np.array(last, np.int32),
            np.array(koff, np.int32), np.array(owner, np.int64))


def split_chunks_padded(indptr: np.ndarray, values: np.ndarray, seq_len: np.ndarray,
                        page_size: int, nsplit: int):
    """The same page-aligned split, laid out chunk-major and padded: pseudo-sequence
    j * B + b is chunk j of sequence b (pages [j*per, (j+1)*per) of its list, per =
    ceil(npages / nsplit)), and a chunk past the end of the list has no pages.  An empty
    pseudo-sequence decodes to the merge identity (out 0, lse -5e4), so a pairwise merge
    of the first half of the chunks with the second, halving log2(nsplit) times, leaves
    each sequence's result in pseudo-sequence b.  A pure re-indexing of the page table.

    Returns (indptr_c [nsplit*B+1], values_c, last_c [nsplit*B], row_off_c [nsplit*B]):
    row_off_c is the chunk's first row in its sequence.
    """
    P = page_size
    B = len(seq_len)
    npg = (indptr[1:] - indptr[:-1]).astype(np.int64)
    per = np.maximum(1, -(-npg // nsplit))
    ip, vals = [0], []
    last = np.zeros(nsplit * B, np.int32)
    roff = np.zeros(nsplit * B, np.int32)
    for j in range(nsplit):
        for b in range(B):
            p0 = min(int(npg[b]), j * int(per[b]))
            p1 = min(int(npg[b]), p0 + int(per[b]))
            vals.extend(values[indptr[b] + p0: indptr[b] + p1].tolist())
            ip.append(len(vals))
            if p1 > p0:
                rows = min(int(seq_len[b]), p1 * P) - p0 * P
                last[j * B + b] = rows - (p1 - p0 - 1) * P
                roff[j * B + b] = p0 * P
    return np.array(ip, np.int32), np.array(vals, np.int32), last, roff
