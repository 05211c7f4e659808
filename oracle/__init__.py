"""fp64 CPU oracle for paged-KV decode attention — TEST INFRASTRUCTURE ONLY.

Thin ctypes wrapper over ``oracle.c`` (plain C, fp64).  Only ``tests/``, the
smoke check in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may
import this package; the CUDA product path never does.  The two share no code:
the only common module is the seeded input generator, which holds none of the
method's arithmetic.

What each function restates (page title / section):
  * ``batch_decode_paged_kv`` — Apache TVM ``_decode_kernels.py``,
    ``_attention_decode_cpu``, written as two-pass softmax attention in fp64.
  * ``batch_decode_paged_kv_mq`` — the same with q_len query tokens per sequence,
    causal among the new tokens (vllm-cpu ``nki_flash_attn.py``,
    ``flash_paged_attention``: context open, active tokens causal).
  * ``merge_state`` — same page, ``_merge_state_inplace_cpu``.
  * ``append_paged_kv_rope`` / ``k_rotated`` — the NKI TKG order (RoPE, then the
    cache update): K stored rotated, the decode rotating only Q.
  * ``append_paged_kv`` — vllm-cpu ``nki_flash_attn.py``, ``reshape_and_cache``,
    on the TVM page layout, with the FP8 encode of the NKI Attention Block TKG
    reference (``k_scale``/``v_scale``, OCP e4m3fn).
  * number formats (bf16 / f16 / e4m3 decode and RNE encode) — from their
    bit-level definitions.
Pins: ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_SRC = os.path.join(_HERE, "oracle.c")

DTYPES = {"f32": 0, "f16": 1, "bf16": 2, "e4m3": 3, "f64": 4}
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (portable flags: no -march, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
             "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            L.oracle_batch_decode_paged_kv.argtypes = [
                P, i32, P, i32, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i64, i32, i32,
                f64, f64, f64, f64, f64, i32, P, P]
            L.oracle_batch_decode_paged_kv_mq.argtypes = [
                P, i32, P, i32, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i64, i32,
                f64, f64, f64, f64, f64, i32, P, P]
            L.oracle_batch_decode_paged_kv.restype = i32
            L.oracle_merge_state.argtypes = [P, P, P, P, i32, i32, i32]
            L.oracle_merge_state.restype = None
            L.oracle_merge_states.argtypes = [P, P, P, P, i32, i32, i32, i32]
            L.oracle_merge_states.restype = None
            L.oracle_append_paged_kv.argtypes = [
                P, i32, P, P, i32, P, i32, i32, i32, i32, i64, ctypes.c_float, ctypes.c_float]
            L.oracle_append_paged_kv.restype = i32
            L.oracle_decode.argtypes = [P, i32, P, i64]
            L.oracle_encode.argtypes = [P, i32, P, i64]
            L.oracle_rope.argtypes = [P, i32, f64, f64, f64]
            L.oracle_append_paged_kv_rope.argtypes = [P, i32, P, P, i32, P, i32, i32, i32, i32,
                                                      i64, ctypes.c_float, ctypes.c_float, P,
                                                      i32, f64, f64]
            L.oracle_rope_interleaved.argtypes = [P, i32, f64, f64, f64]
            L.oracle_attended_offsets.argtypes = [P, P, i32, i32, i32, i32, P, i64]
            L.oracle_attended_offsets.restype = i64
            L.oracle_e4m3_encode.argtypes = [f64]
            L.oracle_e4m3_encode.restype = ctypes.c_uint8
            L.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
            L.oracle_e4m3_to_double.restype = f64
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


_STORAGE = {"f32": np.uint32, "f16": np.uint16, "bf16": np.uint16, "e4m3": np.uint8,
            "f64": np.float64}


def _bits(a, dt):
    """Typed buffers travel as their raw bits (uint16 for bf16/f16, uint8 for e4m3)."""
    a = np.ascontiguousarray(a)
    if dt == "f32" and a.dtype == np.float32:
        return a.view(np.uint32)
    want = _STORAGE[dt]
    if a.dtype != want:
        raise TypeError(f"{dt} buffer must hold {want} bits, got {a.dtype}")
    return a


def decode(bits, dt):
    """Typed bits -> float64 values."""
    b = _bits(bits, dt)
    out = np.empty(b.shape, np.float64)
    lib().oracle_decode(_ptr(b), DTYPES[dt], _ptr(out), b.size)
    return out


def encode(values, dt):
    """float64 values -> typed bits (round to nearest even; e4m3 saturating)."""
    v = _c(values, np.float64)
    out = np.empty(v.shape, _STORAGE[dt] if dt != "f32" else np.uint32)
    lib().oracle_encode(_ptr(v), DTYPES[dt], _ptr(out), v.size)
    return out


def rope(x, pos, rope_scale, rope_theta, interleaved=False):
    """RoPE of one head vector in fp64: rotate-half (reading R2), or the interleaved
    pair layout (rotary_mode 2)."""
    v = _c(x, np.float64).copy()
    f = lib().oracle_rope_interleaved if interleaved else lib().oracle_rope
    f(_ptr(v), v.shape[-1], float(pos), float(rope_scale), float(rope_theta))
    return v


def attended_offsets(indptr, length_info, b, page_size, window):
    """Sequence offsets attended by sequence b, in attended-row order (reading R1)."""
    indptr = _c(indptr, np.int32)
    li = _c(length_info, np.int32)
    B = indptr.size - 1
    cap = int(indptr[-1]) * page_size + 1 + (int(li.max()) if li.size else 0) * 4
    out = np.empty(max(cap, 1), np.int64)
    n = lib().oracle_attended_offsets(_ptr(indptr), _ptr(li), B, b, page_size, int(window),
                                      _ptr(out), out.size)
    return out[:n].copy()


def batch_decode_paged_kv(Q, pages, indptr, values, length_info, k_rope_pos_offset,
                          q_rope_position, *, q_dtype, kv_dtype, H_kv, page_size,
                          rotary_mode=0, rope_scale=1.0, rope_theta=1e4, sm_scale=None,
                          sliding_window=False, k_scale=1.0, v_scale=1.0, mask=None, sink=None,
                          k_rotated=False):
    """Returns (out [B,H_qo,D] f64, lse [B,H_qo] f64 log2 units, status).

    Q: [B,H_qo,D] typed bits; pages: [max_pages,2,H_kv,P,D] typed bits.
    ``mask`` (bool [B,H_qo]) restricts which rows are computed (others are NaN).
    ``sink`` ([H_qo], natural units): a learned logit per query head, one more softmax
    term with a zero value row.  ``k_rotated``: the cache holds K already rotated
    (``append_paged_kv_rope``); only Q is rotated.
    """
    Qb = _bits(Q, q_dtype)
    Pb = _bits(pages, kv_dtype)
    B, H_qo, D = Qb.shape
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(D)
    max_pages = Pb.shape[0]
    assert Pb.shape[1:] == (2, H_kv, page_size, D), Pb.shape
    indptr = _c(indptr, np.int32)
    values = _c(values, np.int32) if values is not None and np.size(values) else np.zeros(1, np.int32)
    li = _c(length_info, np.int32)
    kro = _c(k_rope_pos_offset if k_rope_pos_offset is not None else np.zeros(B), np.int32)
    qrp = _c(q_rope_position if q_rope_position is not None else np.zeros(B), np.int32)
    out = np.full((B, H_qo, D), np.nan)
    lse = np.full((B, H_qo), np.nan)
    m = None if mask is None else _c(mask, np.uint8)
    st = lib().oracle_batch_decode_paged_kv(
        _ptr(Qb), DTYPES[q_dtype], _ptr(Pb), DTYPES[kv_dtype], _ptr(indptr), _ptr(values),
        _ptr(li), _ptr(kro), _ptr(qrp), _ptr(out), _ptr(lse), B, H_qo, H_kv, D, page_size,
        max_pages, int(bool(sliding_window)), int(rotary_mode), float(rope_scale),
        float(rope_theta), float(sm_scale), float(k_scale), float(v_scale), int(bool(k_rotated)),
        _ptr(_sink(sink, H_qo)), _ptr(m))
    if st == -2:
        raise ValueError("oracle: bad arguments")
    return out, lse, st


def _sink(sink, H_qo):
    if sink is None:
        return None
    a = _c(sink, np.float64)
    assert a.shape == (H_qo,), a.shape
    return a


def batch_decode_paged_kv_mq(Q, pages, indptr, values, length_info, k_rope_pos_offset,
                             q_rope_position, *, q_len, q_dtype, kv_dtype, H_kv, page_size,
                             rotary_mode=0, rope_scale=1.0, rope_theta=1e4, sm_scale=None,
                             k_scale=1.0, v_scale=1.0, mask=None, sink=None, k_rotated=False):
    """Multi-query decode: returns (out [B,q_len,H_qo,D] f64, lse [B,q_len,H_qo] f64 log2
    units, status).  Q: [B,q_len,H_qo,D] typed bits (or [B*q_len,H_qo,D]); length_info
    [B] (no sliding window).  Token t of sequence b sees the attended rows
    r < L_b - q_len + 1 + t; its RoPE position is q_rope_position[b] + t.
    """
    if int(q_len) < 1:
        raise ValueError("oracle: q_len must be >= 1")
    Qb = _bits(Q, q_dtype)
    Pb = _bits(pages, kv_dtype)
    H_qo, D = Qb.shape[-2:]
    indptr = _c(indptr, np.int32)
    B = indptr.size - 1
    assert Qb.size == B * q_len * H_qo * D, (Qb.shape, B, q_len)
    Qb = Qb.reshape(B * q_len, H_qo, D)
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(D)
    max_pages = Pb.shape[0]
    assert Pb.shape[1:] == (2, H_kv, page_size, D), Pb.shape
    values = _c(values, np.int32) if values is not None and np.size(values) else np.zeros(1, np.int32)
    li = _c(length_info, np.int32)
    kro = _c(k_rope_pos_offset if k_rope_pos_offset is not None else np.zeros(B), np.int32)
    qrp = _c(q_rope_position if q_rope_position is not None else np.zeros(B), np.int32)
    out = np.full((B * q_len, H_qo, D), np.nan)
    lse = np.full((B * q_len, H_qo), np.nan)
    m = None if mask is None else _c(mask, np.uint8)
    st = lib().oracle_batch_decode_paged_kv_mq(
        _ptr(Qb), DTYPES[q_dtype], _ptr(Pb), DTYPES[kv_dtype], _ptr(indptr), _ptr(values),
        _ptr(li), _ptr(kro), _ptr(qrp), _ptr(out), _ptr(lse), B, int(q_len), H_qo, H_kv, D,
        page_size, max_pages, int(rotary_mode), float(rope_scale), float(rope_theta),
        float(sm_scale), float(k_scale), float(v_scale), int(bool(k_rotated)),
        _ptr(_sink(sink, H_qo)), _ptr(m))
    if st == -2:
        raise ValueError("oracle: bad arguments")
    return out.reshape(B, q_len, H_qo, D), lse.reshape(B, q_len, H_qo), st


def merge_state(V, S, V_other, S_other):
    """fp64 merge of two (V [N,H,D], S [N,H] log2) attention states; returns new (V, S)."""
    V = _c(V, np.float64).copy()
    S = _c(S, np.float64).copy()
    Vo = _c(V_other, np.float64)
    So = _c(S_other, np.float64)
    N, H, D = V.shape
    lib().oracle_merge_state(_ptr(V), _ptr(S), _ptr(Vo), _ptr(So), N, H, D)
    return V, S


def merge_states(V_parts, S_parts):
    """fp64 merge of R attention states at once: V_parts [R,N,H,D], S_parts [R,N,H] (log2);
    returns (V [N,H,D], S [N,H]).  All partners empty (S <= -5e4): V = 0, S = -5e4."""
    Vp = _c(V_parts, np.float64)
    Sp = _c(S_parts, np.float64)
    R, N, H, D = Vp.shape
    V = np.zeros((N, H, D), np.float64)
    S = np.zeros((N, H), np.float64)
    lib().oracle_merge_states(_ptr(Vp), _ptr(Sp), _ptr(V), _ptr(S), R, N, H, D)
    return V, S


def append_paged_kv_rope(pages, k_new, v_new, slot_mapping, positions, *, in_dtype, kv_dtype,
                         page_size, rotary_mode, rope_scale=1.0, rope_theta=1e4, k_scale=1.0,
                         v_scale=1.0):
    """append_paged_kv with each new K row rotated (fp64) at positions[t] first; returns
    (new pages bits, number of out-of-range slots skipped)."""
    Pb = _bits(pages, kv_dtype).copy()
    kb = _bits(k_new, in_dtype)
    vb = _bits(v_new, in_dtype)
    T, H_kv, D = kb.shape
    sm = _c(slot_mapping, np.int64)
    pos = _c(positions, np.int32)
    bad = lib().oracle_append_paged_kv_rope(
        _ptr(Pb), DTYPES[kv_dtype], _ptr(kb), _ptr(vb), DTYPES[in_dtype], _ptr(sm), T, H_kv, D,
        page_size, Pb.shape[0], np.float32(k_scale), np.float32(v_scale), _ptr(pos),
        int(rotary_mode), float(rope_scale), float(rope_theta))
    if bad == -2:
        raise ValueError("oracle: bad arguments")
    return Pb, bad


def append_paged_kv(pages, k_new, v_new, slot_mapping, *, in_dtype, kv_dtype, page_size,
                    k_scale=1.0, v_scale=1.0):
    """Returns (new pages bits, number of out-of-range slots skipped)."""
    Pb = _bits(pages, kv_dtype).copy()
    kb = _bits(k_new, in_dtype)
    vb = _bits(v_new, in_dtype)
    T, H_kv, D = kb.shape
    sm = _c(slot_mapping, np.int64)
    bad = lib().oracle_append_paged_kv(
        _ptr(Pb), DTYPES[kv_dtype], _ptr(kb), _ptr(vb), DTYPES[in_dtype], _ptr(sm), T, H_kv, D,
        page_size, Pb.shape[0], np.float32(k_scale), np.float32(v_scale))
    if bad == -2:
        raise ValueError("oracle: bad arguments")
    return Pb, bad
