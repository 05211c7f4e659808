"""ctypes binding of libpageddecode (include/pageddecode.h).

Argument marshalling only: tensors are turned into device pointers, shapes and
dtype codes, and every call goes to the C ABI.  The library must be built
(``__graft_entry__.build()`` or ``python -m paged_kv_decode_19_gb300.build``);
if it is missing, loading raises — there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

_LIB_PATH = _build.LIB
_lock = threading.Lock()
_lib = None

STATUS = {
    0: "PD_OK",
    1: "PD_ERR_INVALID_ARG",
    2: "PD_ERR_UNSUPPORTED",
    3: "PD_ERR_CUDA",
    4: "PD_ERR_BAD_PAGE",
    5: "PD_ERR_BAD_LENGTH",
    6: "PD_ERR_BAD_SLOT",
    7: "PD_ERR_TIMEOUT",
    8: "PD_ERR_WORKSPACE",
}
DTYPE_CODES = {
    torch.float32: 0,
    torch.float16: 1,
    torch.bfloat16: 2,
    torch.float8_e4m3fn: 3,
}
DTYPE_NAMES = {"f32": 0, "f16": 1, "bf16": 2, "e4m3": 3}

# Every entry point declared in include/pageddecode.h.
EXPORTS = (
    "pd_batch_decode_paged_kv",
    "pd_batch_decode_paged_kv_noalloc",
    "pd_batch_decode_paged_kv_mq",
    "pd_workspace_size_mq",
    "pd_append_paged_kv_rope",
    "pd_merge_state_inplace",
    "pd_merge_states",
    "pd_cp_shard_plan",
    "pd_append_paged_kv",
    "pd_workspace_size",
    "pd_workspace_init",
    "pd_release_stream_workspace",
    "pd_plan",
    "pd_check_device_errors",
    "pd_last_decode_variant",
    "pd_get_last_error_string",
    "pd_version",
)


class PDError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        self.status_name = STATUS.get(status, str(status))
        super().__init__(f"{self.status_name}: {message}")


class DecodeDesc(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32),
        ("H_qo", ctypes.c_int32),
        ("H_kv", ctypes.c_int32),
        ("D", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("q_dtype", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32),
        ("out_dtype", ctypes.c_int32),
        ("sliding_window", ctypes.c_int32),
        ("num_splits", ctypes.c_int32),
        ("max_pages", ctypes.c_int64),
        ("nnz_pages", ctypes.c_int64),
        ("max_kv_len_hint", ctypes.c_int32),
        ("k_scale", ctypes.c_float),
        ("v_scale", ctypes.c_float),
        ("flags", ctypes.c_int32),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("sink", ctypes.c_void_p),
        ("host_indptr", ctypes.c_void_p),
        ("host_length_info", ctypes.c_void_p),
    ]


def lib():
    """Load libpageddecode.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    f"libpageddecode is not built ({_LIB_PATH} missing); run "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(_LIB_PATH)
            P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
            L.pd_batch_decode_paged_kv.argtypes = [P, P, P, P, P, P, P, P, P, i32, f32, f32, f32,
                                                   ctypes.POINTER(DecodeDesc), P]
            L.pd_batch_decode_paged_kv.restype = i32
            L.pd_batch_decode_paged_kv_noalloc.argtypes = L.pd_batch_decode_paged_kv.argtypes
            L.pd_batch_decode_paged_kv_noalloc.restype = i32
            a = list(L.pd_batch_decode_paged_kv.argtypes)
            L.pd_batch_decode_paged_kv_mq.argtypes = a[:9] + [i32] + a[9:]
            L.pd_batch_decode_paged_kv_mq.restype = i32
            L.pd_workspace_size_mq.argtypes = [ctypes.POINTER(DecodeDesc), i32]
            L.pd_workspace_size_mq.restype = ctypes.c_size_t
            L.pd_merge_state_inplace.argtypes = [P, P, P, P, i32, i32, i32, i32, P]
            L.pd_merge_state_inplace.restype = i32
            L.pd_merge_states.argtypes = [P, P, P, P, i64, i64, i32, i32, i32, i32, i32, P]
            L.pd_merge_states.restype = i32
            L.pd_cp_shard_plan.argtypes = [P, P, P, P, i32, i32, i32, i32, P, P, i64, P, P]
            L.pd_cp_shard_plan.restype = i32
            L.pd_append_paged_kv.argtypes = [P, P, P, P, i32, i32, i32, i32, i64, i32, i32, f32,
                                             f32, P]
            L.pd_append_paged_kv.restype = i32
            L.pd_append_paged_kv_rope.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i64, i32,
                                                  i32, f32, f32, i32, f32, f32, P]
            L.pd_append_paged_kv_rope.restype = i32
            L.pd_workspace_size.argtypes = [ctypes.POINTER(DecodeDesc)]
            L.pd_workspace_size.restype = ctypes.c_size_t
            L.pd_workspace_init.argtypes = [P, ctypes.c_size_t, P]
            L.pd_workspace_init.restype = i32
            L.pd_release_stream_workspace.argtypes = [P]
            L.pd_release_stream_workspace.restype = i32
            L.pd_plan.argtypes = [ctypes.POINTER(DecodeDesc), i32, i32, ctypes.POINTER(i32),
                                  ctypes.POINTER(i32), ctypes.POINTER(ctypes.c_size_t)]
            L.pd_plan.restype = i32
            L.pd_check_device_errors.argtypes = [P]
            L.pd_check_device_errors.restype = i32
            L.pd_last_decode_variant.restype = ctypes.c_char_p
            L.pd_get_last_error_string.restype = ctypes.c_char_p
            L.pd_version.restype = i32
            _lib = L
    return _lib


def _check(status: int):
    if status != 0:
        raise PDError(status, lib().pd_get_last_error_string().decode())


def _ptr(t: Optional[torch.Tensor]):
    """Device address of a contiguous tensor (the C functions take it as void*)."""
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    """cudaStream_t of `stream` (a torch stream or a raw handle); None: the current stream."""
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


DECODE_EARLY_INPUTS = 1
DECODE_K_ROTATED = 2


def make_desc(Q, pages, indptr, values, length_info, out, *, num_splits=0, max_kv_len_hint=0,
              k_scale=1.0, v_scale=1.0, workspace=None, early_inputs=False,
              sink=None, k_rotated=False, host_meta=None) -> DecodeDesc:
    """host_meta: optional (indptr, length_info) numpy int32 host copies (the caller keeps
    them alive for the call)."""
    B, H_qo, D = Q.shape
    max_pages, two, H_kv, P, D2 = pages.shape
    if two != 2 or D2 != D:
        raise ValueError(f"pages must be [max_pages, 2, H_kv, P, {D}], got {tuple(pages.shape)}")
    return DecodeDesc(
        B=B, H_qo=H_qo, H_kv=H_kv, D=D, page_size=P, q_dtype=DTYPE_CODES[Q.dtype],
        kv_dtype=DTYPE_CODES[pages.dtype], out_dtype=DTYPE_CODES[out.dtype],
        sliding_window=int(length_info.dim() == 2), num_splits=int(num_splits),
        max_pages=max_pages, nnz_pages=int(values.numel()) if values is not None else 0,
        max_kv_len_hint=int(max_kv_len_hint), k_scale=float(k_scale), v_scale=float(v_scale),
        flags=(DECODE_EARLY_INPUTS if early_inputs else 0) | (DECODE_K_ROTATED if k_rotated else 0),
        workspace=None if workspace is None else workspace.data_ptr(),
        workspace_bytes=0 if workspace is None else workspace.numel() * workspace.element_size(),
        sink=_sink_ptr(sink, H_qo),
        host_indptr=None if host_meta is None else _host_i32(host_meta[0], B + 1),
        host_length_info=None if host_meta is None else _host_i32(host_meta[1], length_info.numel()))


def _host_i32(a, n):
    import numpy as np
    if not isinstance(a, np.ndarray) or a.dtype != np.int32 or not a.flags.c_contiguous or a.size != n:
        raise ValueError(f"host copies must be contiguous numpy int32 arrays of {n} entries")
    return a.__array_interface__["data"][0]


def host_meta_of(indptr, length_info):
    """Host copies (numpy int32) of a page table's indptr and length_info, for host_meta."""
    import numpy as np
    return (np.ascontiguousarray(indptr.cpu().numpy(), dtype=np.int32),
            np.ascontiguousarray(length_info.cpu().numpy(), dtype=np.int32).reshape(-1))


def _sink_ptr(sink, H_qo):
    if sink is None:
        return None
    if sink.dtype != torch.float32 or sink.numel() != H_qo or not sink.is_contiguous():
        raise ValueError("sink must be a contiguous float32 tensor of H_qo values")
    return sink.data_ptr()


def batch_decode_paged_kv(Q, pages, page_table_indptr, page_table_values, length_info,
                          k_rope_pos_offset, q_rope_position, output, lse, rotary_mode=0,
                          rope_scale=1.0, rope_theta=1e4, sm_scale=None, *, k_scale=1.0,
                          v_scale=1.0, num_splits=0, max_kv_len_hint=0, workspace=None,
                          early_inputs=False, sink=None, k_rotated=False, host_meta=None,
                          stream=None):
    """pd_batch_decode_paged_kv on device tensors; writes `output` and `lse`.
    host_meta=(indptr, length_info) numpy int32 host copies: the split is planned on the
    host (desc->host_indptr / host_length_info).
    early_inputs=True sets PD_DECODE_EARLY_INPUTS: only right after append_paged_kv (or
    another kernel that writes none of Q, the page table, lengths and positions)."""
    if sm_scale is None:
        sm_scale = Q.shape[-1] ** -0.5
    desc = make_desc(Q, pages, page_table_indptr, page_table_values, length_info, output,
                     num_splits=num_splits, max_kv_len_hint=max_kv_len_hint, k_scale=k_scale,
                     v_scale=v_scale, workspace=workspace, early_inputs=early_inputs,
                     sink=sink, k_rotated=k_rotated, host_meta=host_meta)
    _check(lib().pd_batch_decode_paged_kv(
        _ptr(Q), _ptr(pages), _ptr(page_table_indptr), _ptr(page_table_values),
        _ptr(length_info), _ptr(k_rope_pos_offset), _ptr(q_rope_position), _ptr(output),
        _ptr(lse), int(rotary_mode), float(rope_scale), float(rope_theta), float(sm_scale),
        ctypes.byref(desc), _stream(stream)))
    return output, lse


def batch_decode_paged_kv_noalloc(Q, pages, page_table_indptr, page_table_values,
                                  length_info, k_rope_pos_offset, q_rope_position, output, lse,
                                  rotary_mode=0, rope_scale=1.0, rope_theta=1e4, sm_scale=None,
                                  *, k_scale=1.0, v_scale=1.0, num_splits=0, max_kv_len_hint=0,
                                  early_inputs=False, sink=None, k_rotated=False, stream=None):
    """pd_batch_decode_paged_kv_noalloc: same result, split scratch in the library's
    static device array (no device allocation)."""
    if sm_scale is None:
        sm_scale = Q.shape[-1] ** -0.5
    desc = make_desc(Q, pages, page_table_indptr, page_table_values, length_info, output,
                     num_splits=num_splits, max_kv_len_hint=max_kv_len_hint, k_scale=k_scale,
                     v_scale=v_scale, early_inputs=early_inputs, sink=sink, k_rotated=k_rotated)
    _check(lib().pd_batch_decode_paged_kv_noalloc(
        _ptr(Q), _ptr(pages), _ptr(page_table_indptr), _ptr(page_table_values),
        _ptr(length_info), _ptr(k_rope_pos_offset), _ptr(q_rope_position), _ptr(output),
        _ptr(lse), int(rotary_mode), float(rope_scale), float(rope_theta), float(sm_scale),
        ctypes.byref(desc), _stream(stream)))
    return output, lse


def batch_decode_paged_kv_mq(Q, pages, page_table_indptr, page_table_values, length_info,
                             k_rope_pos_offset, q_rope_position, output, lse, rotary_mode=0,
                             rope_scale=1.0, rope_theta=1e4, sm_scale=None, *, k_scale=1.0,
                             v_scale=1.0, num_splits=0, max_kv_len_hint=0, workspace=None,
                             early_inputs=False, sink=None, k_rotated=False, host_meta=None,
                             stream=None):
    """pd_batch_decode_paged_kv_mq: Q [B, q_len, H_qo, D], output [B, q_len, H_qo, D],
    lse [B, q_len, H_qo]; token t of a sequence sees its rows up to itself."""
    if Q.dim() != 4:
        raise ValueError("Q must be [B, q_len, H_qo, D]")
    B, q_len, H_qo, D = Q.shape
    if sm_scale is None:
        sm_scale = D ** -0.5
    desc = make_desc(Q[:, 0], pages, page_table_indptr,
                     page_table_values, length_info, output, num_splits=num_splits,
                     max_kv_len_hint=max_kv_len_hint, k_scale=k_scale, v_scale=v_scale,
                     workspace=workspace, early_inputs=early_inputs, sink=sink,
                     k_rotated=k_rotated, host_meta=host_meta)
    _check(lib().pd_batch_decode_paged_kv_mq(
        _ptr(Q), _ptr(pages), _ptr(page_table_indptr), _ptr(page_table_values),
        _ptr(length_info), _ptr(k_rope_pos_offset), _ptr(q_rope_position), _ptr(output),
        _ptr(lse), int(q_len), int(rotary_mode), float(rope_scale), float(rope_theta),
        float(sm_scale), ctypes.byref(desc), _stream(stream)))
    return output, lse


def merge_state_inplace(V, S, V_other, S_other, stream=None):
    """pd_merge_state_inplace: V [N,H,D], S [N,H] float32 updated in place."""
    N, H, D = V.shape
    if V_other.shape != V.shape or V_other.dtype != V.dtype or S.shape != (N, H) or S_other.shape != (N, H):
        raise ValueError("merge_state_inplace: shape/dtype mismatch")
    _check(lib().pd_merge_state_inplace(_ptr(V), _ptr(S), _ptr(V_other), _ptr(S_other), N, H, D,
                                        DTYPE_CODES[V.dtype], _stream(stream)))
    return V, S


def merge_states(V_out, S_out, V_parts, S_parts, stream=None):
    """pd_merge_states: V_parts [R,N,H,D] float32, S_parts [R,N,H] float32 -> V_out [N,H,D]
    (F32/F16/BF16), S_out [N,H] float32."""
    R, N, H, D = V_parts.shape
    if V_parts.dtype != torch.float32 or S_parts.dtype != torch.float32 or S_parts.shape != (R, N, H):
        raise ValueError("merge_states: V_parts [R,N,H,D] and S_parts [R,N,H] must be float32")
    if V_out.shape != (N, H, D) or S_out.shape != (N, H) or S_out.dtype != torch.float32:
        raise ValueError("merge_states: V_out [N,H,D], S_out [N,H] float32")
    _check(lib().pd_merge_states(_ptr(V_out), _ptr(S_out), _ptr(V_parts), _ptr(S_parts),
                                 N * H * D, N * H, R, N, H, D, DTYPE_CODES[V_out.dtype],
                                 _stream(stream)))
    return V_out, S_out


def merge_states_packed(V_out, S_out, packed, stream=None):
    """pd_merge_states on R packed partials: packed [R, N*H*D + N*H] float32, each row a
    partner's outputs followed by its lse (the layout an all-gather of packed partials
    gives)."""
    N, H, D = V_out.shape
    R, width = packed.shape
    if packed.dtype != torch.float32 or width != N * H * (D + 1) or not packed.is_contiguous():
        raise ValueError("merge_states_packed: packed must be float32 [R, N*H*(D+1)]")
    base = packed.data_ptr()
    _check(lib().pd_merge_states(_ptr(V_out), _ptr(S_out), ctypes.c_void_p(base),
                                 ctypes.c_void_p(base + 4 * N * H * D), width, width, R, N, H, D,
                                 DTYPE_CODES[V_out.dtype], _stream(stream)))
    return V_out, S_out


def cp_shard_plan(indptr, values, length_info, k_rope_pos_offset, page_size, world, rank):
    """pd_cp_shard_plan on host int32 arrays: returns (indptr, values, length_info,
    k_rope_pos_offset) of rank `rank`'s page-aligned slice, as numpy int32 arrays."""
    import numpy as np
    ip = np.ascontiguousarray(indptr, np.int32)
    vals = np.ascontiguousarray(values, np.int32)
    li = np.ascontiguousarray(length_info, np.int32)
    B = len(li)
    ko = None if k_rope_pos_offset is None else np.ascontiguousarray(k_rope_pos_offset, np.int32)
    npg = ip[1:] - ip[:-1]
    cap = int(np.sum(-(-npg // world))) if B and world >= 1 else 0
    o_ip = np.zeros(B + 1, np.int32)
    o_vals = np.zeros(max(cap, 1), np.int32)
    o_li = np.zeros(B, np.int32)
    o_ko = np.zeros(B, np.int32)
    p = lambda a: None if a is None else ctypes.c_void_p(a.ctypes.data)
    _check(lib().pd_cp_shard_plan(p(ip), p(vals), p(li), p(ko), B, int(page_size), int(world),
                                  int(rank), p(o_ip), p(o_vals), cap, p(o_li), p(o_ko)))
    return o_ip, o_vals[:o_ip[-1]], o_li, o_ko


def append_paged_kv(pages, k_new, v_new, slot_mapping, k_scale=1.0, v_scale=1.0, stream=None):
    """pd_append_paged_kv: writes new tokens' K/V into their slots (in place)."""
    T, H_kv, D = k_new.shape
    max_pages, _, H2, P, D2 = pages.shape
    if v_new.shape != k_new.shape or H2 != H_kv or D2 != D or slot_mapping.dtype != torch.int64:
        raise ValueError("append_paged_kv: shape/dtype mismatch")
    _check(lib().pd_append_paged_kv(_ptr(pages), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping),
                                    T, H_kv, D, P, max_pages, DTYPE_CODES[k_new.dtype],
                                    DTYPE_CODES[pages.dtype], float(k_scale), float(v_scale),
                                    _stream(stream)))
    return pages


def check_device_errors(stream=None) -> str:
    """Synchronises and returns the device error status name ("PD_OK" if clean)."""
    st = lib().pd_check_device_errors(_stream(stream))
    return STATUS.get(st, str(st))


def workspace_size(desc: DecodeDesc) -> int:
    return int(lib().pd_workspace_size(ctypes.byref(desc)))


def append_paged_kv_rope(pages, k_new, v_new, slot_mapping, positions, rotary_mode=1,
                         rope_scale=1.0, rope_theta=1e4, k_scale=1.0, v_scale=1.0, stream=None):
    """pd_append_paged_kv_rope: appends with each K row rotated at positions[t] (int32)."""
    T, H_kv, D = k_new.shape
    max_pages, _, H2, P, D2 = pages.shape
    if v_new.shape != k_new.shape or H2 != H_kv or D2 != D or slot_mapping.dtype != torch.int64:
        raise ValueError("k_new/v_new [T,H_kv,D] must match pages; slot_mapping int64")
    if positions.dtype != torch.int32 or positions.numel() != T:
        raise ValueError("positions must be int32 [T]")
    _check(lib().pd_append_paged_kv_rope(
        _ptr(pages), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(positions), T, H_kv, D, P,
        max_pages, DTYPE_CODES[k_new.dtype], DTYPE_CODES[pages.dtype], float(k_scale),
        float(v_scale), int(rotary_mode), float(rope_scale), float(rope_theta), _stream(stream)))
    return pages


def release_stream_workspace(stream=None):
    """pd_release_stream_workspace: frees the library-managed workspace of `stream`
    (stream-ordered)."""
    _check(lib().pd_release_stream_workspace(_stream(stream)))


def workspace_init(ws: torch.Tensor, stream=None):
    _check(lib().pd_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def plan(desc: DecodeDesc, num_sms: int, ctas_per_sm: int):
    """Host-only split plan: (schedule, grid_blocks, workspace_bytes); schedule 0 =
    balanced shares of all pages, 1 = one block per (sequence, head slice)."""
    c, g, w = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_size_t()
    _check(lib().pd_plan(ctypes.byref(desc), num_sms, ctas_per_sm, ctypes.byref(c),
                         ctypes.byref(g), ctypes.byref(w)))
    return c.value, g.value, w.value


def last_decode_variant() -> str:
    return lib().pd_last_decode_variant().decode()


def version() -> int:
    return int(lib().pd_version())
