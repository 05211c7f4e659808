"""C-ABI checks that need no GPU: the library loads, exports every entry point that
include/pageddecode.h declares, the struct layout matches, host-side validation
rejects bad arguments before any CUDA call, and the split planner's arithmetic."""
import ctypes
import os
import re

import pytest
import torch

import __graft_entry__
from paged_kv_decode_19_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pageddecode.h")


@pytest.fixture(scope="module")
def L():
    __graft_entry__.build()
    return _lib.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pd_[a-z_]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(_lib.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
    assert L.pd_version() == 10100


def test_desc_layout_matches_header():
    # int32 x10, int64 x2, int32, float x2, int32, void*, size_t, const float*,
    # const int32_t* x2
    assert ctypes.sizeof(_lib.DecodeDesc) == 112
    assert _lib.DecodeDesc.sink.offset == 88
    assert _lib.DecodeDesc.host_indptr.offset == 96
    assert _lib.DecodeDesc.host_length_info.offset == 104
    assert _lib.DecodeDesc.max_pages.offset == 40
    assert _lib.DecodeDesc.flags.offset == 68
    assert _lib.DecodeDesc.workspace.offset == 72
    text = open(HEADER).read()
    assert re.search(r"#define PD_DECODE_EARLY_INPUTS (\d+)", text).group(1) == str(_lib.DECODE_EARLY_INPUTS)
    assert re.search(r"#define PD_DECODE_K_ROTATED (\d+)", text).group(1) == str(_lib.DECODE_K_ROTATED)


def _desc(**kw):
    d = dict(B=4, H_qo=8, H_kv=2, D=128, page_size=16, q_dtype=2, kv_dtype=2, out_dtype=2,
             sliding_window=0, num_splits=0, max_pages=100, nnz_pages=40, max_kv_len_hint=0,
             k_scale=1.0, v_scale=1.0, workspace=None, workspace_bytes=0, sink=None)
    d.update(kw)
    return _lib.DecodeDesc(**d)


@pytest.mark.parametrize("bad,status", [
    (dict(H_qo=7), "PD_ERR_INVALID_ARG"), (dict(D=96), "PD_ERR_UNSUPPORTED"),
    (dict(page_size=0), "PD_ERR_INVALID_ARG"), (dict(q_dtype=3), "PD_ERR_INVALID_ARG"),
    (dict(out_dtype=3), "PD_ERR_INVALID_ARG"), (dict(kv_dtype=3, k_scale=0.0), "PD_ERR_INVALID_ARG"),
    (dict(kv_dtype=1), "PD_ERR_UNSUPPORTED"), (dict(num_splits=-2), "PD_ERR_INVALID_ARG"),
    (dict(max_pages=0), "PD_ERR_INVALID_ARG"), (dict(B=-1), "PD_ERR_INVALID_ARG"),
    (dict(flags=4), "PD_ERR_INVALID_ARG"), (dict(page_size=257), "PD_ERR_INVALID_ARG"),
    (dict(H_kv=0), "PD_ERR_INVALID_ARG"), (dict(nnz_pages=-1), "PD_ERR_INVALID_ARG"),
    (dict(max_pages=1 << 30, H_kv=2, H_qo=8), "PD_ERR_UNSUPPORTED"),
    (dict(kv_dtype=3, v_scale=float("inf")), "PD_ERR_INVALID_ARG"),
    (dict(kv_dtype=3, k_scale=float("nan")), "PD_ERR_INVALID_ARG"),
])
def test_decode_validation_without_gpu(L, bad, status):
    d = _desc(**bad)
    st = L.pd_batch_decode_paged_kv(None, None, None, None, None, None, None, None, None, 0,
                                    1.0, 1e4, 0.1, ctypes.byref(d), None)
    assert _lib.STATUS[st] == status, L.pd_get_last_error_string()


def test_unknown_flag_bits_rejected(L):
    d = _desc(flags=4)
    st = L.pd_batch_decode_paged_kv(None, None, None, None, None, None, None, None, None, 0,
                                    1.0, 1e4, 0.1, ctypes.byref(d), None)
    assert _lib.STATUS[st] == "PD_ERR_INVALID_ARG" and b"flags" in L.pd_get_last_error_string()


def test_append_rope_validation_without_gpu(L):
    f = L.pd_append_paged_kv_rope
    args = lambda mode, D=64, pos=None: (None, None, None, None, pos, 3, 2, D, 16, 10, 2, 2, 1.0,
                                         1.0, mode, 1.0, 1e4, None)
    assert _lib.STATUS[f(*args(0))] == "PD_ERR_INVALID_ARG"
    assert _lib.STATUS[f(*args(3))] == "PD_ERR_INVALID_ARG"
    assert _lib.STATUS[f(*args(1))] == "PD_ERR_INVALID_ARG"  # no positions
    assert _lib.STATUS[f(*args(1, D=63, pos=ctypes.c_void_p(64)))] == "PD_ERR_UNSUPPORTED"


def test_decode_rotary_mode_range(L):
    d = _desc()
    st = L.pd_batch_decode_paged_kv(None, None, None, None, None, None, None, None, None, 3,
                                    1.0, 1e4, 0.1, ctypes.byref(d), None)
    assert _lib.STATUS[st] == "PD_ERR_INVALID_ARG" and b"0, 1 or 2" in L.pd_get_last_error_string()


def test_decode_null_pointers_rejected(L):
    d = _desc()
    st = L.pd_batch_decode_paged_kv(None, None, None, None, None, None, None, None, None, 0,
                                    1.0, 1e4, 0.1, ctypes.byref(d), None)
    assert _lib.STATUS[st] == "PD_ERR_INVALID_ARG"
    st = L.pd_batch_decode_paged_kv(None, None, None, None, None, None, None, None, None, 1,
                                    1.0, 1e4, 0.1, ctypes.byref(d), None)
    assert _lib.STATUS[st] == "PD_ERR_INVALID_ARG"
    assert b"RoPE" in L.pd_get_last_error_string()


def test_decode_rejects_unaligned_q_or_pages(L):
    # the kernels read Q and K/V rows with 16-byte vector loads: a pointer that is only
    # element-aligned must be refused on the host, before any CUDA call (the pointers
    # below are never dereferenced)
    d = _desc()
    p = ctypes.c_void_p
    args = lambda q, pages: (p(q), p(pages), p(64), p(128), p(192), None, None, p(256), p(320), 0,
                             1.0, 1e4, 0.1, ctypes.byref(d), None)
    st = L.pd_batch_decode_paged_kv(*args(4096, 8194))
    assert _lib.STATUS[st] == "PD_ERR_INVALID_ARG" and b"16-byte" in L.pd_get_last_error_string()
    st = L.pd_batch_decode_paged_kv(*args(4098, 8192))
    assert _lib.STATUS[st] == "PD_ERR_INVALID_ARG" and b"16-byte" in L.pd_get_last_error_string()


def test_merge_and_append_validation_without_gpu(L):
    assert _lib.STATUS[L.pd_merge_state_inplace(None, None, None, None, 2, 2, 64, 3, None)] == "PD_ERR_INVALID_ARG"
    assert _lib.STATUS[L.pd_merge_state_inplace(None, None, None, None, 2, 2, 64, 0, None)] == "PD_ERR_INVALID_ARG"
    assert L.pd_merge_state_inplace(None, None, None, None, 0, 2, 64, 0, None) == 0
    assert _lib.STATUS[L.pd_append_paged_kv(None, None, None, None, 3, 2, 64, 16, 10, 3, 2, 1.0, 1.0, None)] == "PD_ERR_INVALID_ARG"
    assert _lib.STATUS[L.pd_append_paged_kv(None, None, None, None, 3, 2, 64, 16, 10, 2, 3, 0.0, 1.0, None)] == "PD_ERR_INVALID_ARG"
    assert L.pd_append_paged_kv(None, None, None, None, 0, 2, 64, 16, 10, 2, 2, 1.0, 1.0, None) == 0


def test_planner_arithmetic(L):
    # llama3-8b-shaped bf16 decode: the tensor-core kernel, 4 independent workers (warps)
    # per block
    d = _desc(B=32, H_qo=32, H_kv=8, nnz_pages=4608, max_pages=16384)
    mode, grid, ws = _lib.plan(d, 148, 3)
    assert mode == 0 and grid == 148 * 3  # balanced: one resident wave
    # counters for 32 x 8 segments + two partial (lse, out[D]) slots per worker
    assert ws >= 32 * 8 * 4 + 2 * grid * 4 * 8 * (128 + 1) * 4
    # num_splits = 1: one worker per (sequence, head slice), no workspace
    m1, g1, w1 = _lib.plan(_desc(B=32, H_qo=32, H_kv=8, nnz_pages=4608, num_splits=1), 148, 3)
    assert m1 == 1 and g1 == 32 * 8 // 4 and w1 == 0
    # group 16: two 8-head slices per KV head -> 16 segments -> 4 blocks of 4 workers
    m2, g2, _ = _lib.plan(_desc(B=4, H_qo=32, H_kv=2, nnz_pages=100, num_splits=1), 148, 3)
    assert g2 == (4 * 2 * 2) // 4
    # n > 1: about n workers per segment (8 x 2 segments x 32), capped at 8 waves
    _, g3, _ = _lib.plan(_desc(B=8, nnz_pages=40000, num_splits=32), 148, 3)
    assert g3 == min(8 * 2 * 32, 8 * 148 * 3 * 4) // 4
    # an fp32 cache runs the SIMT kernel: one worker per block
    _, g5, w5 = _lib.plan(_desc(B=8, nnz_pages=40000, num_splits=32, q_dtype=0, kv_dtype=0,
                                out_dtype=0), 148, 3)
    assert g5 == min(8 * 2 * 32, 8 * 148 * 3)
    assert w5 >= 2 * g5 * 8 * (128 + 1) * 4
    # tiny problems never get more workers than work units (rounded up to a block)
    _, g4, _ = _lib.plan(_desc(B=2, H_qo=8, H_kv=2, nnz_pages=3), 148, 3)
    assert g4 <= -(-(3 + 2) * 2 // 4)


def test_python_binding_rejects_missing_library(tmp_path, monkeypatch):
    monkeypatch.setattr(_lib, "_LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        _lib.lib()


def test_multi_query_validation_without_gpu(L):
    d = _desc()
    args = lambda q_len, dd: (None, None, None, None, None, None, None, None, None, q_len, 0, 1.0,
                              1e4, 0.1, ctypes.byref(dd), None)
    assert _lib.STATUS[L.pd_batch_decode_paged_kv_mq(*args(0, d))] == "PD_ERR_INVALID_ARG"
    dw = _desc(sliding_window=1)
    assert _lib.STATUS[L.pd_batch_decode_paged_kv_mq(*args(2, dw))] == "PD_ERR_UNSUPPORTED"
    # the desc is validated as for the single-token entry point
    assert _lib.STATUS[L.pd_batch_decode_paged_kv_mq(*args(2, _desc(D=96)))] == "PD_ERR_UNSUPPORTED"
    assert L.pd_batch_decode_paged_kv_mq(*args(2, _desc(B=0))) == 0


def test_plain_c_caller(L, tmp_path):
    # the boundary is a C ABI: a C program compiled against include/pageddecode.h and
    # linked with the library sees the same planner and validation results
    import subprocess
    so = _lib._LIB_PATH
    exe = tmp_path / "abi_check"
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                           os.path.join(ROOT, "tests", "c", "abi_check.c"), so, "-o", str(exe),
                           "-Wl,-rpath," + os.path.dirname(so)])
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout
    invalid = {v: k for k, v in _lib.STATUS.items()}["PD_ERR_INVALID_ARG"]
    lines = out.strip().splitlines()
    assert lines[0] == f"version {L.pd_version()}"
    mode, grid, ws = _lib.plan(_desc(B=32, H_qo=32, H_kv=8, nnz_pages=4608, max_pages=16384), 152, 2)
    assert lines[1] == f"plan 0 schedule {mode} grid {grid} workspace {ws}"
    assert lines[2].startswith(f"bad heads {invalid} ") and "H_kv" in lines[2]
    assert lines[3] == f"bad flags {invalid}"
    assert lines[4] == f"bad q_len {invalid}"
    assert lines[5] == f"host alone {invalid}"
    assert lines[6] == f"host decreasing {invalid}"
    # the C compiler's layout of the descriptor is the binding's
    assert lines[7] == (f"desc {ctypes.sizeof(_lib.DecodeDesc)} {_lib.DecodeDesc.host_indptr.offset} "
                        f"{_lib.DecodeDesc.host_length_info.offset}")


def test_stream_workspace_arena_bookkeeping(tmp_path):
    # the per-stream arenas of the library-managed workspace, with fake stream-ordered
    # allocator calls (tests/c/arena_check.cpp): separate buffers per stream, growth
    # that allocates first and releases the old buffer on its stream, zeroed counters,
    # unchanged arena after a failed allocation, release of both buffers once
    import subprocess
    exe = tmp_path / "arena_check"
    subprocess.check_call(["g++", "-std=c++17", "-Wall", "-Werror", "-I",
                           os.path.join(ROOT, "paged_kv_decode_19_gb300", "csrc"),
                           os.path.join(ROOT, "tests", "c", "arena_check.cpp"), "-o", str(exe)])
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == "arena bookkeeping ok"
