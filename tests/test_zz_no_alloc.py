"""pd_batch_decode_paged_kv_noalloc — the decode entry point for callers that cannot
allocate device memory (its split scratch is a static array inside the library).

Called straight through the C ABI (ctypes), twice in a row, and compared both with the
fp64 oracle and with the regular pd_batch_decode_paged_kv on the same inputs, within
the bf16 decode tolerance (max |out| error 2e-2, max |lse| error 2e-3).  The device's
free memory must not change across the calls after the first (the first may load the
library's device code, which holds the static array).  This file is collected last so
that a failure here stops a -x run only after every other test has run; it also passes
on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from paged_kv_decode_19_gb300 import _lib
from paged_kv_decode_19_gb300 import workloads as W
from tests._util import compare, oracle_decode

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _call(fn, wl, out, lse, desc):
    s = wl.spec
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = fn(p(wl.Q), p(wl.pages), p(wl.indptr), p(wl.values), p(wl.length_info),
            p(wl.k_rope_pos_offset), p(wl.q_rope_position), p(out), p(lse), s.rotary_mode,
            ctypes.c_float(s.rope_scale), ctypes.c_float(s.rope_theta),
            ctypes.c_float(wl.sm_scale), ctypes.byref(desc),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


def test_noalloc_matches_regular_entry_point_twice():
    import __graft_entry__
    __graft_entry__.build()
    L = _lib.lib()
    wl = W.make("llama3_8b_bf16", seed=21, reduced=True).to(DEV)
    s = wl.spec
    shape = (s.B, s.H_qo, s.D)
    ref_out = torch.empty(shape, dtype=torch.bfloat16, device=DEV)
    ref_lse = torch.empty((s.B, s.H_qo), dtype=torch.float32, device=DEV)
    # several chunks per sequence, so the split scratch (counters + partials) is used
    hint = int(wl.attended.max())
    desc = _lib.make_desc(wl.Q, wl.pages, wl.indptr, wl.values, wl.length_info, ref_out,
                          num_splits=6, max_kv_len_hint=hint)
    assert L.pd_workspace_size(ctypes.byref(desc)) > 0
    assert _call(L.pd_batch_decode_paged_kv, wl, ref_out, ref_lse, desc) == 0
    assert L.pd_check_device_errors(None) == 0
    ro, rl, st = oracle_decode(wl)
    assert st == 0
    # outputs of the calls below allocated up front: nothing else allocates meanwhile
    outs = [torch.full(shape, float("nan"), dtype=torch.bfloat16, device=DEV) for _ in range(3)]
    lses = [torch.full((s.B, s.H_qo), float("nan"), dtype=torch.float32, device=DEV)
            for _ in range(3)]
    torch.cuda.synchronize()
    free = []
    for out, lse in zip(outs, lses):
        st = _call(L.pd_batch_decode_paged_kv_noalloc, wl, out, lse, desc)
        assert st == 0, L.pd_get_last_error_string()
        assert L.pd_check_device_errors(None) == 0
        torch.cuda.synchronize()
        free.append(torch.cuda.mem_get_info()[0])
    assert free[1:] == free[:1] * (len(free) - 1), free
    for out, lse in zip(outs, lses):
        compare("bf16", out, lse, ro, rl)
        eo = (out.float() - ref_out.float()).abs().max().item()
        el = (lse - ref_lse).abs().max().item()
        assert np.isfinite(eo) and eo <= 2e-2, eo
        assert np.isfinite(el) and el <= 2e-3, el


def test_noalloc_rejects_scratch_beyond_its_maximum():
    L = _lib.lib()
    # 1100 sequences x 8 KV heads asked to split 64 ways: several thousand blocks, two
    # partial (out, lse) slots each -- more than the 16 MiB array holds (the inputs are
    # real, so even a wrongly accepted call would stay in bounds)
    wl = W.make("llama3_8b_bf16", seed=22, reduced=True, B=1100, len_dist=("uniform", 1, 40),
                pool=4000).to(DEV)
    out = torch.empty((wl.spec.B, wl.spec.H_qo, wl.spec.D), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((wl.spec.B, wl.spec.H_qo), dtype=torch.float32, device=DEV)
    desc = _lib.make_desc(wl.Q, wl.pages, wl.indptr, wl.values, wl.length_info, out, num_splits=64)
    assert L.pd_workspace_size(ctypes.byref(desc)) > (16 << 20)
    st = _call(L.pd_batch_decode_paged_kv_noalloc, wl, out, lse, desc)
    assert _lib.STATUS[st] == "PD_ERR_WORKSPACE"
    assert b"16 MiB" in L.pd_get_last_error_string()
    # a caller-supplied workspace is refused (this entry point never takes one)
    ws = torch.empty(1024, dtype=torch.uint8, device=DEV)
    desc2 = _lib.make_desc(wl.Q, wl.pages, wl.indptr, wl.values, wl.length_info, out, workspace=ws)
    assert _lib.STATUS[_call(L.pd_batch_decode_paged_kv_noalloc, wl, out, lse, desc2)] == "PD_ERR_INVALID_ARG"
