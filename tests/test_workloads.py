"""Seeded input generators: structure of the drawn workloads (CPU only)."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_19_gb300 import workloads as W


@pytest.mark.parametrize("name", list(W.SPECS))
def test_reduced_workload_structure(name):
    wl = W.make(name, seed=3, reduced=True)
    s = wl.spec
    ip = wl.indptr.numpy()
    assert ip[0] == 0 and np.all(np.diff(ip) >= 0)
    vals = wl.values.numpy()[: ip[-1]]
    assert len(np.unique(vals)) == len(vals)               # no page shared
    assert vals.min() >= 0 and vals.max() < wl.max_pages
    npages = np.diff(ip)
    assert np.array_equal(npages, (wl.seq_len + s.page_size - 1) // s.page_size)
    li = wl.length_info.numpy()
    last = li if s.window is None else li[0]
    assert np.all((last >= 1) & (last <= s.page_size))
    for b in range(s.B):
        offs = oracle.attended_offsets(ip, li, b, s.page_size, s.window is not None)
        assert len(offs) == wl.attended[b]
        assert np.all(np.diff(offs) > 0) and offs.max() < wl.seq_len[b]
    assert wl.Q.dtype == W.TORCH_DTYPES[s.q_dtype]
    assert wl.pages.dtype == W.TORCH_DTYPES[s.kv_dtype]


def test_seed_determinism():
    a = W.make("llama3_8b_bf16", seed=5, reduced=True)
    b = W.make("llama3_8b_bf16", seed=5, reduced=True)
    assert torch.equal(a.pages.view(torch.int16), b.pages.view(torch.int16))
    assert torch.equal(a.values, b.values)


def test_fp8_workload_scales_and_append_slots():
    wl = W.make("fp8_kv_highconc", seed=1, reduced=True)
    assert 0 < wl.k_scale < 0.1 and 0 < wl.v_scale < 0.1
    P = wl.spec.page_size
    ip, vals = wl.indptr.numpy(), wl.values.numpy()
    for b, slot in enumerate(wl.slot_mapping.numpy()):
        row = wl.seq_len[b] - 1
        assert slot == vals[ip[b] + row // P] * P + row % P


def test_external_split_covers_every_page_once():
    wl = W.make("long_ctx_bf16", seed=2, reduced=True)
    ip, vals = wl.indptr.numpy(), wl.values.numpy()
    ipc, valc, lastc, koff, owner = W.split_chunks(ip, vals, wl.seq_len, 16, 32)
    for b in range(wl.spec.B):
        sel = np.nonzero(owner == b)[0]
        assert 1 <= len(sel) <= 32
        got = np.concatenate([valc[ipc[j]:ipc[j + 1]] for j in sel])
        assert np.array_equal(got, vals[ip[b]:ip[b + 1]])
        rows = sum((ipc[j + 1] - ipc[j] - 1) * 16 + lastc[j] for j in sel)
        assert rows == wl.seq_len[b]


def test_stress_inputs_move_the_running_max():
    """The score-shaping inputs do what the rescale tests rely on: along most (sequence,
    head) rows, some later score exceeds the maximum of the first 16 rows by more than
    2^8 (8 in log2 units), so an online softmax must rescale a non-empty state."""
    l2e = 1.4426950408889634
    for over in (dict(k_ramp=8.0), dict(q_gain=8.0), dict(k_ramp=4.0)):
        wl = W.make("llama3_8b_bf16", seed=201, reduced=True, rotary_mode=0, H_kv=2, H_qo=8,
                    **over)
        s = wl.spec
        Q = wl.Q.float().numpy()
        pages = wl.pages.float().numpy()
        ip, vals = wl.indptr.numpy(), wl.values.numpy()
        moved = total = 0
        for b in range(s.B):
            L = int(wl.seq_len[b])
            if L <= 16:
                continue
            rows = np.arange(L)
            pg = vals[ip[b] + rows // s.page_size]
            for h in range(s.H_qo):
                K = pages[pg, 0, h // (s.H_qo // s.H_kv), rows % s.page_size]
                sc = (K @ Q[b, h]) * wl.sm_scale * l2e
                total += 1
                moved += int(sc[16:].max() - sc[:16].max() > 8.0)
        assert moved >= 0.5 * total, (over, moved, total)
