"""GPU parity of the multi-query decode (pd_batch_decode_paged_kv_mq: q_len query tokens
per sequence, causal among the new tokens) against the fp64 oracle's multi-query form."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_19_gb300 import workloads as W
from tests._util import compare

pd = pytest.importorskip("paged_kv_decode_19_gb300")
pytestmark = pytest.mark.gpu

DEV = "cuda"


def _mq(name, seed, q_len, **kw):
    """A reduced workload plus q_len query tokens per sequence: Q [B, q_len, H_qo, D],
    token t at RoPE position max(L - q_len, 0) + t (its own row's position)."""
    wl = W.make(name, seed=seed, reduced=True, **kw).to(DEV)
    s = wl.spec
    g = torch.Generator(device=DEV)
    g.manual_seed(seed + 7)
    Q = torch.randn((s.B, q_len, s.H_qo, s.D), generator=g, device=DEV).to(W.TORCH_DTYPES[s.q_dtype])
    qpos = np.maximum(wl.attended - q_len, 0).astype(np.int32)
    wl.q_rope_position = torch.from_numpy(qpos).to(DEV)
    return wl, Q


def _oracle(wl, Q, q_len, pages=None):
    s = wl.spec
    return oracle.batch_decode_paged_kv_mq(
        W.bits(Q), W.bits(wl.pages) if pages is None else pages, wl.indptr.cpu().numpy(),
        wl.values.cpu().numpy(), wl.length_info.cpu().numpy(), wl.k_rope_pos_offset.cpu().numpy(),
        wl.q_rope_position.cpu().numpy(), q_len=q_len, q_dtype=s.q_dtype, kv_dtype=s.kv_dtype,
        H_kv=s.H_kv, page_size=s.page_size, rotary_mode=s.rotary_mode, rope_scale=s.rope_scale,
        rope_theta=s.rope_theta, sm_scale=wl.sm_scale, k_scale=wl.k_scale, v_scale=wl.v_scale)


def _gpu(wl, Q, **kw):
    s = wl.spec
    B, q_len = Q.shape[:2]
    out = torch.full((B, q_len, s.H_qo, s.D), float("nan"), dtype=W.TORCH_DTYPES[s.out_dtype], device=DEV)
    lse = torch.full((B, q_len, s.H_qo), float("nan"), dtype=torch.float32, device=DEV)
    pd.batch_decode_paged_kv_mq(Q, wl.pages, wl.indptr, wl.values, wl.length_info,
                                wl.k_rope_pos_offset, wl.q_rope_position, out, lse, s.rotary_mode,
                                s.rope_scale, s.rope_theta, wl.sm_scale, k_scale=wl.k_scale,
                                v_scale=wl.v_scale, **kw)
    return out, lse


def _check(wl, Q, **kw):
    q_len = Q.shape[1]
    out, lse = _gpu(wl, Q, **kw)
    assert pd.check_device_errors() == "PD_OK"
    assert pd.last_decode_variant() == "mma"
    ro, rl, st = _oracle(wl, Q, q_len)
    assert st == 0
    return compare(wl.spec.kv_dtype, out, lse, ro, rl)


@pytest.mark.parametrize("name,over", [("llama3_8b_bf16", {}),
                                       ("window_sink_f16", dict(window=None, sink=0)),
                                       ("fp8_kv_highconc", {})])
@pytest.mark.parametrize("q_len", [2, 3, 5])
def test_mq_matches_oracle(name, over, q_len):
    wl, Q = _mq(name, 30 + q_len, q_len, **over)
    _check(wl, Q)
    _check(wl, Q, num_splits=1)
    _check(wl, Q, num_splits=3, max_kv_len_hint=int(wl.attended.max()))


@pytest.mark.parametrize("kv", ["bf16", "f16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("group,q_len", [(1, 4), (2, 3), (4, 2), (8, 2), (12, 3), (4, 4), (2, 8),
                                         (8, 4), (4, 8), (16, 2), (8, 3)])
def test_mq_group_sweep(kv, D, group, q_len):
    # columns = q_len x group per KV head, cut into slices of <= 8 (packed below 5); 16 and
    # 32 columns (two or four slices) run as grouped slices whose warps walk the same pages
    # side by side, 24 and 36 columns as separate segments
    wl, Q = _mq("llama3_8b_bf16", 50 + group, q_len, q_dtype=kv, kv_dtype=kv, out_dtype=kv, D=D,
                H_kv=2, H_qo=2 * group, B=3, len_dist=("uniform", 1, 300), pool=200,
                rotary_mode=int(group % 2 == 0))
    _check(wl, Q)
    _check(wl, Q, num_splits=4, max_kv_len_hint=300)


@pytest.mark.parametrize("q_len", [2, 4])
def test_mq_fp8_rope_grouped_slices(q_len):
    """FP8 KV with rotate-half RoPE at group 8: 16 or 32 query columns run as grouped
    slices whose warps each rotate a share of every K tile and exchange the rest."""
    wl, Q = _mq("fp8_kv_highconc", 70 + q_len, q_len, rotary_mode=1, rope_theta=1e4)
    _check(wl, Q)
    _check(wl, Q, num_splits=3, max_kv_len_hint=int(wl.attended.max()))


@pytest.mark.parametrize("P,q_len", [(64, 3), (256, 5)])
def test_mq_large_pages(P, q_len):
    """Multi-query decode on pages of several 16-row tiles (the causal limit of the
    new tokens then falls inside a tile of the last page)."""
    wl, Q = _mq("llama3_8b_bf16", 50 + P, q_len, page_size=P, pool="fit")
    _check(wl, Q)
    _check(wl, Q, num_splits=3, max_kv_len_hint=int(wl.attended.max()))


def test_mq_q_len_one_is_the_decode():
    wl, Q = _mq("llama3_8b_bf16", 61, 1)
    out1, lse1 = _gpu(wl, Q)
    s = wl.spec
    out = torch.empty((s.B, s.H_qo, s.D), dtype=W.TORCH_DTYPES[s.out_dtype], device=DEV)
    lse = torch.empty((s.B, s.H_qo), dtype=torch.float32, device=DEV)
    pd.batch_decode_paged_kv(Q[:, 0].contiguous(), wl.pages, wl.indptr, wl.values, wl.length_info,
                             wl.k_rope_pos_offset, wl.q_rope_position, out, lse, s.rotary_mode,
                             s.rope_scale, s.rope_theta, wl.sm_scale)
    assert torch.equal(out1[:, 0], out) and torch.equal(lse1[:, 0], lse)


def test_mq_sequences_shorter_than_q_len():
    # tokens whose causal limit is <= 0 see no row: out = 0, lse = -5e4
    q_len = 4
    wl, Q = _mq("llama3_8b_bf16", 62, q_len, B=7, len_dist=("uniform", 1, 1), pool=64)
    lens = np.array([0, 1, 2, 3, 4, 16, 17], np.int64)
    P = wl.spec.page_size
    npages = (lens + P - 1) // P
    ip = np.concatenate([[0], np.cumsum(npages)]).astype(np.int32)
    vals = np.random.default_rng(3).permutation(wl.max_pages)[: npages.sum()].astype(np.int32)
    last = np.where(npages > 0, lens - (npages - 1) * P, 0).astype(np.int32)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    wl.indptr, wl.values, wl.length_info = t(ip), t(vals), t(last)
    wl.attended = lens
    wl.q_rope_position = t(np.maximum(lens - q_len, 0).astype(np.int32))
    wl.k_rope_pos_offset = t(np.zeros(len(lens), np.int32))
    out, lse = _gpu(wl, Q)
    ro, rl, _ = _oracle(wl, Q, q_len)
    compare("bf16", out, lse, ro, rl)
    assert torch.all(out[0] == 0) and torch.all(lse[0] == -5e4)
    assert torch.all(lse[1, :3] == -5e4) and torch.all(lse[1, 3] > -5e4)


def test_mq_caller_workspace():
    q_len = 3
    wl, Q = _mq("llama3_8b_bf16", 63, q_len)
    s = wl.spec
    out0 = torch.empty((s.B, q_len, s.H_qo, s.D), dtype=torch.bfloat16, device=DEV)
    desc = pd.make_desc(Q[:, 0], wl.pages, wl.indptr, wl.values, wl.length_info, out0)
    n = pd._lib.lib().pd_workspace_size_mq(desc, q_len)
    assert n >= pd._lib.lib().pd_workspace_size(desc) > 0
    ws = torch.empty(n, dtype=torch.uint8, device=DEV)
    pd.workspace_init(ws)
    _check(wl, Q, workspace=ws)


def test_mq_after_append_with_early_inputs():
    # the q_len new tokens are appended (rows L - q_len .. L - 1), then the multi-query
    # decode starts under the append (PD_DECODE_EARLY_INPUTS)
    q_len = 3
    wl, Q = _mq("llama3_8b_bf16", 64, q_len, len_dist=("uniform", 5, 700))
    s = wl.spec
    ip = wl.indptr.cpu().numpy()
    vals = wl.values.cpu().numpy()
    P = s.page_size
    slots = []
    for b in range(s.B):
        for j in range(q_len):
            r = int(wl.seq_len[b]) - q_len + j
            slots.append(int(vals[ip[b] + r // P]) * P + r % P)
    g = torch.Generator(device=DEV)
    g.manual_seed(65)
    k_new = torch.randn((s.B * q_len, s.H_kv, s.D), generator=g, device=DEV).to(torch.bfloat16)
    v_new = torch.randn((s.B * q_len, s.H_kv, s.D), generator=g, device=DEV).to(torch.bfloat16)
    sm = torch.tensor(slots, dtype=torch.int64, device=DEV)
    ref_pages, bad = oracle.append_paged_kv(W.bits(wl.pages), W.bits(k_new), W.bits(v_new),
                                            np.array(slots, np.int64), in_dtype="bf16",
                                            kv_dtype="bf16", page_size=P)
    assert bad == 0
    pd.append_paged_kv(wl.pages, k_new, v_new, sm)
    out, lse = _gpu(wl, Q, early_inputs=True)
    torch.cuda.synchronize()
    assert pd.check_device_errors() == "PD_OK"
    ro, rl, _ = _oracle(wl, Q, q_len, pages=ref_pages)
    compare("bf16", out, lse, ro, rl)


def test_mq_interleaved_rope():
    wl, Q = _mq("llama3_8b_bf16", 66, 2, rotary_mode=2)
    _check(wl, Q)
    _check(wl, Q, num_splits=3, max_kv_len_hint=int(wl.attended.max()))


@pytest.mark.parametrize("splits", [0, 3])
def test_mq_sink_logits(splits):
    q_len = 2
    wl, Q = _mq("llama3_8b_bf16", 67, q_len)
    g = torch.Generator(device=DEV)
    g.manual_seed(68)
    sk = (torch.randn(wl.spec.H_qo, generator=g, device=DEV) * 3).float()
    kw = dict(num_splits=splits, max_kv_len_hint=int(wl.attended.max())) if splits else {}
    out, lse = _gpu(wl, Q, sink=sk, **kw)
    s = wl.spec
    ro, rl, _ = oracle.batch_decode_paged_kv_mq(
        W.bits(Q), W.bits(wl.pages), wl.indptr.cpu().numpy(), wl.values.cpu().numpy(),
        wl.length_info.cpu().numpy(), wl.k_rope_pos_offset.cpu().numpy(),
        wl.q_rope_position.cpu().numpy(), q_len=q_len, q_dtype=s.q_dtype, kv_dtype=s.kv_dtype,
        H_kv=s.H_kv, page_size=s.page_size, rotary_mode=s.rotary_mode, rope_scale=s.rope_scale,
        rope_theta=s.rope_theta, sm_scale=wl.sm_scale, sink=sk.cpu().numpy())
    compare("bf16", out, lse, ro, rl)


@pytest.mark.parametrize("splits", [0, 3])
def test_mq_fp8_interleaved_with_sinks(splits):
    # the next-row features together: E4M3 cache, 2 query tokens, interleaved RoPE,
    # per-head sinks, internal splits
    q_len = 2
    wl, Q = _mq("fp8_kv_highconc", 69, q_len, rotary_mode=2, rope_theta=1e4)
    s = wl.spec
    g = torch.Generator(device=DEV)
    g.manual_seed(70)
    sk = (torch.randn(s.H_qo, generator=g, device=DEV) * 3).float()
    kw = dict(num_splits=splits, max_kv_len_hint=int(wl.attended.max())) if splits else {}
    out, lse = _gpu(wl, Q, sink=sk, **kw)
    assert pd.check_device_errors() == "PD_OK"
    ro, rl, _ = oracle.batch_decode_paged_kv_mq(
        W.bits(Q), W.bits(wl.pages), wl.indptr.cpu().numpy(), wl.values.cpu().numpy(),
        wl.length_info.cpu().numpy(), wl.k_rope_pos_offset.cpu().numpy(),
        wl.q_rope_position.cpu().numpy(), q_len=q_len, q_dtype=s.q_dtype, kv_dtype=s.kv_dtype,
        H_kv=s.H_kv, page_size=s.page_size, rotary_mode=2, rope_scale=s.rope_scale,
        rope_theta=s.rope_theta, sm_scale=wl.sm_scale, k_scale=wl.k_scale, v_scale=wl.v_scale,
        sink=sk.cpu().numpy())
    compare("e4m3", out, lse, ro, rl)


def test_mq_k_rotated_cache_with_sinks_and_early_inputs():
    # K rotated in the cache (Q-only RoPE), sinks, two tokens, the decode started under
    # the previous kernel: the synthetic cache stands for already-rotated K rows
    q_len = 2
    wl, Q = _mq("llama3_8b_bf16", 71, q_len)
    s = wl.spec
    g = torch.Generator(device=DEV)
    g.manual_seed(72)
    sk = (torch.randn(s.H_qo, generator=g, device=DEV) * 3).float()
    out, lse = _gpu(wl, Q, sink=sk, k_rotated=True, early_inputs=True)
    torch.cuda.synchronize()
    assert pd.check_device_errors() == "PD_OK"
    ro, rl, _ = oracle.batch_decode_paged_kv_mq(
        W.bits(Q), W.bits(wl.pages), wl.indptr.cpu().numpy(), wl.values.cpu().numpy(),
        wl.length_info.cpu().numpy(), None, wl.q_rope_position.cpu().numpy(), q_len=q_len,
        q_dtype=s.q_dtype, kv_dtype=s.kv_dtype, H_kv=s.H_kv, page_size=s.page_size,
        rotary_mode=1, rope_scale=s.rope_scale, rope_theta=s.rope_theta, sm_scale=wl.sm_scale,
        sink=sk.cpu().numpy(), k_rotated=True)
    compare("bf16", out, lse, ro, rl)


def test_mq_page8_is_unsupported():
    # pages of 8 rows run on the tensor-core kernel's two-pages-per-tile form, which the
    # multi-query decode does not have
    wl, Q = _mq("llama3_8b_bf16", 66, 2, page_size=8, pool=1200)
    with pytest.raises(pd.PDError, match="UNSUPPORTED"):
        _gpu(wl, Q)
