"""Full-size workloads, in the launch configuration the benchmark times: sampled
(sequence, head) outputs are recomputed one by one by the oracle; size-independent
properties are checked on every output."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_19_gb300 import workloads as W
from tests._util import compare, gpu_decode, kind_of, oracle_decode

pd = pytest.importorskip("paged_kv_decode_19_gb300")
pytestmark = pytest.mark.gpu
DEV = "cuda"
SEED = 1000  # the benchmark's seed for rank 0


def _sample_mask(wl, n_rand=6, seed=0):
    s = wl.spec
    rng = np.random.default_rng(seed)
    mask = np.zeros((s.B, s.H_qo), bool)
    longest = int(np.argmax(wl.attended))
    shortest = int(np.argmin(wl.attended))
    mask[longest, [0, s.H_qo - 1]] = True
    mask[shortest, s.H_qo // 2] = True
    for _ in range(n_rand):
        mask[rng.integers(s.B), rng.integers(s.H_qo)] = True
    return mask


@pytest.mark.parametrize("name", list(W.SPECS))
def test_fullsize_sampled(name):
    wl = W.make(name, seed=SEED, device=DEV)
    s = wl.spec
    kw = dict(num_splits=1) if name == "tiny_fp32" else {}
    ref_pages = None
    if s.append:
        ref_pages, bad = oracle.append_paged_kv(
            W.bits(wl.pages), W.bits(wl.k_new), W.bits(wl.v_new), wl.slot_mapping.cpu().numpy(),
            in_dtype=s.q_dtype, kv_dtype=s.kv_dtype, page_size=s.page_size, k_scale=wl.k_scale,
            v_scale=wl.v_scale)
        assert bad == 0
        pd.append_paged_kv(wl.pages, wl.k_new, wl.v_new, wl.slot_mapping, wl.k_scale, wl.v_scale)
        assert pd.check_device_errors() == "PD_OK"
        assert np.array_equal(W.bits(wl.pages), ref_pages), "append not bit-exact at full size"
    if s.q_len > 1:
        _fullsize_multi_query(wl)
        return
    if s.k_rotated:  # the synthetic cache stands for K rows rotated at append time
        kw["k_rotated"] = True
    out, lse = gpu_decode(wl, **kw)
    assert pd.check_device_errors() == "PD_OK"
    # properties of every output: finite; each output element is a convex combination
    # of V values, so |out| <= max |V| (times v_scale for e4m3)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    vmax = wl.pages[:, 1].float().abs().max().item() * (wl.v_scale if s.kv_dtype == "e4m3" else 1)
    assert out.float().abs().max().item() <= vmax * (1 + 1e-2)
    assert (lse > -5e4).all()
    mask = _sample_mask(wl)
    ro, rl, st = oracle_decode(wl, pages=ref_pages, mask=mask, k_rotated=s.k_rotated)
    assert st == 0
    compare(kind_of(wl), out, lse, ro, rl, mask=mask)


@pytest.mark.parametrize("q_len", [4, 8])
def test_fullsize_multi_query_grouped_slices(q_len):
    """Speculative verification at full size with 4 or 8 query tokens (16 or 32 columns of
    a KV head): grouped slices whose warps share each K tile's rotation."""
    _fullsize_multi_query(W.make("spec_decode_bf16", seed=SEED, device=DEV, q_len=q_len))


def _fullsize_multi_query(wl):
    """Multi-query workload: the same properties, and sampled (sequence, token, head)
    outputs against the oracle's multi-query form."""
    s = wl.spec
    out = torch.empty((s.B, s.q_len, s.H_qo, s.D), dtype=W.TORCH_DTYPES[s.out_dtype], device=DEV)
    lse = torch.empty((s.B, s.q_len, s.H_qo), dtype=torch.float32, device=DEV)
    pd.batch_decode_paged_kv_mq(wl.Q, wl.pages, wl.indptr, wl.values, wl.length_info,
                                wl.k_rope_pos_offset, wl.q_rope_position, out, lse, s.rotary_mode,
                                s.rope_scale, s.rope_theta, wl.sm_scale)
    assert pd.check_device_errors() == "PD_OK"
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    vmax = wl.pages[:, 1].float().abs().max().item()
    assert out.float().abs().max().item() <= vmax * (1 + 1e-2)
    assert (lse > -5e4).all()
    m2 = _sample_mask(wl)
    mask = np.zeros((s.B, s.q_len, s.H_qo), bool)
    for t in range(s.q_len):
        mask[:, t] = np.roll(m2, t, axis=1)
    ro, rl, st = oracle.batch_decode_paged_kv_mq(
        W.bits(wl.Q), W.bits(wl.pages), wl.indptr.cpu().numpy(), wl.values.cpu().numpy(),
        wl.length_info.cpu().numpy(), wl.k_rope_pos_offset.cpu().numpy(),
        wl.q_rope_position.cpu().numpy(), q_len=s.q_len, q_dtype=s.q_dtype, kv_dtype=s.kv_dtype,
        H_kv=s.H_kv, page_size=s.page_size, rotary_mode=s.rotary_mode, rope_scale=s.rope_scale,
        rope_theta=s.rope_theta, sm_scale=wl.sm_scale, mask=mask)
    assert st == 0
    compare(kind_of(wl), out, lse, ro, rl, mask=mask)


def test_fullsize_multi_stage_long_ctx():
    """The benchmark's multi-stage form of the long-context decode at full size: sampled
    outputs against the oracle, and every output against the fused decode."""
    import bench
    wl = W.make("long_ctx_bf16", seed=SEED, device=DEV)
    s = wl.spec
    x = bench._external_split(wl, s.max_splits, DEV)
    out, lse = bench.run_external_split(pd, wl, x, s.max_splits)
    assert pd.check_device_errors() == "PD_OK"
    fo, fl = gpu_decode(wl)
    assert pd.check_device_errors() == "PD_OK"
    assert (out - fo.float()).abs().max().item() <= 2e-2
    assert (lse - fl).abs().max().item() <= 2e-3
    mask = _sample_mask(wl)
    ro, rl, st = oracle_decode(wl, mask=mask)
    assert st == 0
    compare("bf16", out, lse, ro, rl, mask=mask)
