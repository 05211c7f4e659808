"""K rotated at append time: pd_append_paged_kv_rope against the oracle's rotating append,
and decodes with PD_DECODE_K_ROTATED (Q rotated only) against the oracle's decode of the
oracle-rotated cache."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_19_gb300 import workloads as W
from tests._util import compare

pd = pytest.importorskip("paged_kv_decode_19_gb300")
pytestmark = pytest.mark.gpu
DEV = "cuda"


def _ulps(a_bits, b_bits, dt):
    """Distance in units in the last place between two arrays of typed bits."""
    if dt == "e4m3":
        a, b = a_bits.astype(np.int32), b_bits.astype(np.int32)
        sa = np.where(a & 0x80, -(a & 0x7F), a & 0x7F)
        sb = np.where(b & 0x80, -(b & 0x7F), b & 0x7F)
        return np.abs(sa - sb)
    w = np.int64 if dt == "f32" else np.int32
    a, b = a_bits.astype(w), b_bits.astype(w)
    m = (1 << 31) if dt == "f32" else (1 << 15)
    sa = np.where(a & m, -(a & (m - 1)), a)
    sb = np.where(b & m, -(b & (m - 1)), b)
    return np.abs(sa - sb)


@pytest.mark.parametrize("kv,in_dt", [("bf16", "bf16"), ("f16", "f16"), ("e4m3", "bf16"),
                                      ("f32", "f32")])
@pytest.mark.parametrize("mode", [1, 2])
def test_append_rope_matches_oracle(kv, in_dt, mode):
    g = torch.Generator(device=DEV)
    g.manual_seed(100 + mode)
    T, H, D, P, pool = 40, 4, 128, 16, 16
    x = torch.randn((pool, 2, H, P, D), generator=g, device=DEV)
    k_scale = v_scale = 0.05 if kv == "e4m3" else 1.0
    pages = (x / k_scale).to(torch.float8_e4m3fn) if kv == "e4m3" else x.to(W.TORCH_DTYPES[kv])
    k_new = torch.randn((T, H, D), generator=g, device=DEV).to(W.TORCH_DTYPES[in_dt])
    v_new = torch.randn((T, H, D), generator=g, device=DEV).to(W.TORCH_DTYPES[in_dt])
    slots = torch.randperm(pool * P, generator=g, device=DEV)[:T].to(torch.int64)
    slots[3] = -1
    pos = torch.randint(0, 200000, (T,), generator=g, device=DEV, dtype=torch.int32)
    ref, bad = oracle.append_paged_kv_rope(
        W.bits(pages), W.bits(k_new), W.bits(v_new), slots.cpu().numpy(), pos.cpu().numpy(),
        in_dtype=in_dt, kv_dtype=kv, page_size=P, rotary_mode=mode, rope_theta=5e5,
        k_scale=k_scale, v_scale=v_scale)
    assert bad == 0
    pd.append_paged_kv_rope(pages, k_new, v_new, slots, pos, mode, 1.0, 5e5, k_scale, v_scale)
    torch.cuda.synchronize()
    assert pd.check_device_errors() == "PD_OK"
    got = W.bits(pages)
    np.testing.assert_array_equal(got[:, 1], ref[:, 1])  # V: the plain append
    # K: the rotation runs in fp32 here, in fp64 in the oracle
    if kv == "f32":  # stored in fp32: the fp32 rotation's own error, a few 2^-24 of |x|+|y|
        err = np.abs(oracle.decode(got[:, 0], kv) - oracle.decode(ref[:, 0], kv))
        assert err.max() <= 3e-6, err.max()
    else:  # one unit at most, where the exact value sits next to a rounding boundary
        d = _ulps(got[:, 0], ref[:, 0], kv)
        assert d.max() <= 1 and (d > 0).mean() < 1e-3, (d.max(), (d > 0).mean())


def _rotate_cache(wl, mode):
    """Rewrite every attended K row of the workload's cache rotated at its position
    k_rope_pos_offset + r, through pd_append_paged_kv_rope (GPU) and the oracle."""
    s = wl.spec
    P = s.page_size
    ip = wl.indptr.cpu().numpy()
    vals = wl.values.cpu().numpy()
    kro = wl.k_rope_pos_offset.cpu().numpy()
    li = wl.length_info.cpu().numpy()
    slots, pos = [], []
    for b in range(s.B):
        for r in range(int(wl.attended[b])):
            so = r  # sequence offset of attended row r (window: sink rows, then the window)
            if s.window is not None and r >= li[2][b]:
                so = r - int(li[2][b]) + int(li[1][b])
            slots.append(int(vals[ip[b] + so // P]) * P + so % P)
            pos.append(int(kro[b]) + r)
    slots_t = torch.tensor(slots, dtype=torch.int64, device=DEV)
    pos_t = torch.tensor(pos, dtype=torch.int32, device=DEV)
    page_i, off_i = slots_t // P, slots_t % P
    flat = wl.pages.view(wl.pages.shape[0], 2, s.H_kv, P, s.D)
    k_rows = flat[page_i, 0, :, off_i].contiguous()  # [T, H_kv, D] of the cache dtype
    v_rows = flat[page_i, 1, :, off_i].contiguous()
    if s.kv_dtype == "e4m3":  # the append takes 16-bit input: dequantise exactly
        k_rows = (k_rows.float() * wl.k_scale).to(torch.float32)
        v_rows = (v_rows.float() * wl.v_scale).to(torch.float32)
    in_dt = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}[k_rows.dtype]
    ref, bad = oracle.append_paged_kv_rope(
        W.bits(wl.pages), W.bits(k_rows), W.bits(v_rows), np.array(slots, np.int64),
        np.array(pos, np.int32), in_dtype=in_dt, kv_dtype=s.kv_dtype, page_size=P,
        rotary_mode=mode, rope_scale=s.rope_scale, rope_theta=s.rope_theta,
        k_scale=wl.k_scale, v_scale=wl.v_scale)
    assert bad == 0
    pd.append_paged_kv_rope(wl.pages, k_rows, v_rows, slots_t, pos_t, mode, s.rope_scale,
                            s.rope_theta, wl.k_scale, wl.v_scale)
    torch.cuda.synchronize()
    return ref


@pytest.mark.parametrize("name,over", [("llama3_8b_bf16", {}), ("window_sink_f16", {}),
                                       ("fp8_kv_highconc", dict(rotary_mode=1, rope_theta=1e4)),
                                       ("tiny_fp32", dict(rotary_mode=1, rope_theta=1e4))])
@pytest.mark.parametrize("mode", [1, 2])
def test_k_rotated_decode(name, over, mode):
    wl = W.make(name, seed=120 + mode, reduced=True, **dict(over, rotary_mode=mode)).to(DEV)
    s = wl.spec
    ref_pages = _rotate_cache(wl, mode)
    kw = dict(num_splits=1) if name == "tiny_fp32" else {}
    out = torch.empty((s.B, s.H_qo, s.D), dtype=W.TORCH_DTYPES[s.out_dtype], device=DEV)
    lse = torch.empty((s.B, s.H_qo), dtype=torch.float32, device=DEV)
    pd.batch_decode_paged_kv(wl.Q, wl.pages, wl.indptr, wl.values, wl.length_info, None,
                             wl.q_rope_position, out, lse, s.rotary_mode, s.rope_scale,
                             s.rope_theta, wl.sm_scale, k_scale=wl.k_scale, v_scale=wl.v_scale,
                             k_rotated=True, **kw)
    assert pd.check_device_errors() == "PD_OK"
    ro, rl, st = oracle.batch_decode_paged_kv(
        W.bits(wl.Q), ref_pages, wl.indptr.cpu().numpy(), wl.values.cpu().numpy(),
        wl.length_info.cpu().numpy(), None, wl.q_rope_position.cpu().numpy(), q_dtype=s.q_dtype,
        kv_dtype=s.kv_dtype, H_kv=s.H_kv, page_size=s.page_size, rotary_mode=mode,
        rope_scale=s.rope_scale, rope_theta=s.rope_theta, sm_scale=wl.sm_scale,
        sliding_window=s.window is not None, k_scale=wl.k_scale, v_scale=wl.v_scale,
        k_rotated=True)
    assert st == 0
    kind = s.kv_dtype
    if kind == "f32":  # the cache rows themselves may differ by an fp32 ulp
        np.testing.assert_allclose(out.double().cpu().numpy(), ro, rtol=0, atol=1e-5)
        np.testing.assert_allclose(lse.double().cpu().numpy(), rl, rtol=0, atol=1e-5)
    else:
        compare(kind, out, lse, ro, rl)


def test_k_rotated_multi_query():
    q_len = 2
    wl = W.make("llama3_8b_bf16", seed=130, reduced=True).to(DEV)
    s = wl.spec
    ref_pages = _rotate_cache(wl, 1)
    g = torch.Generator(device=DEV)
    g.manual_seed(131)
    Q = torch.randn((s.B, q_len, s.H_qo, s.D), generator=g, device=DEV).to(torch.bfloat16)
    qpos = torch.from_numpy(np.maximum(wl.attended - q_len, 0).astype(np.int32)).to(DEV)
    out = torch.empty((s.B, q_len, s.H_qo, s.D), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((s.B, q_len, s.H_qo), dtype=torch.float32, device=DEV)
    pd.batch_decode_paged_kv_mq(Q, wl.pages, wl.indptr, wl.values, wl.length_info, None, qpos,
                                out, lse, 1, s.rope_scale, s.rope_theta, wl.sm_scale,
                                k_rotated=True, num_splits=3,
                                max_kv_len_hint=int(wl.attended.max()))
    ro, rl, _ = oracle.batch_decode_paged_kv_mq(
        W.bits(Q), ref_pages, wl.indptr.cpu().numpy(), wl.values.cpu().numpy(),
        wl.length_info.cpu().numpy(), None, qpos.cpu().numpy(), q_len=q_len, q_dtype="bf16",
        kv_dtype="bf16", H_kv=s.H_kv, page_size=s.page_size, rotary_mode=1,
        rope_scale=s.rope_scale, rope_theta=s.rope_theta, sm_scale=wl.sm_scale, k_rotated=True)
    compare("bf16", out, lse, ro, rl)
