"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each test ties one part of the oracle to a textbook/library definition, a closed
form, an invariant or a hand-derived fixture, chosen so that a plausible mistake
(dropped term, wrong sign or index, transposed operand, wrong GQA mapping, wrong
page/slot addressing, off-by-one in the window) fails at least one of them.
CPU only.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import logsumexp, softmax

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
LOG2E = 1.0 / math.log(2.0)


def _f32(a):
    return np.asarray(a, np.float32)


def _paged_case(rng, B, H_qo, H_kv, D, P, lens, pool_extra=3, dtype="f32"):
    """Random fp32 paged cache + the dense per-sequence K/V it encodes (gathered
    here with explicit Python loops, independently of the oracle)."""
    npages = [(n + P - 1) // P for n in lens]
    nnz = sum(npages)
    pool = nnz + pool_extra
    perm = rng.permutation(pool).astype(np.int32)
    values = perm[:nnz]
    indptr = np.concatenate([[0], np.cumsum(npages)]).astype(np.int32)
    last = np.array([n - (k - 1) * P if k else 0 for n, k in zip(lens, npages)], np.int32)
    pages = _f32(rng.standard_normal((pool, 2, H_kv, P, D)))
    Q = _f32(rng.standard_normal((B, H_qo, D)))
    dense = []
    for b in range(B):
        Kb = np.zeros((lens[b], H_kv, D))
        Vb = np.zeros((lens[b], H_kv, D))
        for r in range(lens[b]):
            page = values[indptr[b] + r // P]
            Kb[r] = pages[page, 0, :, r % P, :]
            Vb[r] = pages[page, 1, :, r % P, :]
        dense.append((Kb, Vb))
    return Q, pages, indptr, values, last, dense


def _run(Q, pages, indptr, values, li, H_kv, P, **kw):
    return oracle.batch_decode_paged_kv(Q, pages, indptr, values, li, None, None, q_dtype="f32",
                                        kv_dtype="f32", H_kv=H_kv, page_size=P, **kw)


# --------------------------------------------------------------------------- softmax attention

def test_dense_softmax_bruteforce():
    """Tiny cases vs scipy softmax/logsumexp on the dense K/V (textbook attention)."""
    rng = np.random.default_rng(1)
    for (B, H_qo, H_kv, D, P, lens) in [(2, 4, 2, 4, 2, [5, 3]), (2, 2, 1, 4, 4, [1, 4]),
                                         (1, 6, 3, 8, 3, [7])]:
        Q, pages, indptr, values, last, dense = _paged_case(rng, B, H_qo, H_kv, D, P, lens)
        sm = 0.37
        out, lse, st = _run(Q, pages, indptr, values, last, H_kv, P, sm_scale=sm)
        assert st == 0
        g = H_qo // H_kv
        for b in range(B):
            Kb, Vb = dense[b]
            for h in range(H_qo):
                s = sm * (Kb[:, h // g, :] @ Q[b, h].astype(np.float64))
                ref_o = softmax(s) @ Vb[:, h // g, :]
                ref_lse = logsumexp(s) * LOG2E
                np.testing.assert_allclose(out[b, h], ref_o, rtol=0, atol=1e-12)
                assert abs(lse[b, h] - ref_lse) < 1e-12


def test_lse_closed_form_fsum():
    """lse = log2(sum_r exp(sm_scale q.k_r)) with exactly-rounded sums (math.fsum)."""
    rng = np.random.default_rng(2)
    Q, pages, indptr, values, last, dense = _paged_case(rng, 1, 2, 1, 16, 4, [11])
    sm = 0.25
    out, lse, _ = _run(Q, pages, indptr, values, last, 1, 4, sm_scale=sm)
    Kb, Vb = dense[0]
    for h in range(2):
        q = [float(v) for v in Q[0, h]]
        terms = [math.exp(sm * math.fsum(q[d] * float(Kb[r, 0, d]) for d in range(16)))
                 for r in range(11)]
        assert abs(lse[0, h] - math.log2(math.fsum(terms))) < 1e-12


def test_constant_v_gives_constant_out():
    rng = np.random.default_rng(3)
    Q, pages, indptr, values, last, _ = _paged_case(rng, 2, 4, 2, 8, 4, [9, 13])
    pages[:, 1] = 0.625
    out, _, _ = _run(Q, pages, indptr, values, last, 2, 4, sm_scale=1.0)
    np.testing.assert_allclose(out, 0.625, rtol=0, atol=1e-14)


def test_length_one_returns_the_v_row():
    rng = np.random.default_rng(4)
    Q, pages, indptr, values, last, dense = _paged_case(rng, 3, 4, 2, 8, 4, [1, 1, 1])
    sm = 0.5
    out, lse, _ = _run(Q, pages, indptr, values, last, 2, 4, sm_scale=sm)
    for b in range(3):
        Kb, Vb = dense[b]
        for h in range(4):
            np.testing.assert_allclose(out[b, h], Vb[0, h // 2], rtol=0, atol=1e-15)
            s0 = sm * float(np.dot(Kb[0, h // 2], Q[b, h].astype(np.float64)))
            assert abs(lse[b, h] - s0 * LOG2E) < 1e-12


def test_empty_sequence_sentinel():
    rng = np.random.default_rng(5)
    Q, pages, indptr, values, last, _ = _paged_case(rng, 3, 2, 1, 4, 4, [5, 0, 3])
    out, lse, _ = _run(Q, pages, indptr, values, last, 1, 4)
    assert np.all(out[1] == 0.0) and np.all(lse[1] == -5e4)
    assert np.all(np.isfinite(out[[0, 2]]))


def test_page_permutation_invariance():
    """Renaming physical pages (and rewriting the table) leaves the result unchanged."""
    rng = np.random.default_rng(6)
    Q, pages, indptr, values, last, _ = _paged_case(rng, 3, 4, 2, 8, 4, [10, 17, 3], pool_extra=5)
    out0, lse0, _ = _run(Q, pages, indptr, values, last, 2, 4, sm_scale=0.3)
    pool = pages.shape[0]
    sigma = rng.permutation(pool)          # old page p lives at new id sigma[p]
    new_pages = np.empty_like(pages)
    new_pages[sigma] = pages
    out1, lse1, _ = _run(Q, new_pages, indptr, sigma[values].astype(np.int32), last, 2, 4,
                         sm_scale=0.3)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1)


def test_gqa_equals_repeated_kv_heads():
    """GQA with H_kv heads == MHA with every KV head repeated g times."""
    rng = np.random.default_rng(7)
    H_qo, H_kv, D, P = 6, 2, 8, 4
    Q, pages, indptr, values, last, _ = _paged_case(rng, 2, H_qo, H_kv, D, P, [9, 6])
    out_g, lse_g, _ = _run(Q, pages, indptr, values, last, H_kv, P, sm_scale=0.4)
    pages_mha = np.repeat(pages, H_qo // H_kv, axis=2)
    out_m, lse_m, _ = _run(Q, pages_mha, indptr, values, last, H_qo, P, sm_scale=0.4)
    assert np.array_equal(out_g, out_m) and np.array_equal(lse_g, lse_m)


# --------------------------------------------------------------------------- merge

def _split_decode(rng, lens, split_page):
    """Decode each sequence whole, and as two page-aligned parts (RoPE positions of
    the second part start at its first row)."""
    B, H_qo, H_kv, D, P = len(lens), 4, 2, 8, 4
    Q, pages, indptr, values, last, _ = _paged_case(rng, B, H_qo, H_kv, D, P, lens)
    kw = dict(rotary_mode=1, rope_theta=50.0, rope_scale=1.0, sm_scale=0.35)
    qpos = np.array(lens, np.int32)
    full = oracle.batch_decode_paged_kv(Q, pages, indptr, values, last, np.zeros(B, np.int32),
                                        qpos, q_dtype="f32", kv_dtype="f32", H_kv=H_kv,
                                        page_size=P, **kw)
    parts = []
    for lo_hi in (0, 1):
        ip, vals, li, koff = [0], [], [], []
        for b in range(B):
            npg = indptr[b + 1] - indptr[b]
            p0, p1 = (0, split_page) if lo_hi == 0 else (split_page, npg)
            vals.extend(values[indptr[b] + p0: indptr[b] + p1])
            ip.append(len(vals))
            li.append(P if lo_hi == 0 else last[b])
            koff.append(p0 * P)
        parts.append(oracle.batch_decode_paged_kv(
            Q, pages, np.array(ip, np.int32), np.array(vals, np.int32), np.array(li, np.int32),
            np.array(koff, np.int32), qpos, q_dtype="f32", kv_dtype="f32", H_kv=H_kv,
            page_size=P, **kw))
    return full, parts


def test_merge_of_split_equals_unsplit():
    rng = np.random.default_rng(8)
    (fo, fl, _), parts = _split_decode(rng, [21, 14, 9], split_page=2)
    (ao, al, _), (bo, bl, _) = parts
    mo, ml = oracle.merge_state(ao, al, bo, bl)
    np.testing.assert_allclose(mo, fo, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ml, fl, rtol=0, atol=1e-12)


def test_merge_identity_and_commutativity():
    rng = np.random.default_rng(9)
    V = rng.standard_normal((3, 4, 8))
    S = rng.standard_normal((3, 4)) * 3
    V2 = rng.standard_normal((3, 4, 8))
    S2 = rng.standard_normal((3, 4)) * 3
    Vi, Si = oracle.merge_state(V, S, np.zeros_like(V), np.full_like(S, -5e4))
    np.testing.assert_allclose(Vi, V, rtol=0, atol=1e-15)
    np.testing.assert_allclose(Si, S, rtol=0, atol=1e-13)
    a = oracle.merge_state(V, S, V2, S2)
    b = oracle.merge_state(V2, S2, V, S)
    np.testing.assert_allclose(a[0], b[0], rtol=0, atol=1e-14)
    np.testing.assert_allclose(a[1], b[1], rtol=0, atol=1e-14)


def test_merge_weights_closed_form():
    """Merged state equals the lse-weighted average: V = (2^S V + 2^So Vo)/(2^S+2^So)."""
    rng = np.random.default_rng(10)
    V, Vo = rng.standard_normal((2, 3, 5)), rng.standard_normal((2, 3, 5))
    S, So = rng.uniform(-4, 4, (2, 3)), rng.uniform(-4, 4, (2, 3))
    mv, ms = oracle.merge_state(V, S, Vo, So)
    w, wo = 2.0 ** S, 2.0 ** So
    np.testing.assert_allclose(mv, (w[..., None] * V + wo[..., None] * Vo) / (w + wo)[..., None],
                               rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(ms, np.log2(w + wo), rtol=0, atol=1e-13)


# --------------------------------------------------------------------------- window / sink

def test_window_sink_hand_enumeration():
    g = json.load(open(os.path.join(GOLDEN, "window_sink_len40.json")))
    indptr = np.array([0, 3], np.int32)
    li = np.array(g["length_info"], np.int32)
    offs = oracle.attended_offsets(indptr, li, 0, g["page_size"], True)
    assert len(offs) == g["expected_L"]
    assert offs.tolist() == g["expected_offsets"]


def test_window_sink_decode_uses_exactly_those_rows():
    """Window decode == plain decode of a cache that holds only the sink and window
    rows (same order, compacted RoPE positions)."""
    rng = np.random.default_rng(11)
    P, D, H = 16, 8, 2
    Q, pages, indptr, values, last, dense = _paged_case(rng, 1, H, 1, D, P, [40])
    li = np.array([[last[0]], [30], [4]], np.int32)
    kw = dict(rotary_mode=1, rope_theta=100.0, sm_scale=0.5)
    ow, lw, _ = oracle.batch_decode_paged_kv(Q, pages, indptr, values, li, np.zeros(1, np.int32),
                                             np.array([14], np.int32), q_dtype="f32",
                                             kv_dtype="f32", H_kv=1, page_size=P,
                                             sliding_window=True, **kw)
    rows = list(range(4)) + list(range(30, 40))
    Kb, Vb = dense[0]
    P2 = 1
    dpages = np.zeros((len(rows), 2, 1, P2, D), np.float32)
    for i, r in enumerate(rows):
        dpages[i, 0, 0, 0] = Kb[r, 0]
        dpages[i, 1, 0, 0] = Vb[r, 0]
    od, ld, _ = oracle.batch_decode_paged_kv(
        Q, dpages, np.array([0, len(rows)], np.int32), np.arange(len(rows), dtype=np.int32),
        np.array([1], np.int32), np.zeros(1, np.int32), np.array([14], np.int32), q_dtype="f32",
        kv_dtype="f32", H_kv=1, page_size=P2, **kw)
    np.testing.assert_allclose(ow, od, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lw, ld, rtol=0, atol=1e-13)


# --------------------------------------------------------------------------- RoPE

def test_rope_matches_complex_rotation():
    """Rotate-half RoPE == multiplying z_i = x_i + i x_{i+D/2} by exp(i pos s / theta^(2i/D))."""
    rng = np.random.default_rng(12)
    D = 16
    x = rng.standard_normal(D)
    for pos, sc, th in [(0, 1.0, 1e4), (1, 1.0, 100.0), (37, 0.5, 5e5), (4096, 1.0, 5e5)]:
        y = oracle.rope(x, pos, sc, th)
        i = np.arange(D // 2)
        z = (x[: D // 2] + 1j * x[D // 2:]) * np.exp(1j * pos * sc * th ** (-2.0 * i / D))
        np.testing.assert_allclose(y, np.concatenate([z.real, z.imag]), rtol=0, atol=1e-12)


def test_rope_interleaved_matches_complex_rotation():
    """Interleaved layout: z_i = x_{2i} + i x_{2i+1} times the same exp(i angle_i)."""
    rng = np.random.default_rng(22)
    D = 16
    x = rng.standard_normal(D)
    for pos, sc, th in [(0, 1.0, 1e4), (1, 1.0, 100.0), (37, 0.5, 5e5), (4096, 1.0, 5e5)]:
        y = oracle.rope(x, pos, sc, th, interleaved=True)
        i = np.arange(D // 2)
        z = (x[0::2] + 1j * x[1::2]) * np.exp(1j * pos * sc * th ** (-2.0 * i / D))
        want = np.empty(D)
        want[0::2], want[1::2] = z.real, z.imag
        np.testing.assert_allclose(y, want, rtol=0, atol=1e-12)


def test_rope_interleaved_is_rotate_half_on_permuted_dims():
    """Moving dim 2i to i and 2i+1 to i + D/2 turns the interleaved layout into the
    rotate-half one; decode with either layout on correspondingly permuted Q/K gives
    the same output once V is permuted back."""
    rng = np.random.default_rng(23)
    D = 8
    perm = np.concatenate([np.arange(0, D, 2), np.arange(1, D, 2)])  # half layout <- dims
    x = rng.standard_normal(D)
    y = oracle.rope(x, 77, 1.0, 1e3, interleaved=True)
    np.testing.assert_allclose(y[perm], oracle.rope(x[perm], 77, 1.0, 1e3), rtol=0, atol=1e-12)
    Q, pages, indptr, values, last, _ = _paged_case(rng, 2, 4, 2, D, 4, [9, 3])
    kro, qrp = np.array([2, 5], np.int32), np.array([11, 8], np.int32)
    kw = dict(q_dtype="f32", kv_dtype="f32", H_kv=2, page_size=4, rope_theta=1e3)
    o_il, l_il, _ = oracle.batch_decode_paged_kv(Q, pages, indptr, values, last, kro, qrp,
                                                 rotary_mode=2, **kw)
    o_hf, l_hf, _ = oracle.batch_decode_paged_kv(np.ascontiguousarray(Q[..., perm]),
                                                 np.ascontiguousarray(pages[..., perm]), indptr,
                                                 values, last, kro, qrp, rotary_mode=1, **kw)
    np.testing.assert_allclose(o_il[..., perm], o_hf, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l_il, l_hf, rtol=0, atol=1e-12)


def test_rope_identity_at_zero_and_norm():
    rng = np.random.default_rng(13)
    x = rng.standard_normal(8)
    assert np.array_equal(oracle.rope(x, 0, 1.0, 1e4), x)
    y = oracle.rope(x, 123, 1.0, 1e4)
    assert abs(np.linalg.norm(y) - np.linalg.norm(x)) < 1e-12


def test_rope_relativity():
    """q(p).k(p') depends only on p - p'."""
    rng = np.random.default_rng(14)
    q, k = rng.standard_normal(16), rng.standard_normal(16)
    ref = np.dot(oracle.rope(q, 10, 1.0, 1e4), oracle.rope(k, 3, 1.0, 1e4))
    for shift in (1, 50, 1000):
        got = np.dot(oracle.rope(q, 10 + shift, 1.0, 1e4), oracle.rope(k, 3 + shift, 1.0, 1e4))
        assert abs(got - ref) < 1e-11


def test_decode_rope_positions():
    """K row r is rotated at k_rope_pos_offset + r and Q at q_rope_position: shifting
    both by the same amount leaves the output unchanged (relativity through the
    whole decode)."""
    rng = np.random.default_rng(15)
    Q, pages, indptr, values, last, _ = _paged_case(rng, 2, 4, 2, 8, 4, [11, 6])
    kw = dict(q_dtype="f32", kv_dtype="f32", H_kv=2, page_size=4, rotary_mode=1,
              rope_theta=30.0, sm_scale=0.4)
    a = oracle.batch_decode_paged_kv(Q, pages, indptr, values, last, np.array([0, 0], np.int32),
                                     np.array([11, 6], np.int32), **kw)
    b = oracle.batch_decode_paged_kv(Q, pages, indptr, values, last, np.array([5, 9], np.int32),
                                     np.array([16, 15], np.int32), **kw)
    np.testing.assert_allclose(a[0], b[0], rtol=0, atol=1e-11)
    np.testing.assert_allclose(a[1], b[1], rtol=0, atol=1e-11)
    c = oracle.batch_decode_paged_kv(Q, pages, indptr, values, last, np.array([0, 0], np.int32),
                                     np.array([12, 6], np.int32), **kw)
    assert not np.allclose(a[0][0], c[0][0])


# --------------------------------------------------------------------------- number formats

def test_e4m3_golden_codes():
    g = json.load(open(os.path.join(GOLDEN, "e4m3_codes.json")))
    for code, val in g["codes"].items():
        v = oracle.decode(np.array([int(code, 16)], np.uint8), "e4m3")[0]
        assert v == val and math.copysign(1, v) == math.copysign(1, val), code
    for code in g["nan_codes"]:
        assert np.isnan(oracle.decode(np.array([int(code, 16)], np.uint8), "e4m3")[0])
    for case in g["encode_cases"]:
        assert oracle.encode(np.array([case["x"]]), "e4m3")[0] == int(case["code"], 16), case


def test_e4m3_decode_all_codes_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.decode(codes, "e4m3")
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])


def test_e4m3_roundtrip_and_ties():
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.decode(codes, "e4m3")
    finite = ~np.isnan(vals)
    back = oracle.encode(vals[finite], "e4m3")
    assert np.array_equal(back, codes[finite])
    pos = np.sort(np.unique(vals[finite & (vals > 0)]))
    mids = (pos[:-1] + pos[1:]) / 2
    enc = oracle.encode(mids, "e4m3")
    lo = oracle.encode(pos[:-1], "e4m3")
    hi = oracle.encode(pos[1:], "e4m3")
    want = np.where(lo % 2 == 0, lo, hi)  # ties to the even mantissa
    assert np.array_equal(enc, want)


def test_e4m3_encode_vs_torch_in_range():
    rng = np.random.default_rng(16)
    x = np.concatenate([rng.standard_normal(20000) * 50, rng.uniform(-448, 448, 20000),
                        rng.standard_normal(5000) * 1e-3]).astype(np.float32)
    mine = oracle.encode(x.astype(np.float64), "e4m3")
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(mine, ref)


@pytest.mark.parametrize("dt,tdt", [("bf16", torch.bfloat16), ("f16", torch.float16)])
def test_16bit_formats_vs_torch(dt, tdt):
    rng = np.random.default_rng(17)
    x = np.concatenate([rng.standard_normal(50000), rng.standard_normal(2000) * 1e-6,
                        rng.standard_normal(2000) * 1e4]).astype(np.float32)
    mine = oracle.encode(x.astype(np.float64), dt)
    ref = torch.from_numpy(x).to(tdt).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine, ref)
    dec = oracle.decode(ref, dt)
    assert np.array_equal(dec, torch.from_numpy(x).to(tdt).double().numpy())


# --------------------------------------------------------------------------- append

def test_append_matches_index_put_scatter():
    """Oracle append == torch index_put_ scatter ([VLLM] reshape_and_cache semantics)
    on the [max_pages,2,H_kv,P,D] layout; negative slots skipped; exact copy."""
    rng = np.random.default_rng(18)
    T, H_kv, D, P, pool = 7, 3, 8, 4, 6
    pages = rng.standard_normal((pool, 2, H_kv, P, D)).astype(np.float32)
    k = rng.standard_normal((T, H_kv, D)).astype(np.float32)
    v = rng.standard_normal((T, H_kv, D)).astype(np.float32)
    slots = np.array([0, 5, -1, 23, 9, -7, 14], np.int64)
    got, bad = oracle.append_paged_kv(pages, k, v, slots, in_dtype="f32", kv_dtype="f32",
                                      page_size=P)
    assert bad == 0
    ref = torch.from_numpy(pages.copy())
    keep = slots >= 0
    s = torch.from_numpy(slots[keep])
    blk, off = torch.div(s, P, rounding_mode="floor"), s % P
    hh = torch.arange(H_kv)
    ref[blk[:, None], 0, hh[None, :], off[:, None]] = torch.from_numpy(k[keep])
    ref[blk[:, None], 1, hh[None, :], off[:, None]] = torch.from_numpy(v[keep])
    assert np.array_equal(got.view(np.float32), ref.numpy())


def test_append_fp8_quantisation_vs_torch():
    """bf16 input -> e4m3 cache: code = e4m3_rne(fl32(x) / scale), checked against
    torch's fp32 division + e4m3fn cast (RNE) for in-range values."""
    rng = np.random.default_rng(19)
    T, H_kv, D, P, pool = 5, 2, 16, 4, 3
    pages = np.zeros((pool, 2, H_kv, P, D), np.uint8)
    kt = torch.from_numpy(rng.standard_normal((T, H_kv, D)).astype(np.float32)).bfloat16()
    vt = torch.from_numpy(rng.standard_normal((T, H_kv, D)).astype(np.float32)).bfloat16()
    ks, vs = np.float32(4.1 / 448), np.float32(3.7 / 448)
    slots = np.array([0, 3, 4, 11, -1], np.int64)
    kb = kt.view(torch.int16).numpy().view(np.uint16)
    vb = vt.view(torch.int16).numpy().view(np.uint16)
    got, bad = oracle.append_paged_kv(pages, kb, vb, slots, in_dtype="bf16", kv_dtype="e4m3",
                                      page_size=P, k_scale=ks, v_scale=vs)
    assert bad == 0
    for t in range(T):
        if slots[t] < 0:
            continue
        page, off = slots[t] // P, slots[t] % P
        for kv, src, sc in ((0, kt, ks), (1, vt, vs)):
            q = (src[t].float() / torch.tensor(sc)).clamp(-448, 448)
            ref = q.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(got[page, kv, :, off, :], ref)


def test_append_out_of_range_slot_counted():
    pages = np.zeros((2, 2, 1, 4, 4), np.float32)
    k = np.ones((2, 1, 4), np.float32)
    got, bad = oracle.append_paged_kv(pages, k, k, np.array([8, 3], np.int64), in_dtype="f32",
                                      kv_dtype="f32", page_size=4)
    assert bad == 1 and got.view(np.float32)[0, 0, 0, 3].tolist() == [1.0] * 4


# --------------------------------------------------------------------------- multi-query decode

def _run_mq(Q, pages, indptr, values, li, H_kv, P, q_len, **kw):
    return oracle.batch_decode_paged_kv_mq(Q, pages, indptr, values, li, kw.pop("kro", None),
                                           kw.pop("qrp", None), q_len=q_len, q_dtype="f32",
                                           kv_dtype="f32", H_kv=H_kv, page_size=P, **kw)


def test_mq_dense_causal_bruteforce():
    """q_len query tokens per sequence vs scipy softmax on the dense K/V with the causal
    limit written out: token t sees rows 0 .. L - q_len + t (none when that is < 0)."""
    rng = np.random.default_rng(11)
    for (H_qo, H_kv, D, P, lens, q_len) in [(4, 2, 4, 2, [5, 3, 7], 3), (2, 1, 4, 4, [2, 6], 3),
                                            (3, 3, 8, 3, [4], 4)]:
        B = len(lens)
        _, pages, indptr, values, last, dense = _paged_case(rng, B, H_qo, H_kv, D, P, lens)
        Q = _f32(rng.standard_normal((B, q_len, H_qo, D)))
        sm = 0.41
        out, lse, st = _run_mq(Q, pages, indptr, values, last, H_kv, P, q_len, sm_scale=sm)
        assert st == 0 and out.shape == (B, q_len, H_qo, D)
        g = H_qo // H_kv
        for b in range(B):
            Kb, Vb = dense[b]
            for t in range(q_len):
                n = lens[b] - q_len + 1 + t  # rows 0 .. n-1
                for h in range(H_qo):
                    if n <= 0:
                        assert np.all(out[b, t, h] == 0) and lse[b, t, h] == -5e4
                        continue
                    s = sm * (Kb[:n, h // g, :] @ Q[b, t, h].astype(np.float64))
                    np.testing.assert_allclose(out[b, t, h], softmax(s) @ Vb[:n, h // g, :],
                                               rtol=0, atol=1e-12)
                    assert abs(lse[b, t, h] - logsumexp(s) * LOG2E) < 1e-12


def test_mq_single_token_is_decode():
    rng = np.random.default_rng(12)
    Q, pages, indptr, values, last, _ = _paged_case(rng, 3, 4, 2, 8, 4, [9, 1, 6])
    o1, l1, _ = _run(Q, pages, indptr, values, last, 2, 4, sm_scale=0.3)
    o2, l2, _ = _run_mq(Q, pages, indptr, values, last, 2, 4, 1, sm_scale=0.3)
    assert np.array_equal(o1, o2[:, 0]) and np.array_equal(l1, l2[:, 0])


def test_mq_token_equals_truncated_decode_with_rope():
    """Token t = a single-token decode of the sequence cut to its first L - q_len + 1 + t
    rows (last_page_len adjusted) with the query at q_rope_position + t."""
    rng = np.random.default_rng(13)
    P, q_len, H_qo, H_kv, D = 4, 3, 4, 2, 8
    lens = [10, 5]
    B = len(lens)
    _, pages, indptr, values, last, _ = _paged_case(rng, B, H_qo, H_kv, D, P, lens)
    Q = _f32(rng.standard_normal((B, q_len, H_qo, D)))
    kro = np.array([3, 0], np.int32)
    qrp = np.array([20, 7], np.int32)
    kw = dict(rotary_mode=1, rope_theta=100.0, sm_scale=0.35)
    out, lse, st = _run_mq(Q, pages, indptr, values, last, H_kv, P, q_len, kro=kro, qrp=qrp, **kw)
    assert st == 0
    for b in range(B):
        for t in range(q_len):
            n = lens[b] - q_len + 1 + t
            npg = (n + P - 1) // P
            ip = np.array([0, npg], np.int32)
            vals = values[indptr[b]:indptr[b] + npg]
            li = np.array([n - (npg - 1) * P], np.int32)
            o1, l1, _ = oracle.batch_decode_paged_kv(
                Q[b:b + 1, t], pages, ip, vals, li, kro[b:b + 1], qrp[b:b + 1] + t, q_dtype="f32",
                kv_dtype="f32", H_kv=H_kv, page_size=P, **kw)
            np.testing.assert_allclose(out[b, t], o1[0], rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[b, t], l1[0], rtol=0, atol=1e-12)


def test_mq_rejects_bad_q_len():
    rng = np.random.default_rng(14)
    Q, pages, indptr, values, last, _ = _paged_case(rng, 1, 2, 1, 4, 4, [5])
    with pytest.raises(ValueError):
        oracle.batch_decode_paged_kv_mq(Q, pages, indptr, values, last, None, None, q_len=0,
                                        q_dtype="f32", kv_dtype="f32", H_kv=1, page_size=4)


# --------------------------------------------------------------------------- learned sinks

def test_sink_bruteforce_and_virtual_row():
    """A per-head sink logit joins the softmax with a zero value row: brute force with
    scipy on the dense K/V plus one extra score, for decode and multi-query decode."""
    rng = np.random.default_rng(31)
    H_qo, H_kv, D, P, lens = 4, 2, 8, 4, [7, 0, 2]
    B = len(lens)
    Q, pages, indptr, values, last, dense = _paged_case(rng, B, H_qo, H_kv, D, P, lens)
    sink = rng.standard_normal(H_qo) * 2
    sm = 0.3
    out, lse, st = _run(Q, pages, indptr, values, last, H_kv, P, sm_scale=sm, sink=sink)
    assert st == 0
    g = H_qo // H_kv
    for b in range(B):
        Kb, Vb = dense[b]
        for h in range(H_qo):
            s = np.concatenate([sm * (Kb[:, h // g, :] @ Q[b, h].astype(np.float64)), [sink[h]]])
            Vx = np.concatenate([Vb[:, h // g, :], np.zeros((1, D))])
            np.testing.assert_allclose(out[b, h], softmax(s) @ Vx, rtol=0, atol=1e-12)
            assert abs(lse[b, h] - logsumexp(s) * LOG2E) < 1e-12
    # an empty sequence keeps only the sink: out 0, lse = sink in log2 units
    assert np.all(out[1] == 0) and np.allclose(lse[1], sink * LOG2E, rtol=0, atol=1e-12)
    Qm = _f32(rng.standard_normal((B, 2, H_qo, D)))
    o2, l2, _ = _run_mq(Qm, pages, indptr, values, last, H_kv, P, 2, sm_scale=sm, sink=sink)
    for b in range(B):
        Kb, Vb = dense[b]
        for t in range(2):
            n = max(lens[b] - 2 + 1 + t, 0)
            for h in range(H_qo):
                s = np.concatenate([sm * (Kb[:n, h // g, :] @ Qm[b, t, h].astype(np.float64)),
                                    [sink[h]]])
                Vx = np.concatenate([Vb[:n, h // g, :], np.zeros((1, D))])
                np.testing.assert_allclose(o2[b, t, h], softmax(s) @ Vx, rtol=0, atol=1e-12)
                assert abs(l2[b, t, h] - logsumexp(s) * LOG2E) < 1e-12


def test_sink_is_one_merge_with_a_zero_state():
    """Adding the sink equals merge_state of the sink-free result with the state
    (V = 0, S = sink log2 e): the sink enters once, wherever the split falls."""
    rng = np.random.default_rng(32)
    Q, pages, indptr, values, last, _ = _paged_case(rng, 2, 4, 2, 8, 4, [9, 5])
    sink = rng.standard_normal(4)
    o0, l0, _ = _run(Q, pages, indptr, values, last, 2, 4)
    o1, l1, _ = _run(Q, pages, indptr, values, last, 2, 4, sink=sink)
    Vm, Sm = oracle.merge_state(o0, l0, np.zeros_like(o0), np.broadcast_to(sink * LOG2E, l0.shape))
    np.testing.assert_allclose(o1, Vm, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, Sm, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- K rotated at append time

@pytest.mark.parametrize("mode", [1, 2])
def test_append_rope_rows_equal_rotated_then_encoded(mode):
    """Each appended K row is the pinned RoPE of the input row at its position, then the
    pinned encoder; V rows are the plain append's."""
    rng = np.random.default_rng(40 + mode)
    T, H, D, P, pool = 5, 2, 8, 4, 6
    pages = oracle.encode(rng.standard_normal((pool, 2, H, P, D)), "bf16")
    k = oracle.encode(rng.standard_normal((T, H, D)), "bf16")
    v = oracle.encode(rng.standard_normal((T, H, D)), "bf16")
    slots = np.array([3, 9, -1, 17, 22], np.int64)
    pos = np.array([5, 100, 7, 4096, 0], np.int32)
    got, bad = oracle.append_paged_kv_rope(pages, k, v, slots, pos, in_dtype="bf16",
                                           kv_dtype="bf16", page_size=P, rotary_mode=mode,
                                           rope_theta=1e3)
    plain, _ = oracle.append_paged_kv(pages, k, v, slots, in_dtype="bf16", kv_dtype="bf16",
                                      page_size=P)
    assert bad == 0
    np.testing.assert_array_equal(got[:, 1], plain[:, 1])  # V untouched by RoPE
    kd = oracle.decode(k, "bf16")
    for t in range(T):
        if slots[t] < 0:
            continue
        page, off = divmod(int(slots[t]), P)
        for h in range(H):
            want = oracle.encode(oracle.rope(kd[t, h], pos[t], 1.0, 1e3, interleaved=mode == 2), "bf16")
            np.testing.assert_array_equal(got[page, 0, h, off], want)


def test_k_rotated_decode_equals_rope_decode_on_exact_values():
    """A cache whose K rows were rotated beforehand (fp64, stored as f32), decoded with
    k_rotated, equals the rotating decode of the original cache up to that f32 storage."""
    rng = np.random.default_rng(44)
    Q, pages, indptr, values, last, dense = _paged_case(rng, 2, 4, 2, 8, 4, [9, 6])
    kro = np.array([3, 0], np.int32)
    qrp = np.array([12, 6], np.int32)
    kw = dict(q_dtype="f32", kv_dtype="f32", H_kv=2, page_size=4, rotary_mode=1, rope_theta=1e3)
    o_ref, l_ref, _ = oracle.batch_decode_paged_kv(Q, pages, indptr, values, last, kro, qrp, **kw)
    rot = pages.copy()
    for b in range(2):
        for r in range(int(indptr[b + 1] - indptr[b]) * 4):
            if r >= [9, 6][b]:
                break
            page = values[indptr[b] + r // 4]
            for h in range(2):
                rot[page, 0, h, r % 4] = oracle.rope(pages[page, 0, h, r % 4], kro[b] + r, 1.0, 1e3)
    o_kr, l_kr, _ = oracle.batch_decode_paged_kv(Q, _f32(rot), indptr, values, last, kro, qrp,
                                                 k_rotated=True, **kw)
    np.testing.assert_allclose(o_kr, o_ref, rtol=0, atol=1e-5)
    np.testing.assert_allclose(l_kr, l_ref, rtol=0, atol=1e-5)


# --------------------------------------------------------------------------- merge of R states

def _chunk_decodes(rng, lens, R, P=4, rope=True):
    """Each sequence decoded whole, and as R page-aligned chunks (chunk r: pages
    [r per, (r+1) per), per = ceil(npages / R); a chunk past the end of the page list is
    empty), each chunk a pseudo-sequence whose RoPE positions start at its first row."""
    B, H_qo, H_kv, D = len(lens), 4, 2, 8
    Q, pages, indptr, values, last, _ = _paged_case(rng, B, H_qo, H_kv, D, P, lens)
    kw = dict(rotary_mode=1 if rope else 0, rope_theta=50.0, rope_scale=1.0, sm_scale=0.35,
              q_dtype="f32", kv_dtype="f32", H_kv=H_kv, page_size=P)
    qpos = np.array(lens, np.int32)
    full = oracle.batch_decode_paged_kv(Q, pages, indptr, values, last, np.zeros(B, np.int32),
                                        qpos, **kw)
    Vp, Sp = [], []
    for r in range(R):
        ip, vals, li, koff = [0], [], [], []
        for b in range(B):
            npg = int(indptr[b + 1] - indptr[b])
            per = -(-npg // R) if npg else 1
            p0, p1 = min(npg, r * per), min(npg, (r + 1) * per)
            vals.extend(values[indptr[b] + p0: indptr[b] + p1])
            ip.append(len(vals))
            rows = min(lens[b], p1 * P) - p0 * P if p1 > p0 else 0
            li.append(rows - (p1 - p0 - 1) * P if p1 > p0 else 0)
            koff.append(p0 * P)
        o, l, st = oracle.batch_decode_paged_kv(
            Q, pages, np.array(ip, np.int32), np.array(vals if vals else [0], np.int32),
            np.array(li, np.int32), np.array(koff, np.int32), qpos, **kw)
        assert st == 0
        Vp.append(o)
        Sp.append(l)
    return full, np.stack(Vp), np.stack(Sp)


@pytest.mark.parametrize("R", [2, 3, 8])
def test_merge_states_of_chunks_equals_unsplit(R):
    # sequences shorter than R pages leave some chunks empty (their state is the
    # empty sentinel, which must add nothing); an empty sequence stays empty
    rng = np.random.default_rng(40 + R)
    lens = [21, 14, 9, 3, 0, 33]
    (fo, fl, _), Vp, Sp = _chunk_decodes(rng, lens, R)
    assert (Sp == -5e4).any()
    mo, ml = oracle.merge_states(Vp, Sp)
    np.testing.assert_allclose(mo, fo, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ml, fl, rtol=0, atol=1e-12)
    assert np.all(mo[4] == 0) and np.all(ml[4] == -5e4)


def test_merge_states_is_the_pairwise_fold_and_order_free():
    rng = np.random.default_rng(50)
    R, N, H, D = 5, 3, 4, 6
    Vp = rng.standard_normal((R, N, H, D))
    Sp = rng.uniform(-6, 6, (R, N, H))
    mo, ml = oracle.merge_states(Vp, Sp)
    fo, fl = Vp[0], Sp[0]
    for r in range(1, R):
        fo, fl = oracle.merge_state(fo, fl, Vp[r], Sp[r])
    np.testing.assert_allclose(mo, fo, rtol=0, atol=1e-13)
    np.testing.assert_allclose(ml, fl, rtol=0, atol=1e-13)
    perm = rng.permutation(R)
    po, pl = oracle.merge_states(Vp[perm], Sp[perm])
    np.testing.assert_allclose(po, mo, rtol=0, atol=1e-14)
    np.testing.assert_allclose(pl, ml, rtol=0, atol=1e-13)
    # closed form of one row
    w = 2.0 ** Sp[:, 1, 2]
    np.testing.assert_allclose(mo[1, 2], (w[:, None] * Vp[:, 1, 2]).sum(0) / w.sum(), rtol=1e-13, atol=1e-14)


def test_merge_states_empty_partners():
    rng = np.random.default_rng(51)
    Vp = rng.standard_normal((3, 2, 2, 4))
    Sp = rng.uniform(-3, 3, (3, 2, 2))
    Vp[1], Sp[1] = 0.0, -5e4                 # an empty partner adds nothing
    mo, ml = oracle.merge_states(Vp, Sp)
    ro, rl = oracle.merge_states(Vp[[0, 2]], Sp[[0, 2]])
    np.testing.assert_allclose(mo, ro, rtol=0, atol=1e-15)
    np.testing.assert_allclose(ml, rl, rtol=0, atol=1e-13)
    Sp[:, 0, 1] = -5e4                       # every partner empty: the empty state
    Vp[:, 0, 1] = 0.0
    mo, ml = oracle.merge_states(Vp, Sp)
    assert np.all(mo[0, 1] == 0) and ml[0, 1] == -5e4
