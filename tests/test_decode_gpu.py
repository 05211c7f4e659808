"""GPU parity of batch_decode_paged_kv against the fp64 oracle (called through the
C ABI).  Reduced workloads are compared element by element; edge cases and the
error path follow."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_19_gb300 import workloads as W
from tests._util import compare, gpu_decode, kind_of, oracle_decode

pd = pytest.importorskip("paged_kv_decode_19_gb300")
pytestmark = pytest.mark.gpu

DEV = "cuda"


def _wl(name, seed, **kw):
    return W.make(name, seed=seed, reduced=True, **kw).to(DEV)


def _check(wl, expect_variant=None, **kw):
    out, lse = gpu_decode(wl, **kw)
    assert pd.check_device_errors() == "PD_OK"
    if expect_variant:
        assert pd.last_decode_variant() == expect_variant
    ro, rl, st = oracle_decode(wl)
    assert st == 0
    return compare(kind_of(wl), out, lse, ro, rl)


@pytest.mark.parametrize("seed", [0, 1])
@pytest.mark.parametrize("splits", [1, 0])
def test_tiny_fp32(seed, splits):
    wl = W.make("tiny_fp32", seed=seed).to(DEV)
    _check(wl, "simt", num_splits=splits)


@pytest.mark.parametrize("seed", [0, 3])
def test_llama3_bf16_rope_mma(seed):
    _check(_wl("llama3_8b_bf16", seed), "mma")


def test_llama3_bf16_rope_page8_and_page4():
    """Page size 8 runs on the tensor-core kernel with two pages per 16-row tile; page
    size 4 is outside it and the SIMT kernel serves it."""
    _check(_wl("llama3_8b_bf16", 4, page_size=8, pool=1200), "mma")
    _check(_wl("llama3_8b_bf16", 4, page_size=8, pool=1200), "mma", num_splits=5,
           max_kv_len_hint=700)
    _check(_wl("llama3_8b_bf16", 5, page_size=4, pool=2400), "simt")


@pytest.mark.parametrize("seed", [0, 1])
def test_long_context_internal_split(seed):
    wl = _wl("long_ctx_bf16", seed)
    _check(wl, "mma")
    # force many chunks per sequence
    _check(wl, "mma", num_splits=32, max_kv_len_hint=int(wl.attended.max()))


def test_long_context_external_split_merge_tree():
    """Config-3 flow: decode each page-aligned chunk as a pseudo-sequence (fp32
    partials), then merge pairwise with merge_state_inplace in a tree."""
    wl = _wl("long_ctx_bf16", 2)
    s = wl.spec
    ipc, valc, lastc, koff, owner = W.split_chunks(wl.indptr.cpu().numpy(), wl.values.cpu().numpy(),
                                                   wl.seq_len, s.page_size, 32)
    nchunk = np.bincount(owner, minlength=s.B)
    assert 16 <= nchunk.max() <= 32
    Bc = len(owner)
    Qc = wl.Q[torch.from_numpy(owner).to(DEV)].contiguous()
    out = torch.empty((Bc, s.H_qo, s.D), dtype=torch.float32, device=DEV)
    lse = torch.empty((Bc, s.H_qo), dtype=torch.float32, device=DEV)
    t = lambda a: torch.from_numpy(a).to(DEV)
    pd.batch_decode_paged_kv(Qc, wl.pages, t(ipc), t(valc), t(lastc), t(koff), t(koff), out, lse,
                             0, 1.0, 1e4, wl.sm_scale, num_splits=1)
    # tree: level by level, merge chunk 2i+1 into chunk 2i of each sequence
    idx = [list(np.nonzero(owner == b)[0]) for b in range(s.B)]
    while max(len(x) for x in idx) > 1:
        dst, src = [], []
        for b in range(s.B):
            x = idx[b]
            dst += x[0:len(x) - 1:2]
            src += x[1:len(x):2]
            idx[b] = x[0::2]
        di, si = t(np.array(dst)), t(np.array(src))
        V, S = out[di].contiguous(), lse[di].contiguous()
        pd.merge_state_inplace(V, S, out[si].contiguous(), lse[si].contiguous())
        out[di], lse[di] = V, S
    first = [x[0] for x in idx]
    assert pd.check_device_errors() == "PD_OK"
    ro, rl, _ = oracle_decode(wl)
    compare("bf16", out[first], lse[first], ro, rl)


def test_long_context_multi_stage_flow_of_the_bench():
    """The multi-stage flow the benchmark times beside the fused decode (32 padded
    chunk-major pseudo-sequences, fp32 partials, 5 halving merge rounds) against the
    oracle's unsplit decode."""
    import bench
    wl = _wl("long_ctx_bf16", 3)
    x = bench._external_split(wl, 32, DEV)
    out, lse = bench.run_external_split(pd, wl, x, 32)
    assert pd.check_device_errors() == "PD_OK"
    ro, rl, st = oracle_decode(wl)
    assert st == 0
    compare("bf16", out, lse, ro, rl)


@pytest.mark.parametrize("seed", [0, 5])
def test_window_sink_f16(seed):
    _check(_wl("window_sink_f16", seed), "mma")


def test_window_sink_f16_split():
    wl = _wl("window_sink_f16", 6)
    _check(wl, "mma", num_splits=7, max_kv_len_hint=int(wl.attended.max()))


@pytest.mark.parametrize("seed", [0, 7])
def test_fp8_append_then_decode(seed):
    wl = _wl("fp8_kv_highconc", seed)
    s = wl.spec
    ref_pages, bad = oracle.append_paged_kv(
        W.bits(wl.pages), W.bits(wl.k_new), W.bits(wl.v_new), wl.slot_mapping.cpu().numpy(),
        in_dtype=s.q_dtype, kv_dtype="e4m3", page_size=s.page_size, k_scale=wl.k_scale,
        v_scale=wl.v_scale)
    assert bad == 0
    pd.append_paged_kv(wl.pages, wl.k_new, wl.v_new, wl.slot_mapping, wl.k_scale, wl.v_scale)
    assert pd.check_device_errors() == "PD_OK"
    assert np.array_equal(W.bits(wl.pages), ref_pages), "append not bit-exact"
    out, lse = gpu_decode(wl)
    assert pd.last_decode_variant() == "mma"
    ro, rl, _ = oracle_decode(wl, pages=ref_pages)
    compare("e4m3", out, lse, ro, rl)


@pytest.mark.parametrize("name", ["fp8_kv_highconc", "llama3_8b_bf16", "window_sink_f16"])
def test_early_inputs_decode_starts_under_append(name):
    # With PD_DECODE_EARLY_INPUTS the decode reads Q and the page table while the append
    # before it still runs (programmatic dependent launch): the rows the append writes
    # must reach it, and of two such steps on the same out/lse the second must stand.
    wl = _wl(name, 21, append=True)
    other = _wl(name, 22, append=True)
    s = wl.spec
    ref_pages, bad = oracle.append_paged_kv(
        W.bits(wl.pages), W.bits(wl.k_new), W.bits(wl.v_new), wl.slot_mapping.cpu().numpy(),
        in_dtype=s.q_dtype, kv_dtype=s.kv_dtype, page_size=s.page_size, k_scale=wl.k_scale,
        v_scale=wl.v_scale)
    assert bad == 0
    out = torch.empty((s.B, s.H_qo, s.D), dtype=W.TORCH_DTYPES[s.out_dtype], device=DEV)
    lse = torch.empty((s.B, s.H_qo), dtype=torch.float32, device=DEV)
    for w in (other, wl):
        pd.append_paged_kv(w.pages, w.k_new, w.v_new, w.slot_mapping, w.k_scale, w.v_scale)
        pd.batch_decode_paged_kv(w.Q, w.pages, w.indptr, w.values, w.length_info,
                                 w.k_rope_pos_offset, w.q_rope_position, out, lse,
                                 s.rotary_mode, s.rope_scale, s.rope_theta, w.sm_scale,
                                 k_scale=w.k_scale, v_scale=w.v_scale, early_inputs=True)
    torch.cuda.synchronize()
    assert pd.check_device_errors() == "PD_OK"
    assert np.array_equal(W.bits(wl.pages), ref_pages)
    ro, rl, _ = oracle_decode(wl, pages=ref_pages)
    compare(kind_of(wl), out, lse, ro, rl)


@pytest.mark.parametrize("name", ["llama3_8b_bf16", "window_sink_f16", "tiny_fp32"])
def test_back_to_back_decodes_with_early_inputs(name):
    # Decodes launched one after another with PD_DECODE_EARLY_INPUTS (as the bench's
    # back-to-back timing runs them): each one's start-up runs under the previous one's
    # tail, on the same stream workspace and the same out / lse; every result must stand.
    wls = [_wl(name, 40 + i) for i in range(3)]
    s = wls[0].spec
    host = [pd.host_meta_of(w.indptr, w.length_info) for w in wls]
    outs = [torch.empty((s.B, s.H_qo, s.D), dtype=W.TORCH_DTYPES[s.out_dtype], device=DEV) for _ in wls]
    lses = [torch.empty((s.B, s.H_qo), dtype=torch.float32, device=DEV) for _ in wls]
    shared_out = torch.empty_like(outs[0])
    shared_lse = torch.empty_like(lses[0])
    for rep in range(2):
        for i, w in enumerate(wls):
            o, l = (outs[i], lses[i]) if rep == 0 else (shared_out, shared_lse)
            pd.batch_decode_paged_kv(w.Q, w.pages, w.indptr, w.values, w.length_info,
                                     w.k_rope_pos_offset, w.q_rope_position, o, l,
                                     s.rotary_mode, s.rope_scale, s.rope_theta, w.sm_scale,
                                     k_scale=w.k_scale, v_scale=w.v_scale, early_inputs=True,
                                     host_meta=host[i] if i != 1 else None)
    torch.cuda.synchronize()
    assert pd.check_device_errors() == "PD_OK"
    for i, w in enumerate(wls):
        ro, rl, _ = oracle_decode(w)
        compare(kind_of(w), outs[i], lses[i], ro, rl)
    ro, rl, _ = oracle_decode(wls[-1])
    compare(kind_of(wls[-1]), shared_out, shared_lse, ro, rl)


def test_fp8_f16_query_and_simt_variant():
    wl = _wl("fp8_kv_highconc", 8, q_dtype="f16", out_dtype="f16")
    _check(wl, "mma")
    wl2 = _wl("fp8_kv_highconc", 9, page_size=8)
    _check(wl2, "mma")
    wl3 = _wl("fp8_kv_highconc", 9, page_size=4)
    _check(wl3, "simt")


@pytest.mark.parametrize("kv", ["bf16", "f16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("group", [1, 2, 4, 8, 12, 16])
def test_shape_sweep(kv, D, group):
    rope = group % 2 == 0
    wl = _wl("llama3_8b_bf16", 10 + group, q_dtype=kv, kv_dtype=kv, out_dtype=kv, D=D,
             H_kv=2, H_qo=2 * group, B=3, len_dist=("uniform", 1, 300), pool=200,
             rotary_mode=int(rope))
    _check(wl, "mma")
    _check(wl, "mma", num_splits=4, max_kv_len_hint=300)


@pytest.mark.parametrize("group", [1, 2, 4, 12])
@pytest.mark.parametrize("rope", [0, 1])
def test_fp8_group_sweep(group, rope):
    # small slices (<= 4 heads) pack Q's lo part into the spare MMA columns; group 12
    # has an 8-head slice and a 4-head slice per KV head
    wl = _wl("fp8_kv_highconc", 40 + group, H_kv=2, H_qo=2 * group, B=3,
             len_dist=("lognormal", 200, 0.5, 1, 500), pool=64, rotary_mode=rope,
             rope_theta=1e4)
    _check(wl, "mma")
    _check(wl, "mma", num_splits=3, max_kv_len_hint=500)


@pytest.mark.parametrize("splits", [0, 1])
def test_batch_above_start_scan_cache(splits):
    # more than 1024 sequences: the tensor-core kernel's start-up scan takes its
    # two-pass path (per-sequence unit counts no longer kept in shared memory)
    wl = _wl("llama3_8b_bf16", 77, B=1100, len_dist=("uniform", 1, 40), pool=4000)
    _check(wl, "mma", num_splits=splits)


@pytest.mark.parametrize("D", [64, 128, 256])
def test_fp32_dims(D):
    wl = W.make("tiny_fp32", seed=D, D=D, rotary_mode=1, rope_theta=1e4).to(DEV)
    _check(wl, "simt")


def test_out_dtype_f32_for_bf16_cache():
    wl = _wl("llama3_8b_bf16", 11)
    _check(wl, "mma", out_dtype="f32")


# ----------------------------------------------------------------------------- edge cases

def _custom(lens, P=16, window=None, sink=0, H_qo=8, H_kv=2, D=128, dt="bf16", seed=0, rope=0):
    """Workload with explicit lengths (0 allowed)."""
    wl = W.make("llama3_8b_bf16", seed=seed, reduced=True, B=len(lens), H_qo=H_qo, H_kv=H_kv,
                D=D, page_size=P, q_dtype=dt, kv_dtype=dt, out_dtype=dt, pool=64,
                rotary_mode=rope, len_dist=("uniform", 1, 1))
    lens = np.array(lens, np.int64)
    npages = (lens + P - 1) // P
    rng = np.random.default_rng(seed + 100)
    vals = rng.permutation(wl.max_pages)[: npages.sum()].astype(np.int32)
    indptr = np.concatenate([[0], np.cumsum(npages)]).astype(np.int32)
    last = np.where(npages > 0, lens - (npages - 1) * P, 0).astype(np.int32)
    if window is None:
        li = last
        att = lens
    else:
        win_off = np.maximum(sink, lens - window).astype(np.int32)
        li = np.stack([last, win_off, np.full(len(lens), sink, np.int32)]).astype(np.int32)
        att = np.where(npages > 0, lens - win_off + sink, 0)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    spec = W.spec("llama3_8b_bf16", True, B=len(lens), H_qo=H_qo, H_kv=H_kv, D=D, page_size=P,
                  q_dtype=dt, kv_dtype=dt, out_dtype=dt, window=window, sink=sink, rotary_mode=rope)
    return W.Workload(spec=spec, Q=wl.Q, pages=wl.pages, indptr=t(indptr),
                      values=t(vals if len(vals) else np.zeros(1, np.int32)), length_info=t(li),
                      k_rope_pos_offset=t(np.zeros(len(lens), np.int32)),
                      q_rope_position=t(att.astype(np.int32)), seq_len=lens, attended=att,
                      sm_scale=wl.sm_scale).to(DEV)


def test_edge_empty_len1_fullpage():
    wl = _custom([0, 1, 16, 32, 17, 0, 15])
    out, lse = gpu_decode(wl)
    assert pd.check_device_errors() == "PD_OK"
    ro, rl, _ = oracle_decode(wl)
    compare("bf16", out, lse, ro, rl)
    assert torch.all(out[0] == 0) and torch.all(lse[0] == -5e4)
    assert torch.all(out[5] == 0) and torch.all(lse[5] == -5e4)


def test_edge_window_cases():
    # window >= len, sink = 0, window start in the middle of a page, sink crossing a page
    for lens, window, sink in [([10, 40, 100], 200, 0), ([40, 57, 123], 10, 0),
                               ([40, 57, 123], 10, 4), ([90, 91], 30, 20)]:
        wl = _custom(lens, window=window, sink=sink, dt="f16", rope=1)
        _check(wl)
        _check(wl, num_splits=3, max_kv_len_hint=int(wl.attended.max()))


@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_edge_rope_short_rows_large_positions(dt):
    # one to four rows per sequence: each lse rests on a few scores, so the rounding of
    # the rotated K to f16 is not averaged away; positions near 2^17 give large angles
    wl = _custom([1 + i % 4 for i in range(64)], H_qo=32, H_kv=8, dt=dt, rope=1, seed=5)
    wl.k_rope_pos_offset += 131000
    wl.q_rope_position += 131000
    ro, rl, _ = oracle_decode(wl)
    for kw in ({}, {"num_splits": 1}):
        out, lse = gpu_decode(wl, **kw)
        assert pd.check_device_errors() == "PD_OK"
        compare(dt, out, lse, ro, rl)
        # one f16 rounding of the rotated K (N(0,1) data, D = 128) gives an lse error of
        # about 3e-4 rms on a one-row sequence; a bf16 rounding would give 8x that
        rms = float(np.sqrt(np.mean((lse.double().cpu().numpy() - rl) ** 2)))
        assert rms <= 6e-4, rms


@pytest.mark.parametrize("P", [1, 3, 8, 24, 32, 48, 64, 128, 256])
@pytest.mark.parametrize("rope", [0, 1])
def test_page_size_sweep(P, rope):
    """Page sizes across the accepted range [1, 256]: multiples of 16 run on the
    tensor-core kernel (several 16-row tiles per page, a partial last tile), and 8 as two
    pages per tile; the others on the SIMT kernel; lengths of one row, a full page, a page plus one row, several
    pages, and empty; whole sequences and forced splits."""
    lens = [1, P, P + 1, 2 * P + 3, 5 * P - 1, 0, 7]
    wl = _custom(lens, P=P, rope=rope, seed=P)
    want = "mma" if P % 16 == 0 or P == 8 else "simt"
    _check(wl, want)
    _check(wl, want, num_splits=3, max_kv_len_hint=int(wl.attended.max()))


@pytest.mark.parametrize("P", [8, 24, 48, 256])
def test_page_size_window_sink(P):
    """Sliding window and sink rows on pages of several tiles: the window start falls
    inside a page and inside a tile."""
    lens = [3 * P + 5, 2 * P, P + 40]
    wl = _custom(lens, P=P, window=P + 21, sink=4, dt="f16", rope=1, seed=P + 1)
    want = "mma" if P % 16 == 0 or P == 8 else "simt"
    _check(wl, want)
    _check(wl, want, num_splits=3, max_kv_len_hint=int(wl.attended.max()))


def test_edge_more_chunks_than_pages():
    wl = _custom([33, 5, 70])
    _check(wl, num_splits=64, max_kv_len_hint=70)


def test_edge_all_empty_and_b0():
    wl = _custom([0, 0, 0])
    out, lse = gpu_decode(wl)
    assert pd.check_device_errors() == "PD_OK"
    assert torch.all(out == 0) and torch.all(lse == -5e4)
    wl0 = _custom([5])
    Q0 = wl0.Q[:0]
    out0 = torch.empty((0, 8, 128), dtype=torch.bfloat16, device=DEV)
    lse0 = torch.empty((0, 8), dtype=torch.float32, device=DEV)
    pd.batch_decode_paged_kv(Q0, wl0.pages, wl0.indptr[:1], wl0.values, wl0.length_info[:0],
                             None, None, out0, lse0)


def test_caller_workspace():
    wl = _wl("long_ctx_bf16", 3)
    s = wl.spec
    out = torch.empty((s.B, s.H_qo, s.D), dtype=torch.bfloat16, device=DEV)
    desc = pd.make_desc(wl.Q, wl.pages, wl.indptr, wl.values, wl.length_info, out)
    n = pd.workspace_size(desc)
    assert n > 0
    ws = torch.empty(n, dtype=torch.uint8, device=DEV)
    pd.workspace_init(ws)
    for _ in range(2):  # counters must be left at zero for the next call
        o, l = gpu_decode(wl, workspace=ws)
        assert pd.check_device_errors() == "PD_OK"
        ro, rl, _ = oracle_decode(wl)
        compare("bf16", o, l, ro, rl)
    small = torch.empty(n // 2, dtype=torch.uint8, device=DEV)
    with pytest.raises(pd.PDError, match="WORKSPACE"):
        gpu_decode(wl, workspace=small)


def test_bad_page_id_is_reported_not_trapped():
    wl = _custom([40, 20])
    vals = wl.values.clone()
    vals[1] = wl.max_pages + 5  # out of range: the row block is skipped, error recorded
    bad = W.Workload(**{**wl.__dict__, "values": vals})
    out, lse = gpu_decode(bad)
    assert pd.check_device_errors() == "PD_ERR_BAD_PAGE"
    assert pd.check_device_errors() == "PD_OK"  # the word was cleared
    # both sides exclude the rows of the bad page and agree on the rest
    ro, rl, st = oracle_decode(bad)
    assert st == -1
    compare("bf16", out, lse, ro, rl)


def test_repeatable_and_stream():
    wl = _wl("llama3_8b_bf16", 12)
    o1, l1 = gpu_decode(wl)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        o2, l2 = gpu_decode(wl, stream=st)
    st.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_split_counters_survive_layout_changes():
    """A split call with few (sequence, head) counters followed by one with many: the
    second call's counters must not see the first call's partial results."""
    a = _wl("long_ctx_bf16", 13)
    _check(a, "mma", num_splits=16, max_kv_len_hint=int(a.attended.max()))
    b = _wl("window_sink_f16", 14, B=24)
    _check(b, "mma", num_splits=3, max_kv_len_hint=int(b.attended.max()))
    _check(a, "mma", num_splits=16, max_kv_len_hint=int(a.attended.max()))


def test_caller_workspace_reused_across_layouts():
    a = _wl("long_ctx_bf16", 15)
    b = _wl("window_sink_f16", 16, B=24)
    sizes = []
    for wl in (a, b):
        s = wl.spec
        out = torch.empty((s.B, s.H_qo, s.D), dtype=wl.Q.dtype, device=DEV)
        sizes.append(pd.workspace_size(pd.make_desc(wl.Q, wl.pages, wl.indptr, wl.values,
                                                     wl.length_info, out)))
    ws = torch.empty(max(sizes), dtype=torch.uint8, device=DEV)
    pd.workspace_init(ws)
    for wl in (a, b, a, b):
        _check(wl, "mma", workspace=ws)


# ----------------------------------------------------------------------------- interleaved RoPE

@pytest.mark.parametrize("kv", ["bf16", "f16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("group", [2, 4, 8])
def test_rope_interleaved_mma(kv, D, group):
    # rotary_mode 2: the pair (2i, 2i + 1) shares frequency i (one A-fragment register)
    wl = _wl("llama3_8b_bf16", 80 + group, q_dtype=kv, kv_dtype=kv, out_dtype=kv, D=D,
             H_kv=2, H_qo=2 * group, B=3, len_dist=("uniform", 1, 300), pool=200, rotary_mode=2)
    _check(wl, "mma")
    _check(wl, "mma", num_splits=3, max_kv_len_hint=300)


def test_rope_interleaved_fp8_and_window():
    _check(_wl("fp8_kv_highconc", 90, rotary_mode=2, rope_theta=1e4), "mma")
    _check(_wl("window_sink_f16", 91, rotary_mode=2), "mma")


@pytest.mark.parametrize("D", [64, 128, 256])
def test_rope_interleaved_simt(D):
    wl = W.make("tiny_fp32", seed=92 + D, D=D, rotary_mode=2, rope_theta=1e4).to(DEV)
    _check(wl, "simt")
    _check(_wl("llama3_8b_bf16", 93, page_size=4, pool=2400, rotary_mode=2), "simt")
    _check(_wl("llama3_8b_bf16", 93, page_size=8, pool=1200, rotary_mode=2), "mma")


# ----------------------------------------------------------------------------- learned sinks

def _sink(wl, seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    return (torch.randn(wl.spec.H_qo, generator=g, device=DEV) * 3).float()


@pytest.mark.parametrize("name,over", [("llama3_8b_bf16", {}), ("fp8_kv_highconc", {}),
                                       ("window_sink_f16", {}), ("tiny_fp32", {})])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_sink_logits(name, over, splits):
    # a per-head logit joins the softmax with a zero value row, once per (sequence, head)
    # whether the segment is split or not
    wl = _wl(name, 94, **over)
    sk = _sink(wl, 95)
    kw = dict(num_splits=splits)
    if splits == 3:
        kw["max_kv_len_hint"] = int(wl.attended.max())
    out, lse = gpu_decode(wl, sink=sk, **kw)
    assert pd.check_device_errors() == "PD_OK"
    ro, rl, st = oracle_decode(wl, sink=sk.cpu().numpy())
    assert st == 0
    compare(kind_of(wl), out, lse, ro, rl)


def test_sink_empty_sequence_and_noalloc():
    wl = _custom([0, 5, 40], seed=9)
    sk = _sink(wl, 96)
    out, lse = gpu_decode(wl, sink=sk)
    ro, rl, _ = oracle_decode(wl, sink=sk.cpu().numpy())
    compare("bf16", out, lse, ro, rl)
    assert torch.all(out[0] == 0)
    torch.testing.assert_close(lse[0], sk * 1.4426950408889634, rtol=0, atol=1e-5)
    s = wl.spec
    out2 = torch.empty_like(out)
    lse2 = torch.empty_like(lse)
    pd.batch_decode_paged_kv_noalloc(wl.Q, wl.pages, wl.indptr, wl.values, wl.length_info,
                                     wl.k_rope_pos_offset, wl.q_rope_position, out2, lse2,
                                     s.rotary_mode, s.rope_scale, s.rope_theta, wl.sm_scale,
                                     sink=sk)
    assert torch.equal(out2, out) and torch.equal(lse2, lse)


# ----------------------------------------------------------------------------- workspace per stream

def test_library_workspace_two_streams_concurrently():
    """Split decodes of two different workloads in flight at once on two streams, both
    with the library-managed workspace: each stream has its own arena, so neither sees
    the other's arrival counters or partial slots; each matches the oracle."""
    a = _wl("long_ctx_bf16", 300)
    b = _wl("window_sink_f16", 301, B=16)
    ra, rb = oracle_decode(a), oracle_decode(b)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    outs = []
    for rep in range(3):
        with torch.cuda.stream(sa):
            oa, la = gpu_decode(a, stream=sa, num_splits=16, max_kv_len_hint=int(a.attended.max()))
        with torch.cuda.stream(sb):
            ob, lb = gpu_decode(b, stream=sb, num_splits=5, max_kv_len_hint=int(b.attended.max()))
        outs.append((oa, la, ob, lb))
    torch.cuda.synchronize()
    assert pd.check_device_errors() == "PD_OK"
    for oa, la, ob, lb in outs:
        compare("bf16", oa, la, ra[0], ra[1])
        compare("f16", ob, lb, rb[0], rb[1])
    for st in (sa, sb):
        pd.release_stream_workspace(st)
    pd.release_stream_workspace(torch.cuda.Stream())  # no arena: nothing to do


def test_library_workspace_grows_behind_work_in_flight():
    """A small split decode, then at once a much larger one on the same stream: the
    arena grows while the first kernel may still run (the old buffer is released
    stream-ordered, after it); both results match the oracle."""
    st = torch.cuda.Stream()
    pd.release_stream_workspace(st)
    small = _wl("llama3_8b_bf16", 302, B=2)
    big = _wl("llama3_8b_bf16", 303, B=40, len_dist=("uniform", 100, 900), pool=3000)
    rs, rb = oracle_decode(small), oracle_decode(big)
    torch.cuda.synchronize()
    with torch.cuda.stream(st):
        o1, l1 = gpu_decode(small, stream=st, num_splits=3, max_kv_len_hint=700)
        o2, l2 = gpu_decode(big, stream=st, num_splits=24, max_kv_len_hint=900)
        o3, l3 = gpu_decode(small, stream=st, num_splits=3, max_kv_len_hint=700)
    st.synchronize()
    assert pd.check_device_errors() == "PD_OK"
    compare("bf16", o1, l1, rs[0], rs[1])
    compare("bf16", o2, l2, rb[0], rb[1])
    compare("bf16", o3, l3, rs[0], rs[1])
    pd.release_stream_workspace(st)
