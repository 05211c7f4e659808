"""The online softmax's rescale of a non-empty state, against the fp64 oracle.

The decode kernels keep a running maximum m per query column and rescale the output
accumulators and the denominator by 2^(m_old - m_new) when it moves (Apache TVM
`_decode_kernels.py`, `batch_decode_paged_kv`: the m / d / O update of the online
softmax).  The tensor-core kernel moves m lazily, only when a score exceeds it by more
than 2^8.  On the N(0,1) inputs of the serving loads that happens on a worker's first
tile alone, where O and d are still zero, so the multiply of a non-empty state is never
reached.  The inputs here reach it on many tiles:

  rising   every cached K row at sequence offset o is scaled by 1 + k_ramp * o / (len-1):
           scores grow along the sequence, and the running maximum jumps by more than the
           slack several times per segment;
  peaked   Q scaled by q_gain: a sharp softmax whose maximum moves on later tiles.

Each runs whole and with forced splits, with the query packing of small slices (<= 4
columns, split operands), multi-query columns, E4M3 caches, RoPE in the kernel and RoPE
at append time, and once at full size in the benchmark's launch configuration.  A wrong
pairing of rescale factors to accumulator columns, or a wrong column reduction of the
tile maximum, changes outputs by O(1) here.

Tolerances.  Where the kernel multiplies K as stored (no RoPE, RoPE on Q only, E4M3
codes, which are exact in f16), a score carries fp32-level error and the contract's
tolerances apply unchanged (bf16/f16: out 2e-2, lse 2e-3; e4m3: 3e-2).  Where it
rotates K itself, the rotated K is rounded once to f16 (relative error <= 2^-11 per
element), so a score's error scales with the magnitude of q and k: scores `gain` times
those of N(0,1) inputs (gain = (1 + k_ramp) * q_gain) get lse tolerance 2e-3 * gain.
A score error ds moves the output by at most about ln 2 * ds * max|v| (max|v| < 5 for
these draws), so out gets max(2e-2, 3 * lse tolerance).
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_19_gb300 import workloads as W
from tests._util import TOL, compare, gpu_decode, oracle_decode

pd = pytest.importorskip("paged_kv_decode_19_gb300")
pytestmark = pytest.mark.gpu
DEV = "cuda"


def _tol(spec, krot_in_kernel):
    to, tl = TOL[spec.kv_dtype]
    if krot_in_kernel:
        gain = (1.0 + spec.k_ramp) * spec.q_gain
        tl = tl * gain
        to = max(to, 3.0 * tl)
    return to, tl


def _cmp(spec, out, lse, ro, rl, krot_in_kernel, mask=None):
    og = out.float().cpu().double().numpy()
    lg = lse.float().cpu().double().numpy()
    if mask is not None:
        og, lg, ro, rl = og[mask], lg[mask], ro[mask], rl[mask]
    assert np.all(np.isfinite(og)) and np.all(np.isfinite(lg)), "non-finite GPU output"
    to, tl = _tol(spec, krot_in_kernel)
    eo, el = np.abs(og - ro).max(), np.abs(lg - rl).max()
    assert eo <= to, f"out max abs error {eo:.4e} > {to:.3e}"
    assert el <= tl, f"lse max abs error {el:.4e} > {tl:.3e}"
    return eo, el


def _run(wl, krot_in_kernel, splits=(0, 1, 3), **kw):
    ro, rl, st = oracle_decode(wl)
    assert st == 0
    for sp in splits:
        extra = dict(num_splits=sp)
        if sp > 1:
            extra["max_kv_len_hint"] = int(wl.attended.max())
        out, lse = gpu_decode(wl, **extra, **kw)
        assert pd.check_device_errors() == "PD_OK"
        _cmp(wl.spec, out, lse, ro, rl, krot_in_kernel)


@pytest.mark.parametrize("kv", ["bf16", "f16"])
@pytest.mark.parametrize("group", [2, 4, 8])
@pytest.mark.parametrize("profile", [dict(k_ramp=8.0), dict(q_gain=8.0)])
def test_rescale_16bit_no_rope(kv, group, profile):
    # bf16/f16 Q equal to the cache type: the unsplit-operand QK (no query packing)
    wl = W.make("llama3_8b_bf16", seed=200 + group, reduced=True, q_dtype=kv, kv_dtype=kv,
                out_dtype=kv, H_kv=2, H_qo=2 * group, rotary_mode=0, **profile).to(DEV)
    _run(wl, krot_in_kernel=False)


@pytest.mark.parametrize("group", [2, 4, 8, 12])
@pytest.mark.parametrize("profile", [dict(k_ramp=8.0), dict(q_gain=8.0)])
def test_rescale_fp8(group, profile):
    # E4M3 KV with a bf16 query: split-operand QK; slices of <= 4 columns pack Q's lo part
    # into the spare MMA columns (groups 2 and 4, and the 4-column slice of group 12)
    wl = W.make("fp8_kv_highconc", seed=210 + group, reduced=True, H_kv=2, H_qo=2 * group,
                B=4, pool=96, **profile).to(DEV)
    _run(wl, krot_in_kernel=False)


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("profile", [dict(k_ramp=4.0), dict(q_gain=4.0)])
def test_rescale_rope_in_kernel(mode, profile):
    # llama3 shapes (group 4: packed split-operand slices) and the window + sink load
    # (group 8), K rotated in the tile loop
    wl = W.make("llama3_8b_bf16", seed=220 + mode, reduced=True, rotary_mode=mode,
                **profile).to(DEV)
    _run(wl, krot_in_kernel=True)
    ws = W.make("window_sink_f16", seed=222 + mode, reduced=True, rotary_mode=mode,
                **profile).to(DEV)
    _run(ws, krot_in_kernel=True)


@pytest.mark.parametrize("name", ["llama3_8b_bf16", "window_sink_f16", "fp8_kv_highconc"])
def test_rescale_rope_at_append(name):
    # the cache holds K rotated at append time (rotation preserves the ramp's row
    # norms); the decode rotates Q only and multiplies K as stored
    from tests.test_rope_cache_gpu import _rotate_cache
    over = dict(rotary_mode=1, rope_theta=1e4) if name == "fp8_kv_highconc" else {}
    wl = W.make(name, seed=230, reduced=True, k_ramp=8.0, **over).to(DEV)
    s = wl.spec
    ref_pages = _rotate_cache(wl, s.rotary_mode)
    ro, rl, st = oracle.batch_decode_paged_kv(
        W.bits(wl.Q), ref_pages, wl.indptr.cpu().numpy(), wl.values.cpu().numpy(),
        wl.length_info.cpu().numpy(), None, wl.q_rope_position.cpu().numpy(), q_dtype=s.q_dtype,
        kv_dtype=s.kv_dtype, H_kv=s.H_kv, page_size=s.page_size, rotary_mode=s.rotary_mode,
        rope_scale=s.rope_scale, rope_theta=s.rope_theta, sm_scale=wl.sm_scale,
        sliding_window=s.window is not None, k_scale=wl.k_scale, v_scale=wl.v_scale,
        k_rotated=True)
    assert st == 0
    for sp in (0, 1, 3):
        kw = dict(num_splits=sp, max_kv_len_hint=int(wl.attended.max()) if sp > 1 else 0)
        out = torch.empty((s.B, s.H_qo, s.D), dtype=W.TORCH_DTYPES[s.out_dtype], device=DEV)
        lse = torch.empty((s.B, s.H_qo), dtype=torch.float32, device=DEV)
        pd.batch_decode_paged_kv(wl.Q, wl.pages, wl.indptr, wl.values, wl.length_info, None,
                                 wl.q_rope_position, out, lse, s.rotary_mode, s.rope_scale,
                                 s.rope_theta, wl.sm_scale, k_scale=wl.k_scale,
                                 v_scale=wl.v_scale, k_rotated=True, **kw)
        assert pd.check_device_errors() == "PD_OK"
        _cmp(s, out, lse, ro, rl, krot_in_kernel=False)


@pytest.mark.parametrize("q_len,group,rope", [(2, 4, 0), (3, 4, 0), (2, 8, 0), (4, 2, 0),
                                              (2, 4, 1)])
def test_rescale_multi_query(q_len, group, rope):
    # (token, head) columns; the causal limit masks each token's own later rows
    from tests.test_mq_gpu import _gpu, _oracle
    wl = W.make("llama3_8b_bf16", seed=240 + q_len + group, reduced=True, H_kv=2,
                H_qo=2 * group, rotary_mode=rope, k_ramp=8.0 if not rope else 4.0).to(DEV)
    s = wl.spec
    g = torch.Generator(device=DEV)
    g.manual_seed(241)
    Q = torch.randn((s.B, q_len, s.H_qo, s.D), generator=g, device=DEV).to(torch.bfloat16)
    wl.q_rope_position = torch.from_numpy(np.maximum(wl.attended - q_len, 0).astype(np.int32)).to(DEV)
    ro, rl, st = _oracle(wl, Q, q_len)
    assert st == 0
    for sp in (0, 1, 3):
        kw = dict(num_splits=sp, max_kv_len_hint=int(wl.attended.max()) if sp > 1 else 0)
        out, lse = _gpu(wl, Q, **kw)
        assert pd.check_device_errors() == "PD_OK"
        _cmp(s, out, lse, ro, rl, krot_in_kernel=bool(rope))


@pytest.mark.parametrize("profile", [dict(k_ramp=8.0), dict(q_gain=8.0)])
def test_rescale_fp32_simt(profile):
    # the SIMT kernel (fp32 cache) keeps its own running maximum per warp
    wl = W.make("tiny_fp32", seed=250, **profile).to(DEV)
    ro, rl, st = oracle_decode(wl)
    assert st == 0
    for sp in (0, 1):
        out, lse = gpu_decode(wl, num_splits=sp)
        assert pd.check_device_errors() == "PD_OK"
        compare("f32", out, lse, ro, rl)


def test_rescale_fullsize_bench_launch():
    """Llama-3 shapes at full size with the rising profile, in the benchmark's launch
    configuration (automatic split, early inputs), RoPE in the kernel: sampled
    (sequence, head) outputs against the oracle."""
    from tests.test_fullsize_gpu import _sample_mask
    wl = W.make("llama3_8b_bf16", seed=1000, device=DEV, k_ramp=4.0)
    out, lse = gpu_decode(wl, early_inputs=True)
    assert pd.check_device_errors() == "PD_OK"
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    mask = _sample_mask(wl, n_rand=8, seed=3)
    ro, rl, st = oracle_decode(wl, mask=mask)
    assert st == 0
    _cmp(wl.spec, out, lse, ro, rl, krot_in_kernel=True, mask=mask)
