"""Shared helpers of the parity tests: run the CUDA path and the oracle on the same
seeded workload and compare with the tolerances of the decode contract."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_kv_decode_19_gb300 import workloads as W

# Tolerances (written here, used by every parity test):
#   fp32       per (sequence, head) output vector: max_d |gpu - ref| <= 1e-5 * max_d |ref|
#              (norm-wise relative error; elementwise relative error is ill-posed for
#              components that are near-zero results of cancellation), lse |d| <= 1e-5 *
#              max(1, |ref|)
#   bf16/f16   max |out - ref| <= 2e-2, max |lse - ref| <= 2e-3 (log2 units)
#   e4m3 KV    max |out - ref| <= 3e-2, max |lse - ref| <= 3e-2 vs the oracle on the
#              dequantised cache
TOL = {"f32": (None, None), "bf16": (2e-2, 2e-3), "f16": (2e-2, 2e-3), "e4m3": (3e-2, 3e-2)}


def oracle_decode(wl: W.Workload, pages=None, mask=None, **over):
    s = wl.spec
    kw = dict(q_dtype=s.q_dtype, kv_dtype=s.kv_dtype, H_kv=s.H_kv, page_size=s.page_size,
              rotary_mode=s.rotary_mode, rope_scale=s.rope_scale, rope_theta=s.rope_theta,
              sm_scale=wl.sm_scale, sliding_window=s.window is not None, k_scale=wl.k_scale,
              v_scale=wl.v_scale, mask=mask)
    kw.update(over)
    return oracle.batch_decode_paged_kv(
        W.bits(wl.Q), W.bits(wl.pages) if pages is None else pages, wl.indptr.cpu().numpy(),
        wl.values.cpu().numpy(), wl.length_info.cpu().numpy(), wl.k_rope_pos_offset.cpu().numpy(),
        wl.q_rope_position.cpu().numpy(), **kw)


def gpu_decode(wl: W.Workload, out_dtype=None, **kw):
    """Run the CUDA path on a workload already on the GPU; returns (out, lse) tensors."""
    import paged_kv_decode_19_gb300 as pd
    s = wl.spec
    odt = W.TORCH_DTYPES[out_dtype or s.out_dtype]
    out = torch.full((s.B, s.H_qo, s.D), float("nan"), dtype=odt, device=wl.Q.device)
    lse = torch.full((s.B, s.H_qo), float("nan"), dtype=torch.float32, device=wl.Q.device)
    pd.batch_decode_paged_kv(wl.Q, wl.pages, wl.indptr, wl.values, wl.length_info,
                             wl.k_rope_pos_offset, wl.q_rope_position, out, lse,
                             s.rotary_mode, s.rope_scale, s.rope_theta, wl.sm_scale,
                             k_scale=wl.k_scale, v_scale=wl.v_scale, **kw)
    return out, lse


def compare(kind, out_gpu, lse_gpu, out_ref, lse_ref, mask=None):
    """Assert parity; returns (max abs out err, max abs lse err)."""
    og = out_gpu.float().cpu().double().numpy()
    lg = lse_gpu.float().cpu().double().numpy()
    if mask is not None:
        og, lg, out_ref, lse_ref = og[mask], lg[mask], out_ref[mask], lse_ref[mask]
    assert np.all(np.isfinite(og)) and np.all(np.isfinite(lg)), "non-finite GPU output"
    eo = np.abs(og - out_ref)
    el = np.abs(lg - lse_ref)
    if kind == "f32":
        row_max = np.abs(out_ref).max(axis=-1, keepdims=True)
        bound = 1e-5 * np.maximum(row_max, 1e-30)
        assert np.all(eo <= bound), f"fp32 out error {eo.max():.3e} (worst ratio {(eo / bound).max():.2f})"
        assert np.all(el <= 1e-5 * np.maximum(1.0, np.abs(lse_ref))), f"fp32 lse error {el.max():.3e}"
    else:
        to, tl = TOL[kind]
        assert eo.max() <= to, f"{kind} out max abs error {eo.max():.4e} > {to}"
        assert el.max() <= tl, f"{kind} lse max abs error {el.max():.4e} > {tl}"
    return float(eo.max()), float(el.max())


def kind_of(wl: W.Workload) -> str:
    """Tolerance class of a workload: its KV element type."""
    return wl.spec.kv_dtype
