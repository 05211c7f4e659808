"""GPU parity of merge_state_inplace and append_paged_kv (C ABI) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_19_gb300 import workloads as W

pd = pytest.importorskip("paged_kv_decode_19_gb300")
pytestmark = pytest.mark.gpu
DEV = "cuda"


# f32: fp32-level; bf16/f16: the 16-bit bound of the decode contract (max abs 2e-2),
# which covers rounding the merged values (|v| up to ~5) to the storage type.
@pytest.mark.parametrize("dt,tol", [("f32", 2e-6), ("bf16", 2e-2), ("f16", 2e-2)])
@pytest.mark.parametrize("shape", [(8, 32, 128), (3, 5, 64), (1, 1, 256), (7, 3, 96)])
def test_merge_state(dt, tol, shape):
    g = torch.Generator().manual_seed(hash((dt, shape)) & 0xffff)
    N, H, D = shape
    tdt = W.TORCH_DTYPES[dt]
    V = torch.randn(N, H, D, generator=g).to(tdt)
    Vo = torch.randn(N, H, D, generator=g).to(tdt)
    S = (torch.randn(N, H, generator=g) * 4).float()
    So = (torch.randn(N, H, generator=g) * 4).float()
    S[0, 0] = -5e4  # identity partner on one row
    ref_v, ref_s = oracle.merge_state(oracle.decode(W.bits(V), dt), S.double().numpy(),
                                      oracle.decode(W.bits(Vo), dt), So.double().numpy())
    Vd, Sd = V.to(DEV), S.to(DEV)
    pd.merge_state_inplace(Vd, Sd, Vo.to(DEV), So.to(DEV))
    torch.cuda.synchronize()
    assert np.abs(Vd.double().cpu().numpy() - ref_v).max() <= tol
    assert np.abs(Sd.double().cpu().numpy() - ref_s).max() <= 1e-5 * max(1.0, np.abs(ref_s).max())
    # S = -5e4 on the first input: result equals the partner row
    np.testing.assert_allclose(Vd[0, 0].double().cpu().numpy(),
                               oracle.decode(W.bits(Vo[0, 0]), dt), atol=tol)


def test_merge_identity_partner():
    V = torch.randn(4, 8, 128, device=DEV)
    S = torch.randn(4, 8, device=DEV)
    V0, S0 = V.clone(), S.clone()
    pd.merge_state_inplace(V, S, torch.zeros_like(V), torch.full_like(S, -5e4))
    torch.cuda.synchronize()
    assert torch.allclose(V, V0, atol=1e-6) and torch.allclose(S, S0, atol=1e-5)


@pytest.mark.parametrize("in_dt,kv_dt", [("bf16", "bf16"), ("f16", "f16"), ("f32", "f32"),
                                         ("bf16", "e4m3"), ("f16", "e4m3"), ("f32", "e4m3"),
                                         ("f32", "bf16"), ("f32", "f16"), ("bf16", "f16"),
                                         ("f16", "bf16")])
@pytest.mark.parametrize("D", [64, 128])
def test_append_bit_exact(in_dt, kv_dt, D):
    g = torch.Generator().manual_seed(D + len(in_dt) * 7 + len(kv_dt))
    T, H, P, pool = 37, 4, 16, 12
    x = torch.randn(pool, 2, H, P, D, generator=g) * 3
    ks, vs = 11.0 / 448, 9.5 / 448
    if kv_dt == "e4m3":
        pages = torch.empty(x.shape, dtype=torch.float8_e4m3fn)
        pages[:, 0] = (x[:, 0] / ks).to(torch.float8_e4m3fn)
        pages[:, 1] = (x[:, 1] / vs).to(torch.float8_e4m3fn)
    else:
        pages = x.to(W.TORCH_DTYPES[kv_dt])
    k = (torch.randn(T, H, D, generator=g) * 4).to(W.TORCH_DTYPES[in_dt])
    v = (torch.randn(T, H, D, generator=g) * 4).to(W.TORCH_DTYPES[in_dt])
    k[0, 0, :4] = torch.tensor([1e4, -1e4, 0.0, -0.0]).to(k.dtype)  # saturation and signed zero
    slots = torch.from_numpy(np.random.default_rng(D).permutation(pool * P)[:T].astype(np.int64))
    slots[3] = -1
    slots[7] = -1
    ref, bad = oracle.append_paged_kv(W.bits(pages), W.bits(k), W.bits(v), slots.numpy(),
                                      in_dtype=in_dt, kv_dtype=kv_dt, page_size=P, k_scale=ks,
                                      v_scale=vs)
    assert bad == 0
    pg = pages.to(DEV)
    pd.append_paged_kv(pg, k.to(DEV), v.to(DEV), slots.to(DEV), ks, vs)
    assert pd.check_device_errors() == "PD_OK"
    assert np.array_equal(W.bits(pg), ref)


def test_append_out_of_range_slot_reported():
    pages = torch.zeros(2, 2, 1, 16, 64, dtype=torch.bfloat16, device=DEV)
    k = torch.ones(2, 1, 64, dtype=torch.bfloat16, device=DEV)
    slots = torch.tensor([5, 32], dtype=torch.int64, device=DEV)
    pd.append_paged_kv(pages, k, k, slots)
    assert pd.check_device_errors() == "PD_ERR_BAD_SLOT"
    assert torch.all(pages[0, :, 0, 5] == 1) and int((pages != 0).sum()) == 2 * 64
