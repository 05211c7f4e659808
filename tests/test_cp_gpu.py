"""Context-parallel decode on one GPU: the ranks' slices are decoded in turn (each into
its row of the buffer an all-gather would fill), then combined with pd_merge_states;
the result is compared with the oracle's unsplit decode.  pd_merge_states itself is
compared with the oracle's merge of R states on random states, in both partner layouts,
every output type and with empty partners."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_19_gb300 import workloads as W
from tests._util import compare, oracle_decode

pd = pytest.importorskip("paged_kv_decode_19_gb300")
from paged_kv_decode_19_gb300 import cp  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _cp_decode_one_gpu(wl, world, **kw):
    s = wl.spec
    B, H, D = s.B, s.H_qo, s.D
    gathered = torch.full((world, cp.packed_width(B, H, D)), float("nan"), dtype=torch.float32,
                          device=DEV)
    for r in range(world):
        sh = cp.shard(wl.indptr, wl.values, wl.length_info, wl.k_rope_pos_offset, s.page_size,
                      world, r, DEV)
        cp.decode_partial(wl.Q, wl.pages, sh, wl.q_rope_position, gathered[r], s.rotary_mode,
                          s.rope_scale, s.rope_theta, wl.sm_scale, k_scale=wl.k_scale,
                          v_scale=wl.v_scale, **kw)
    out = torch.full((B, H, D), float("nan"), dtype=W.TORCH_DTYPES[s.out_dtype], device=DEV)
    lse = torch.full((B, H), float("nan"), dtype=torch.float32, device=DEV)
    cp.combine(gathered, out, lse)
    assert pd.check_device_errors() == "PD_OK"
    return out, lse


@pytest.mark.parametrize("name", ["llama3_8b_bf16", "long_ctx_bf16", "fp8_kv_highconc"])
@pytest.mark.parametrize("world", [2, 3, 8])
def test_context_parallel_equals_unsplit(name, world):
    over = dict(rotary_mode=1, rope_theta=1e4) if name == "fp8_kv_highconc" else {}
    wl = W.make(name, seed=400 + world, reduced=True, **over).to(DEV)
    ro, rl, st = oracle_decode(wl)
    assert st == 0
    for splits in (0, 1):
        out, lse = _cp_decode_one_gpu(wl, world, num_splits=splits)
        compare(wl.spec.kv_dtype, out, lse, ro, rl)


def test_context_parallel_short_and_empty_sequences():
    # sequences of fewer pages than ranks leave some ranks an empty slice
    wl = W.make("llama3_8b_bf16", seed=410, reduced=True, B=6, len_dist=("uniform", 0, 40),
                pool=64).to(DEV)
    assert (wl.seq_len < 4 * wl.spec.page_size).all()
    ro, rl, _ = oracle_decode(wl)
    out, lse = _cp_decode_one_gpu(wl, 4)
    compare("bf16", out, lse, ro, rl)
    empty = wl.seq_len == 0
    if empty.any():
        assert torch.all(lse[torch.from_numpy(empty).to(DEV)] == -5e4)


@pytest.mark.parametrize("R,D", [(1, 128), (2, 128), (5, 128), (33, 128), (70, 128), (3, 64),
                                 (6, 256), (4, 96), (7, 320), (35, 40)])
@pytest.mark.parametrize("odt", ["f32", "bf16", "f16"])
def test_merge_states_matches_oracle(R, D, odt):
    # partner counts below, at and above a warp (the lanes hold the first 32 weights), and
    # head dims of one chunk per lane, ragged ones and more than 256 (several chunks)
    g = torch.Generator(device=DEV)
    g.manual_seed(R * 1000 + D)
    N, H = 5, 6
    Vp = torch.randn((R, N, H, D), generator=g, device=DEV)
    Sp = torch.rand((R, N, H), generator=g, device=DEV) * 20 - 10
    Sp[0, 1] = -5e4                     # an empty partner
    Vp[0, 1] = 0
    if R > 1:
        Sp[:, 2, 3] = -5e4              # a row whose partners are all empty
        Vp[:, 2, 3] = 0
    ro, rl = oracle.merge_states(Vp.double().cpu().numpy(), Sp.double().cpu().numpy())
    out = torch.full((N, H, D), float("nan"), dtype=W.TORCH_DTYPES[odt], device=DEV)
    lse = torch.full((N, H), float("nan"), dtype=torch.float32, device=DEV)
    pd.merge_states(out, lse, Vp, Sp)
    torch.cuda.synchronize()
    tol = 1e-5 if odt == "f32" else 2e-2
    np.testing.assert_allclose(out.double().cpu().numpy(), ro, rtol=0, atol=tol)
    np.testing.assert_allclose(lse.double().cpu().numpy(), rl, rtol=0, atol=1e-4)
    # the packed layout (one [out | lse] block per partner) gives the same result
    packed = torch.cat([Vp.reshape(R, -1), Sp.reshape(R, -1)], dim=1).contiguous()
    out2 = torch.empty_like(out)
    lse2 = torch.empty_like(lse)
    pd.merge_states_packed(out2, lse2, packed)
    torch.cuda.synchronize()
    assert torch.equal(out2, out) and torch.equal(lse2, lse)
