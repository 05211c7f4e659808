"""The decode captured in a CUDA graph and replayed on new inputs.

A serving loop captures the step once and replays it with the next step's Q, pages and
page table copied into the same device buffers. With the split planned on the device
(no host copies of the page table), the replayed kernels read whatever those buffers
hold at replay time, so every replay must match the oracle on its own inputs."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_19_gb300 import workloads as W
from tests._util import compare, kind_of, oracle_decode

pd = pytest.importorskip("paged_kv_decode_19_gb300")
pytestmark = pytest.mark.gpu
DEV = "cuda"


def _variant(wl, seed):
    """Same shapes as wl: new Q and cache contents, page ids permuted within the pool and
    new last-page lengths (so new attended lengths)."""
    s = wl.spec
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    Q = torch.randn(wl.Q.shape, generator=g, device=DEV).to(wl.Q.dtype)
    pages = torch.randn(wl.pages.shape, generator=g, device=DEV).to(wl.pages.dtype)
    rng = np.random.default_rng(seed)
    max_pages = wl.pages.shape[0]
    values = rng.permutation(max_pages)[: wl.values.numel()].astype(np.int32)
    assert wl.length_info.dim() == 1, "no sliding window here"
    npages = np.diff(wl.indptr.cpu().numpy())
    li = rng.integers(1, s.page_size + 1, size=s.B).astype(np.int32)
    li[npages == 0] = 0
    return dataclasses.replace(wl, Q=Q, pages=pages,
                               values=torch.from_numpy(values).to(DEV),
                               length_info=torch.from_numpy(li).to(DEV))


def _oracle_of(v):
    s = v.spec
    if s.q_len == 1:
        return oracle_decode(v)
    return oracle.batch_decode_paged_kv_mq(
        W.bits(v.Q), W.bits(v.pages), v.indptr.cpu().numpy(), v.values.cpu().numpy(),
        v.length_info.cpu().numpy(), v.k_rope_pos_offset.cpu().numpy(),
        v.q_rope_position.cpu().numpy(), q_len=s.q_len, q_dtype=s.q_dtype, kv_dtype=s.kv_dtype,
        H_kv=s.H_kv, page_size=s.page_size, rotary_mode=s.rotary_mode, rope_scale=s.rope_scale,
        rope_theta=s.rope_theta, sm_scale=v.sm_scale)


@pytest.mark.parametrize("name", ["llama3_8b_bf16", "fp8_kv_highconc", "tiny_fp32",
                                  "spec_decode_bf16"])
def test_decode_replayed_from_cuda_graph(name):
    wl = W.make(name, seed=90, reduced=True).to(DEV)
    s = wl.spec
    variants = [wl, _variant(wl, 91), _variant(wl, 92)]
    # the step's device buffers, refilled before each replay
    buf = {k: getattr(wl, k).clone() for k in ("Q", "pages", "indptr", "values", "length_info",
                                               "k_rope_pos_offset", "q_rope_position")}
    qd = (s.B,) if s.q_len == 1 else (s.B, s.q_len)
    out = torch.empty(qd + (s.H_qo, s.D), dtype=W.TORCH_DTYPES[s.out_dtype], device=DEV)
    lse = torch.empty(qd + (s.H_qo,), dtype=torch.float32, device=DEV)
    kw = dict(num_splits=1) if name == "tiny_fp32" else {}
    api = pd.batch_decode_paged_kv if s.q_len == 1 else pd.batch_decode_paged_kv_mq

    def step():
        api(buf["Q"], buf["pages"], buf["indptr"], buf["values"], buf["length_info"],
            buf["k_rope_pos_offset"], buf["q_rope_position"], out, lse, s.rotary_mode,
            s.rope_scale, s.rope_theta, wl.sm_scale, k_scale=wl.k_scale, v_scale=wl.v_scale,
            **kw)

    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        step()  # warm-up on the capture stream (its workspace, the kernels' attributes)
    cap.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        step()
    torch.cuda.synchronize()
    for v in variants[1:] + variants[:1]:
        for k in buf:
            buf[k].copy_(getattr(v, k))
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert pd.check_device_errors() == "PD_OK"
        ro, rl, st = _oracle_of(v)
        assert st == 0
        compare(kind_of(v), out, lse, ro, rl)


def test_capture_without_a_ready_workspace_is_refused():
    """A split decode captured on a stream whose library workspace was never sized: the
    call is refused with PD_ERR_WORKSPACE before anything is enqueued (no allocation
    behind the graph's back), and the stream stays usable."""
    wl = W.make("llama3_8b_bf16", seed=93, reduced=True).to(DEV)
    s = wl.spec
    out = torch.empty((s.B, s.H_qo, s.D), dtype=W.TORCH_DTYPES[s.out_dtype], device=DEV)
    lse = torch.empty((s.B, s.H_qo), dtype=torch.float32, device=DEV)
    cap = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    refused = None
    with torch.cuda.graph(graph, stream=cap):
        try:
            pd.batch_decode_paged_kv(wl.Q, wl.pages, wl.indptr, wl.values, wl.length_info,
                                     wl.k_rope_pos_offset, wl.q_rope_position, out, lse,
                                     s.rotary_mode, s.rope_scale, s.rope_theta, wl.sm_scale,
                                     num_splits=4, max_kv_len_hint=int(wl.attended.max()))
        except pd.PDError as e:
            refused = e
    assert refused is not None and refused.status_name == "PD_ERR_WORKSPACE"
    torch.cuda.synchronize()
    with torch.cuda.stream(cap):  # the same call outside capture runs and is right
        pd.batch_decode_paged_kv(wl.Q, wl.pages, wl.indptr, wl.values, wl.length_info,
                                 wl.k_rope_pos_offset, wl.q_rope_position, out, lse,
                                 s.rotary_mode, s.rope_scale, s.rope_theta, wl.sm_scale,
                                 num_splits=4, max_kv_len_hint=int(wl.attended.max()))
    cap.synchronize()
    assert pd.check_device_errors() == "PD_OK"
    ro, rl, _ = oracle_decode(wl)
    compare(kind_of(wl), out, lse, ro, rl)
