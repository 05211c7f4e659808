"""Context-parallel decode, host side (no GPU): the library's shard plan
(pd_cp_shard_plan, a host-only C call) and the exchange / combine bookkeeping of
paged_kv_decode_19_gb300.cp with two gloo ranks on CPU.  Each rank's slice is decoded by
the fp64 oracle here (standing in for the GPU decode), exchanged with the module's
all-gather, and combined with the oracle's merge of R states; every rank must end with
the oracle's unsplit decode."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from paged_kv_decode_19_gb300 import _lib
from paged_kv_decode_19_gb300 import workloads as W


def _lib_or_skip():
    try:
        return _lib.lib()
    except RuntimeError as e:  # pragma: no cover
        pytest.skip(str(e))


@pytest.mark.parametrize("world", [1, 2, 3, 4, 7])
def test_shard_plan_covers_every_page_once(world):
    _lib_or_skip()
    wl = W.make("llama3_8b_bf16", seed=31, reduced=True, B=7, len_dist=("uniform", 0, 90),
                pool=200)
    P = wl.spec.page_size
    ip, vals, li = wl.indptr.numpy(), wl.values.numpy(), wl.length_info.numpy()
    ko = np.arange(wl.spec.B, dtype=np.int32) * 1000  # nonzero offsets: positions carried over
    got_pages = [[] for _ in range(wl.spec.B)]
    rows = np.zeros(wl.spec.B, np.int64)
    for r in range(world):
        sip, svals, sli, sko = _lib.cp_shard_plan(ip, vals, li, ko, P, world, r)
        for b in range(wl.spec.B):
            pg = list(svals[sip[b]:sip[b + 1]])
            n = len(pg)
            if n:
                # the chunk's first row sits at the global row where its pages start
                start = len(got_pages[b]) * P
                assert sko[b] == ko[b] + start
                assert 1 <= sli[b] <= P
                rows[b] += (n - 1) * P + sli[b]
            else:
                assert sli[b] == 0
            got_pages[b] += pg
    for b in range(wl.spec.B):
        assert got_pages[b] == list(vals[ip[b]:ip[b + 1]])  # in order, each page once
        assert rows[b] == wl.seq_len[b]


def test_shard_plan_argument_errors():
    L = _lib_or_skip()
    ip = np.array([0, 2], np.int32)
    vals = np.array([3, 4], np.int32)
    for li, world, rank in (([5], 2, 2), ([5], 0, 0), ([0], 2, 0), ([17], 2, 0)):
        with pytest.raises(_lib.PDError, match="INVALID_ARG"):
            _lib.cp_shard_plan(ip, vals, np.array(li, np.int32), None, 16, world, rank)
    assert L.pd_cp_shard_plan(None, None, None, None, 0, 16, 2, 0,
                              np.zeros(1, np.int32).ctypes.data, None, 0, None, None) == 0


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _oracle_decode(wl, ip, vals, li, ko):
    s = wl.spec
    return oracle.batch_decode_paged_kv(
        W.bits(wl.Q), W.bits(wl.pages), ip, vals if len(vals) else np.zeros(1, np.int32), li, ko,
        wl.q_rope_position.numpy(), q_dtype=s.q_dtype, kv_dtype=s.kv_dtype, H_kv=s.H_kv,
        page_size=s.page_size, rotary_mode=s.rotary_mode, rope_scale=s.rope_scale,
        rope_theta=s.rope_theta, sm_scale=wl.sm_scale)


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from paged_kv_decode_19_gb300 import cp
        wl = W.make("llama3_8b_bf16", seed=32, reduced=True, B=4, len_dist=("uniform", 0, 120),
                    pool=200)
        s = wl.spec
        ip, vals, li = wl.indptr.numpy(), wl.values.numpy(), wl.length_info.numpy()
        ko = wl.k_rope_pos_offset.numpy()
        sip, svals, sli, sko = _lib.cp_shard_plan(ip, vals, li, ko, s.page_size, world, rank)
        o, l, st = _oracle_decode(wl, sip, svals, sli, sko)
        assert st == 0
        B, H, D = s.B, s.H_qo, s.D
        packed = torch.empty(cp.packed_width(B, H, D), dtype=torch.float32)
        packed[:B * H * D] = torch.from_numpy(o.reshape(-1))
        packed[B * H * D:] = torch.from_numpy(l.reshape(-1))
        gathered = cp.exchange(packed, world)
        assert gathered.shape == (world, packed.numel())
        assert torch.equal(gathered[rank], packed)
        g = gathered.double().numpy()
        Vp = g[:, :B * H * D].reshape(world, B, H, D)
        Sp = g[:, B * H * D:].reshape(world, B, H)
        mo, ml = oracle.merge_states(Vp, Sp)
        ro, rl, _ = _oracle_decode(wl, ip, vals, li, wl.k_rope_pos_offset.numpy())
        # the partials crossed the exchange as float32: fp32 rounding of out and lse
        q.put((rank, float(np.abs(mo - ro).max()), float(np.abs(ml - rl).max())))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_two_gloo_ranks_exchange_and_combine(world):
    _lib_or_skip()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, eo, el in got:
        assert eo < 1e-6 and el < 1e-5, (rank, eo, el)
