"""Context-parallel decode: each sequence's context split across ranks.

Each of `world` ranks holds a page-aligned slice of every sequence's context
(``pd_cp_shard_plan``; the NKI Attention Block TKG reference's ``CP``: each rank holds
an S_ctx/CP slice of the prior KV cache).  A rank decodes its slice with
``pd_batch_decode_paged_kv`` into a float32 partial (out, lse), packed in one buffer
``[B*H_qo*D outputs | B*H_qo lse]``.  The ranks all-gather the packed partials, the one
exchange of the path (``B*H_qo*(D+1)`` floats per rank; the KV cache never moves), and
every rank combines the ``world`` partials with ``pd_merge_states`` (the merge formula of
TVM ``merge_state_inplace`` over all partners at once).  The result equals the unsplit
decode.

Everything here is argument marshalling: the shard plan, the decode and the merge run
in libpageddecode, the exchange in ``torch.distributed`` (NCCL between GPUs).
"""
from __future__ import annotations

import dataclasses

import torch

from . import _lib


@dataclasses.dataclass
class Shard:
    """One rank's slice of the context, as device int32 tensors."""
    indptr: torch.Tensor
    values: torch.Tensor
    length_info: torch.Tensor
    k_rope_pos_offset: torch.Tensor
    world: int
    rank: int


def shard(indptr, values, length_info, k_rope_pos_offset, page_size: int, world: int, rank: int,
          device) -> Shard:
    """Rank `rank`'s page-aligned slice (pd_cp_shard_plan on the host copies of the page
    table), moved to `device`."""
    host = lambda t: None if t is None else (t.cpu().numpy() if torch.is_tensor(t) else t)
    ip, vals, li, ko = _lib.cp_shard_plan(host(indptr), host(values), host(length_info),
                                          host(k_rope_pos_offset), page_size, world, rank)
    t = lambda a: torch.from_numpy(a).to(device)
    if len(vals) == 0:  # the decode reads no entry; keep a valid pointer
        vals = ip[:1].copy()
    return Shard(t(ip), t(vals), t(li), t(ko), world, rank)


def packed_width(B: int, H_qo: int, D: int) -> int:
    return B * H_qo * (D + 1)


def decode_partial(Q, pages, sh: Shard, q_rope_position, packed: torch.Tensor, rotary_mode=0,
                   rope_scale=1.0, rope_theta=1e4, sm_scale=None, **kw):
    """Decode this rank's slice into `packed` (float32 [B*H_qo*(D+1)]): the partial output
    [B, H_qo, D] followed by its lse [B, H_qo]."""
    B, H_qo, D = Q.shape
    n = B * H_qo * D
    if packed.dtype != torch.float32 or packed.numel() != packed_width(B, H_qo, D):
        raise ValueError("packed must be float32 [B*H_qo*(D+1)]")
    out = packed[:n].view(B, H_qo, D)
    lse = packed[n:].view(B, H_qo)
    _lib.batch_decode_paged_kv(Q, pages, sh.indptr, sh.values, sh.length_info,
                               sh.k_rope_pos_offset, q_rope_position, out, lse, rotary_mode,
                               rope_scale, rope_theta, sm_scale, **kw)
    return packed


def exchange(packed: torch.Tensor, world: int, group=None) -> torch.Tensor:
    """All-gather of every rank's packed partial: returns [world, width] (row r = rank r's)."""
    if world == 1:
        return packed.view(1, -1)
    import torch.distributed as dist
    gathered = torch.empty((world, packed.numel()), dtype=packed.dtype, device=packed.device)
    if dist.get_backend(group) == "nccl":
        dist.all_gather_into_tensor(gathered.view(-1), packed, group=group)
    else:
        dist.all_gather(list(gathered.unbind(0)), packed, group=group)
    return gathered


def combine(gathered: torch.Tensor, out: torch.Tensor, lse: torch.Tensor, stream=None):
    """pd_merge_states over the gathered packed partials into out [B,H_qo,D], lse [B,H_qo]."""
    return _lib.merge_states_packed(out, lse, gathered, stream=stream)


def context_parallel_decode(Q, pages, sh: Shard, q_rope_position, out, lse, rotary_mode=0,
                            rope_scale=1.0, rope_theta=1e4, sm_scale=None, group=None, **kw):
    """The whole step on this rank: decode the slice, exchange, combine into out / lse."""
    B, H_qo, D = Q.shape
    packed = torch.empty(packed_width(B, H_qo, D), dtype=torch.float32, device=Q.device)
    decode_partial(Q, pages, sh, q_rope_position, packed, rotary_mode, rope_scale, rope_theta,
                   sm_scale, **kw)
    gathered = exchange(packed, sh.world, group)
    return combine(gathered, out, lse)
