"""Context parallelism across ranks: combine the per-shard attention states.

Each rank decodes the same query rows against one round-robin shard of the KV
(rank r holds shard r) and produces that shard's normalised (O, LSE); the shards'
states are then combined through their LSEs ("Speculative decode + DCP on
gfx1250", Problem: a decode over a round-robin context-parallel shard returns its
LSE so the shards can be merged).  The exchange is one all-gather of (O, LSE) in
rank order; the merge is ``mla_merge_states`` on the local GPU.  Plumbing only:
the arithmetic runs in the library's merge kernel.
"""
from typing import Optional, Tuple

from . import mla_merge_states


def gather_states(o_local, lse_local, group=None) -> Tuple["object", "object"]:
    """All-gather every rank's (O [rows..., dv], LSE [rows...]) for the same query
    rows: returns O [world, rows..., dv] and LSE [world, rows...], entry r from rank
    r of ``group``.  Works on any backend that all-gathers the tensors' device and
    dtype (NCCL on GPUs, gloo on host tensors)."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    o_all = o_local.new_empty((world,) + tuple(o_local.shape))
    l_all = lse_local.new_empty((world,) + tuple(lse_local.shape))
    dist.all_gather(list(o_all.unbind(0)), o_local.contiguous(), group=group)
    dist.all_gather(list(l_all.unbind(0)), lse_local.contiguous(), group=group)
    return o_all, l_all


def cp_merge(o_local, lse_local, o_out, lse_out, group=None, stream: Optional[object] = None) -> None:
    """Gather the shards' states from every rank of ``group`` and merge them into
    o_out [rows..., dv] (bf16 or fp32) and lse_out [rows...] (fp32) on this rank's
    GPU.  Every rank ends with the same merged result."""
    o_all, l_all = gather_states(o_local, lse_local, group)
    world = o_all.shape[0]
    dv = o_local.shape[-1]
    rows = lse_local.numel()
    mla_merge_states(o_all.view(world, rows, dv), l_all.view(world, rows), o_out.view(rows, dv),
                     lse_out.view(rows), stream)
