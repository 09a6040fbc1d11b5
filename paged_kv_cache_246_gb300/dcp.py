"""Decode context parallelism across processes: the exchange step.

Each rank of a decode context parallel group holds every sequence's tokens
j with j % world == rank (backends.utils CommonAttentionMetadata
dcp_local_seq_lens are the local lengths).  A decode is three steps: every
rank computes its share over its own keys (paged_attn_decode_dcp_partial),
the shares are all-gathered rank-major, and every rank merges them
(paged_attn_dcp_combine).  This module is the middle step and the
composition; the arithmetic is in the library's kernels.
"""
from __future__ import annotations

from typing import Optional

import torch
import torch.distributed as dist

from . import binding as B


def gather_shares(part_o: torch.Tensor, part_ml: torch.Tensor, group=None):
    """All-gather one share per rank, stacked rank-major: returns
    ([world, *part_o.shape], [world, *part_ml.shape])."""
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    if world == 1:
        return part_o.unsqueeze(0), part_ml.unsqueeze(0)
    outs_o = [torch.empty_like(part_o) for _ in range(world)]
    outs_ml = [torch.empty_like(part_ml) for _ in range(world)]
    dist.all_gather(outs_o, part_o.contiguous(), group=group)
    dist.all_gather(outs_ml, part_ml.contiguous(), group=group)
    return torch.stack(outs_o), torch.stack(outs_ml)


def dcp_decode(out: torch.Tensor, query: torch.Tensor, kv_cache: torch.Tensor,
               block_tables: torch.Tensor, seq_lens: torch.Tensor, query_len: int,
               max_seq_len: int, params: B.AttnParams, group=None,
               workspace: Optional[torch.Tensor] = None) -> None:
    """This rank's decode of a batch whose tokens are spread over the group:
    out [num_seqs * query_len, heads * head_size] on every rank.  kv_cache /
    block_tables are the rank's own; seq_lens are global."""
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    rank = dist.get_rank(group) if dist.is_initialized() else 0
    rows = seq_lens.numel() * int(query_len)
    part_o = torch.empty((rows * params.num_heads, params.head_size), dtype=torch.float32,
                         device=query.device)
    part_ml = torch.empty((rows * params.num_heads, 2), dtype=torch.float32,
                          device=query.device)
    B.paged_attn_decode_dcp_partial(part_o, part_ml, query, kv_cache, block_tables, seq_lens,
                                    query_len, max_seq_len, world, rank, params, workspace)
    parts_o, parts_ml = gather_shares(part_o, part_ml, group)
    B.paged_attn_dcp_combine(out, parts_o, parts_ml, params)
