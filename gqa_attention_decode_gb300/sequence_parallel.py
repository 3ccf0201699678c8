"""Decode over a KV cache sharded by sequence position across ranks.

The design record "ADR-0060: AHBM GQA Fused Attention Kernel (Llama3-70B)"
places the KV sequence in contiguous blocks, one per rank (section 2.1: rank r
holds positions [r*Bk, (r+1)*Bk), and its valid length is
clamp(seqlen - r*Bk, 0, Bk)); every rank attends over its own block, and the
per-rank states are combined by the log-sum-exp reduction of section 4.

Here each rank runs ``gqa_attn_decode`` on its block (its own GPU), the
(O, lse) states of all ranks are gathered with ``torch.distributed.all_gather``
(staged through host memory when the process group is gloo, which has no
CUDA all-gather), and ``gqa_attn_merge_states`` combines them on the GPU.  A
rank whose block holds no key of a sequence contributes lse = -inf, which the
merge treats as the identity.  This module only orders and moves tensors; all
arithmetic runs in the library's kernels.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import _binding as _b


def block_seqlens(seqlens: torch.Tensor, block: int, rank: int) -> torch.Tensor:
    """Valid keys of each sequence inside rank `rank`'s block of `block` positions:
    clamp(seqlen - rank * block, 0, block), int32 like the input."""
    if block <= 0 or rank < 0:
        raise ValueError("block must be positive and rank non-negative")
    return (seqlens.to(torch.int64) - rank * block).clamp(0, block).to(torch.int32)


def gather_states(o: torch.Tensor, lse: torch.Tensor, group=None):
    """All-gathers every rank's (O, lse) and stacks them in rank order:
    returns (o_parts [P, ...], lse_parts [P, ...]) on o's device."""
    world = dist.get_world_size(group)
    host = dist.get_backend(group) == "gloo"
    src_o = o.cpu() if host else o.contiguous()
    src_l = lse.cpu() if host else lse.contiguous()
    outs_o = [torch.empty_like(src_o) for _ in range(world)]
    outs_l = [torch.empty_like(src_l) for _ in range(world)]
    dist.all_gather(outs_o, src_o, group=group)
    dist.all_gather(outs_l, src_l, group=group)
    o_parts = torch.stack(outs_o).to(o.device)
    lse_parts = torch.stack(outs_l).to(lse.device)
    return o_parts.contiguous(), lse_parts.contiguous()


def decode_sequence_parallel(q, k_block, v_block, seqlens, scale, group=None, num_splits=0):
    """Decode (T_q = 1) of sequences whose KV cache is split across the ranks of
    `group` in contiguous blocks of k_block.shape[2] positions.

    q [B, H_q, d] bf16 (the same on every rank); k_block, v_block
    [B, H_kv, block, d] bf16, this rank's positions [rank*block, (rank+1)*block);
    seqlens [B] int32 on q's device, each sequence's total length.  Every rank
    returns the combined (O [B, H_q, d] bf16, lse [B, H_q] fp32).
    """
    rank = dist.get_rank(group)
    block = k_block.shape[2]
    local = block_seqlens(seqlens, block, rank)
    o, lse = _b.gqa_attn_decode(q, k_block, v_block, local, scale, num_splits=num_splits)
    o_parts, lse_parts = gather_states(o, lse, group)
    return _b.gqa_attn_merge_states(o_parts, lse_parts)
