"""Decode and causal prefill over a sequence sharded by position across ranks.

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
merge treats as the identity.

Prefill follows the record's section 5.5 ring ("PREFILL, with SP (Ring KV)"):
the K/V blocks rotate around the ranks and each rank folds every block it
receives into its query rows, skipping blocks wholly after them.  The record
keeps one query head per rank and all query rows; here each rank holds a
contiguous chunk of the sequence -- its query rows and its K/V rows, all heads
-- so the ring also carries the sequence that does not fit one GPU.  At step
t rank r holds the K/V chunk of rank src = (r - t) mod N: the diagonal chunk
(src = r) is attended causally, chunks wholly before the query chunk
(src < r) without a mask (the causal prefill call with q_offset = (r - src) *
C puts every row past the chunk's last key), and chunks wholly after (src >
r) are skipped.  The per-step (O, lse) states are combined at the end with
``gqa_attn_merge_states``.

This module only orders and moves tensors; all arithmetic runs in the
library's kernels.
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


def ring_schedule(rank: int, world: int, chunk: int):
    """Steps of the ring for `rank`: a list of (src, q_offset) for t = 0..world-1,
    src the rank whose K/V chunk is held at step t and q_offset the position of
    the query chunk relative to that K/V chunk, or None when the chunk lies
    wholly after the query chunk (skipped)."""
    if world <= 0 or not 0 <= rank < world or chunk <= 0:
        raise ValueError("need 0 <= rank < world and a positive chunk")
    steps = []
    for t in range(world):
        src = (rank - t) % world
        steps.append((src, (rank - src) * chunk if src <= rank else None))
    return steps


def ring_pass(tensors, group=None):
    """Sends `tensors` to the next rank of the ring and returns the ones received
    from the previous rank (same shapes and dtypes), staged through host memory
    when the process group is gloo."""
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    host = dist.get_backend(group) == "gloo"

    def peer(i):
        return dist.get_global_rank(group, i) if group is not None else i
    nxt, prv = peer((rank + 1) % world), peer((rank - 1) % world)
    out_src = [t.cpu() if host else t.contiguous() for t in tensors]
    received = [torch.empty_like(t) for t in out_src]
    reqs = []
    for t_out, t_in in zip(out_src, received):
        reqs.append(dist.isend(t_out, nxt, group=group))
        reqs.append(dist.irecv(t_in, prv, group=group))
    for r in reqs:
        r.wait()
    return [r.to(t.device) for r, t in zip(received, tensors)]


def ring_prefill_causal(q, k, v, scale, group=None):
    """Causal prefill of a sequence split in equal contiguous chunks across the
    ranks of `group` (rank r holds positions [r*C, (r+1)*C)).

    q [B, H_q, C, d] bf16 (this rank's query rows); k, v [B, H_kv, C, d] bf16
    (this rank's K/V rows), all on this rank's GPU.  Returns this rank's
    (O [B, H_q, C, d] bf16, lse [B, H_q, C] fp32) of the whole causal prefill.
    """
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    chunk = q.shape[2]
    if k.shape[2] != chunk or v.shape != k.shape:
        raise ValueError("every rank holds a query chunk and a K/V chunk of the same length")
    parts_o, parts_l = [], []
    cur = [k, v]
    for t, (src, q_offset) in enumerate(ring_schedule(rank, world, chunk)):
        if q_offset is not None:
            o_t, l_t = _b.gqa_attn_prefill_causal(q, cur[0], cur[1], scale, q_offset)
            parts_o.append(o_t)
            parts_l.append(l_t)
        if t + 1 < world:
            cur = ring_pass(cur, group)
    return _b.gqa_attn_merge_states(torch.stack(parts_o), torch.stack(parts_l))
