"""Sequence-parallel decode and ring prefill across ranks: the host side on CPU
ranks (gloo, 2 and 3).

The record's section 2.1 places the KV sequence in contiguous per-rank blocks
and section 4 combines the per-rank (O, lse) states.  Here two CPU processes
each take one block of a cache, compute their block's state with the oracle,
exchange the states with the package's ``gather_states`` (the all-gather the
GPU path uses), and merge them with the oracle's merge_states; the result
must equal the oracle's decode over the whole cache.  One sequence has no key
in the second block (its state there is lse = -inf).  The ring prefill of
section 5.5 is run the same way: the K/V chunks travel around three ranks
with the package's ring_pass and the oracle computes every step.
"""
import os
import socket
import sys

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_block_seqlens_clamps_to_each_block():
    sys.path.insert(0, ROOT)
    from gqa_attention_decode_gb300 import block_seqlens
    sl = torch.tensor([4096, 1500, 0, 2048, 2049], dtype=torch.int32)
    assert block_seqlens(sl, 2048, 0).tolist() == [2048, 1500, 0, 2048, 2048]
    assert block_seqlens(sl, 2048, 1).tolist() == [2048, 0, 0, 0, 1]
    assert block_seqlens(sl, 2048, 2).tolist() == [0, 0, 0, 0, 0]
    assert block_seqlens(sl, 2048, 1).dtype == torch.int32


def _worker(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import gqa_synth
    import oracle
    from gqa_attention_decode_gb300 import block_seqlens, gather_states
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        B, H_q, H_kv, S, d = 3, 16, 2, 600, 128
        block = S // world
        q, k, v, sl = gqa_synth.decode_inputs(B, H_q, H_kv, S, d, seed=91,
                                              seqlens=[600, 250, 301])
        lo = rank * block
        local = block_seqlens(sl, block, rank)
        o_i, l_i = oracle.decode(q.float().numpy(), k[:, :, lo:lo + block].float().numpy(),
                                 v[:, :, lo:lo + block].float().numpy(), local.numpy(), 0.1)
        o_parts, l_parts = gather_states(torch.from_numpy(o_i), torch.from_numpy(l_i))
        assert o_parts.shape == (world, B, H_q, d) and l_parts.shape == (world, B, H_q)
        o, lse = oracle.merge_states(o_parts.numpy(), l_parts.numpy())
        o_ref, lse_ref = oracle.decode(q.float().numpy(), k.float().numpy(), v.float().numpy(),
                                       sl.numpy(), 0.1)
        results[rank] = (float(np.abs(o - o_ref).max()), float(np.abs(lse - lse_ref).max()),
                         bool(np.isneginf(l_parts[1, 1].numpy()).all()))
    finally:
        dist.destroy_process_group()


def test_gathered_block_states_merge_to_the_whole_decode():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        mp.start_processes(_worker, args=(2, _free_port(), results), nprocs=2,
                           start_method="spawn")
        for rank in (0, 1):
            o_err, l_err, empty_is_neg_inf = results[rank]
            assert o_err < 1e-12 and l_err < 1e-12
            assert empty_is_neg_inf        # sequence 1 has no key in block 1


def test_ring_schedule_skips_future_chunks():
    sys.path.insert(0, ROOT)
    from gqa_attention_decode_gb300 import ring_schedule
    assert ring_schedule(0, 3, 8) == [(0, 0), (2, None), (1, None)]
    assert ring_schedule(2, 3, 8) == [(2, 0), (1, 8), (0, 16)]
    assert ring_schedule(1, 4, 5) == [(1, 0), (0, 5), (3, None), (2, None)]
    # every rank visits every chunk once and computes exactly the chunks at or before its own
    for world in (1, 2, 5):
        for rank in range(world):
            steps = ring_schedule(rank, world, 7)
            assert sorted(s for s, _ in steps) == list(range(world))
            assert [s for s, off in steps if off is not None] == list(range(rank, -1, -1))


def _ring_worker(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import gqa_synth
    import oracle
    from gqa_attention_decode_gb300 import ring_pass, ring_schedule
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        B, H_q, H_kv, C, d = 1, 8, 2, 40, 128
        q, k, v = gqa_synth.prefill_inputs(B, H_q, H_kv, world * C, world * C, d, seed=95)
        sl = slice(rank * C, (rank + 1) * C)
        qc, cur = q[:, :, sl], [k[:, :, sl].contiguous(), v[:, :, sl].contiguous()]
        parts_o, parts_l, seen = [], [], []
        for t, (src, q_off) in enumerate(ring_schedule(rank, world, C)):
            # the chunk held now is rank src's: the ring delivered the right rows
            assert torch.equal(cur[0], k[:, :, src * C:(src + 1) * C])
            seen.append(src)
            if q_off is not None:
                po, pl = oracle.prefill_causal(qc.float().numpy(), cur[0].float().numpy(),
                                               cur[1].float().numpy(), q_off, 0.1)
                parts_o.append(po.reshape(-1, d))
                parts_l.append(pl.reshape(-1))
            if t + 1 < world:
                cur = ring_pass(cur)
        o, lse = oracle.merge_states(np.stack(parts_o), np.stack(parts_l))
        o_ref, lse_ref = oracle.prefill_causal(q.float().numpy(), k.float().numpy(),
                                               v.float().numpy(), 0, 0.1)
        results[rank] = (float(np.abs(o.reshape(B, H_q, C, d) - o_ref[:, :, sl]).max()),
                         float(np.abs(lse.reshape(B, H_q, C) - lse_ref[:, :, sl]).max()), seen)
    finally:
        dist.destroy_process_group()


def test_ring_prefill_steps_merge_to_the_causal_prefill():
    """Three CPU ranks pass their K/V chunks around the ring; each folds the
    chunks at or before its query chunk (oracle attention per step, log-sum-exp
    merge) and must get its rows of the whole causal prefill."""
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        mp.start_processes(_ring_worker, args=(3, _free_port(), results), nprocs=3,
                           start_method="spawn")
        for rank in range(3):
            o_err, l_err, seen = results[rank]
            assert o_err < 1e-12 and l_err < 1e-12
            assert seen == [(rank - t) % 3 for t in range(3)]
