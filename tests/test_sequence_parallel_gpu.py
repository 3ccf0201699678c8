"""Sequence-parallel decode and ring prefill through the C ABI on several ranks
(gloo, one GPU).

Two processes share the one GPU; each holds one contiguous block of a
Llama3-70B-shaped KV cache (the record's section 2.1 placement), runs
gqa_attn_decode on it, the (O, lse) states are all-gathered through host
memory over gloo, and gqa_attn_merge_states combines them (section 4).  The
ranks' kernels never wait on each other: the only exchange is the host-side
all-gather between launches.  Every rank's result is compared with the fp64
oracle over the whole cache; one sequence has no key in the second block and
one request ends exactly at the block boundary.  The ring prefill (section
5.5) rotates K/V chunks between the ranks the same way, host-side between
launches.
"""
import math
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.dirname(os.path.abspath(__file__))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    sys.path.insert(0, TESTS)
    import gqa_synth
    import oracle
    import gqa_attention_decode_gb300 as gqa
    from parity import compare
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    gqa.load_library()
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        B, H_q, H_kv, S, d = 3, 64, 8, 8192, 128
        block = S // world
        scale = 1 / math.sqrt(d)
        q, k, v, sl = gqa_synth.decode_inputs(B, H_q, H_kv, S, d, seed=93,
                                              seqlens=[8192, 3000, 4096])
        lo = rank * block
        kb = k[:, :, lo:lo + block].contiguous().to(dev)
        vb = v[:, :, lo:lo + block].contiguous().to(dev)
        o, lse = gqa.decode_sequence_parallel(q.to(dev), kb, vb, sl.to(dev), scale)
        torch.cuda.synchronize()
        o_ref, lse_ref = oracle.decode(q.float().numpy(), k.float().numpy(), v.float().numpy(),
                                       sl.numpy(), scale)
        res = compare(o, lse, o_ref, lse_ref, f"sequence-parallel decode, rank {rank}")
        assert gqa.gqa_attn_device_status() == gqa.GQA_OK
        results[rank] = res["o_max"]
    finally:
        dist.destroy_process_group()


def test_two_rank_sequence_parallel_decode_matches_oracle():
    from gqa_attention_decode_gb300 import build
    build.build()                         # once, before the ranks load the library
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        mp.start_processes(_worker, args=(2, _free_port(), results), nprocs=2,
                           start_method="spawn")
        assert sorted(results.keys()) == [0, 1]
        assert results[0] == results[1]   # both ranks merged the same gathered states


def _ring_worker(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    sys.path.insert(0, TESTS)
    import gqa_synth
    import oracle
    import gqa_attention_decode_gb300 as gqa
    from parity import compare
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    gqa.load_library()
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        B, H_q, H_kv, C, d = 1, 64, 8, 640, 128
        scale = 1 / math.sqrt(d)
        q, k, v = gqa_synth.prefill_inputs(B, H_q, H_kv, world * C, world * C, d, seed=97)
        sl = slice(rank * C, (rank + 1) * C)
        o, lse = gqa.ring_prefill_causal(q[:, :, sl].contiguous().to(dev),
                                         k[:, :, sl].contiguous().to(dev),
                                         v[:, :, sl].contiguous().to(dev), scale)
        torch.cuda.synchronize()
        # the oracle for this rank's rows: positions rank*C.., every key up to each
        o_ref, lse_ref = oracle.prefill_causal(q[:, :, sl].float().numpy(),
                                               k[:, :, :(rank + 1) * C].float().numpy(),
                                               v[:, :, :(rank + 1) * C].float().numpy(),
                                               rank * C, scale)
        res = compare(o, lse, o_ref, lse_ref, f"ring prefill, rank {rank} of {world}")
        assert gqa.gqa_attn_device_status() == gqa.GQA_OK
        results[rank] = res["o_max"]
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_ring_prefill_matches_oracle(world):
    """The record's section 5.5 ring on `world` ranks sharing the GPU: each holds a
    640-token chunk of a Llama3-70B-shaped sequence, the K/V chunks rotate over
    gloo, every rank folds the chunks at or before its own (causal on the
    diagonal, unmasked before it, later ones skipped) and merges the states."""
    from gqa_attention_decode_gb300 import build
    build.build()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        mp.start_processes(_ring_worker, args=(world, _free_port(), results), nprocs=world,
                           start_method="spawn")
        assert sorted(results.keys()) == list(range(world))
