"""Calls on several streams at once, from several host threads, and inside
captured CUDA graphs.

The library keeps no per-call state outside the caller's buffers (the device
status word aside), so decode and prefill calls on different streams may run
concurrently, and a call sequence captured into a CUDA graph replays with the
results of eager calls.  Every result here is compared bit for bit with the
same call made alone (the kernels are deterministic), and once with the fp64
oracle.
"""
import math
import threading

import numpy as np
import pytest
import torch

import gqa_synth
import oracle
import gqa_attention_decode_gb300 as gqa
from parity import compare

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None
SCALE = 1 / math.sqrt(128)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gqa_attention_decode_gb300 import build
    build.build()
    gqa.load_library()
    torch.cuda.set_device(0)
    yield
    assert gqa.gqa_attn_device_status() == gqa.GQA_OK


def _decode_problem(seed):
    q, k, v, sl = gqa_synth.decode_inputs(2, 64, 8, 8192, 128, seed=seed, device=DEV,
                                          seqlens=[8192, 3001])
    return q, k, v, sl.to(DEV)


def _prefill_problem(seed):
    return gqa_synth.prefill_inputs(1, 64, 8, 1024, 4096, 128, seed=seed, device=DEV)


def test_concurrent_streams_match_lone_calls():
    dq, dk, dv, dsl = _decode_problem(101)
    pq, pk, pv = _prefill_problem(102)
    # alone, on the default stream
    o_d, l_d = gqa.gqa_attn_decode(dq, dk, dv, dsl, SCALE)
    o_p, l_p = gqa.gqa_attn_prefill_causal(pq, pk, pv, SCALE, 3072)
    torch.cuda.synchronize()
    # at once: decode on one stream, prefill on another, repeated so they overlap
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    torch.cuda.synchronize()
    for _ in range(4):
        with torch.cuda.stream(s1):
            outs.append(("d",) + gqa.gqa_attn_decode(dq, dk, dv, dsl, SCALE, stream=s1))
        with torch.cuda.stream(s2):
            outs.append(("p",) + gqa.gqa_attn_prefill_causal(pq, pk, pv, SCALE, 3072, stream=s2))
    torch.cuda.synchronize()
    for kind, o, l in outs:
        ref_o, ref_l = (o_d, l_d) if kind == "d" else (o_p, l_p)
        assert torch.equal(o, ref_o) and torch.equal(l, ref_l)
    o_ref, l_ref = oracle.decode(dq.float().cpu().numpy(), dk.float().cpu().numpy(),
                                 dv.float().cpu().numpy(), dsl.cpu().numpy(), SCALE)
    compare(o_d, l_d, o_ref, l_ref, "decode alone")


def test_calls_from_several_host_threads():
    problems = [_decode_problem(110 + i) for i in range(4)]
    lone = []
    for q, k, v, sl in problems:
        lone.append(gqa.gqa_attn_decode(q, k, v, sl, SCALE))
    torch.cuda.synchronize()
    results = [None] * len(problems)
    errors = []

    def work(i):
        try:
            s = torch.cuda.Stream()
            q, k, v, sl = problems[i]
            with torch.cuda.stream(s):
                for _ in range(3):
                    results[i] = gqa.gqa_attn_decode(q, k, v, sl, SCALE, stream=s)
            s.synchronize()
        except Exception as e:  # reported below, on the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(problems))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for (o, l), (o_ref, l_ref) in zip(results, lone):
        assert torch.equal(o, o_ref) and torch.equal(l, l_ref)


def test_captured_graph_replays_eager_results():
    dq, dk, dv, dsl = _decode_problem(121)
    pq, pk, pv = _prefill_problem(122)
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    ws = torch.empty(gqa.gqa_attn_decode_workspace_size(2, 64, 8, 8192, 128, sms),
                     dtype=torch.uint8, device=DEV)
    pws = torch.empty(gqa.gqa_attn_prefill_causal_workspace_size(1, 64, 8, 1024, 4096, 128,
                                                                 3072, sms),
                      dtype=torch.uint8, device=DEV)
    o = torch.empty((2, 64, 128), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((2, 64), dtype=torch.float32, device=DEV)
    po = torch.empty_like(pq)
    plse = torch.empty((1, 64, 1024), dtype=torch.float32, device=DEV)

    def calls():
        gqa.gqa_attn_decode(dq, dk, dv, dsl, SCALE, 0, o, lse, ws)
        gqa.gqa_attn_prefill_causal(pq, pk, pv, SCALE, 3072, po, plse, pws)

    calls()
    torch.cuda.synchronize()
    eager = [t.clone() for t in (o, lse, po, plse)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        calls()
    for t in (o, lse, po, plse):
        t.fill_(float("nan"))
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for got, want in zip((o, lse, po, plse), eager):
        assert torch.equal(got, want)
    # new inputs written in place are picked up by the next replay
    dq.copy_(gqa_synth.bf16_normal(tuple(dq.shape), 123, DEV))
    g.replay()
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.decode(dq.float().cpu().numpy(), dk.float().cpu().numpy(),
                                 dv.float().cpu().numpy(), dsl.cpu().numpy(), SCALE)
    compare(o, lse, o_ref, l_ref, "decode after a graph replay with new q")
