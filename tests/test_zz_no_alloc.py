"""gqa_attn_decode_noalloc: decode for callers that cannot allocate device memory.

Such callers (code inside an allocator or memory pool that must not re-enter
it, runtimes that forbid allocation after start-up) get their split partials
written to the library's fixed static scratch instead of a workspace they
would have to allocate.  These tests call the entry point through the C ABI
and check it against the fp64 oracle and against gqa_attn_decode, with the
parity tolerances used everywhere else, on consecutive calls (the scratch
keeps the previous call's contents, which must not leak into the next
result), including the ragged batch of 16 sequences in a 128K-key cache,
whose partials fill most of the scratch.  The file sorts last so a run that
stops at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import gqa_synth
import oracle
import gqa_attention_decode_gb300 as gqa
from parity import compare, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    from gqa_attention_decode_gb300 import build
    build.build()
    gqa.load_library()
    torch.cuda.set_device(0)
    return torch.device("cuda", 0)


def _problem(dev, B, H_q, H_kv, S_max, seqlens, seed):
    q, k, v, sl = gqa_synth.decode_inputs(B, H_q, H_kv, S_max, 128, seed=seed, device=dev,
                                          seqlens=seqlens)
    return q, k, v, sl.to(dev)


def _oracle(q, k, v, sl, scale):
    """The oracle one sequence at a time, on its valid keys only."""
    B, H_q, d = q.shape
    o = np.zeros((B, H_q, d))
    lse = np.zeros((B, H_q))
    for b, n in enumerate(sl.cpu().tolist()):
        o[b:b + 1], lse[b:b + 1] = oracle.decode(
            to_f64(q[b:b + 1]), k[b:b + 1, :, :n].float().cpu().numpy(),
            v[b:b + 1, :, :n].float().cpu().numpy(), [n], scale)
    return o, lse


def test_noalloc_matches_oracle_on_consecutive_calls(dev):
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    w = gqa_synth.WORKLOADS["ragged_decode_b16"]
    rq, rk, rv, rsl = gqa_synth.workload_decode_inputs(w, dev)
    gqa_synth.fill_padding(rk, rsl, float("nan"))
    gqa_synth.fill_padding(rv, rsl, float("nan"))
    ragged_ws = gqa.gqa_attn_decode_workspace_size(w.B, w.H_q, w.H_kv, w.S_max, w.d, sms, 0)
    # the ragged batch's partials take most of the scratch (about 33 MiB of 48)
    assert gqa.GQA_NOALLOC_SCRATCH_BYTES // 2 < ragged_ws <= gqa.GQA_NOALLOC_SCRATCH_BYTES
    problems = [
        (_problem(dev, 1, 64, 8, 32768, None, 21), 0),            # one Llama3-70B layer, 32K keys
        ((rq, rk, rv, rsl.to(dev)), 0),                           # ragged batch of 16, 128K cache
        (_problem(dev, 3, 16, 2, 1000, [1, 333, 1000], 22), 7),   # ragged, 7 requested splits
        (_problem(dev, 1, 64, 8, 32768, None, 23), 0),            # back to the first shape
    ]
    for (q, k, v, sl), splits in problems:
        ref_o, ref_lse = gqa.gqa_attn_decode(q, k, v, sl, 128 ** -0.5, num_splits=splits)
        o = torch.full_like(ref_o, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        gqa.gqa_attn_decode_noalloc(q, k, v, sl, 128 ** -0.5, num_splits=splits, o=o, lse=lse)
        torch.cuda.synchronize()
        what = f"noalloc B={q.shape[0]} S_max={k.shape[2]}"
        o_ref, lse_ref = _oracle(q, k, v, sl, 128 ** -0.5)
        compare(o, lse, o_ref, lse_ref, what + " vs oracle")
        compare(o, lse, to_f64(ref_o), to_f64(ref_lse), what + " vs workspace decode")
    assert gqa.gqa_attn_device_status() == gqa.GQA_OK


def test_noalloc_rejects_problems_beyond_the_scratch(dev):
    lib = gqa.load_library()
    # 64 sequences x 64 query heads in a 128K-key cache need about 135 MB of
    # partials, more than GQA_NOALLOC_SCRATCH_BYTES: rejected before any launch
    # (the pointers are never touched).
    fake = ctypes.c_void_p(1 << 20)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.gqa_attn_decode_noalloc(fake, fake, fake, fake, 64, 64, 8, 131072, 128,
                                     128 ** -0.5, 0, fake, fake, stream)
    assert rc == gqa.GQA_ERR_WORKSPACE
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    assert gqa.gqa_attn_decode_workspace_size(64, 64, 8, 131072, 128, sms, 0) > \
        gqa.GQA_NOALLOC_SCRATCH_BYTES
