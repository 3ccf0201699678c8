"""gqa_attn_decode_noalloc: decode for callers that cannot allocate device memory.

Such callers (code inside an allocator or memory pool that must not re-enter
it, runtimes that forbid allocation after start-up) get their split partials
written to the library's fixed static scratch instead of a workspace they
would have to allocate.  These tests call the entry point through the C ABI
and check it against gqa_attn_decode, with the parity tolerances used
everywhere else, on consecutive calls (the scratch keeps the previous call's
contents, which must not leak into the next result).  The file sorts last so
a run that stops at the first failure has already run every other test.
"""
import ctypes

import pytest
import torch

import gqa_synth
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


def test_noalloc_matches_workspace_decode_on_consecutive_calls(dev):
    problems = [
        (_problem(dev, 1, 64, 8, 32768, None, 21), 0),            # one Llama3-70B layer, 32K keys
        (_problem(dev, 3, 16, 2, 1000, [1, 333, 1000], 22), 7),   # ragged, 7 requested splits
        (_problem(dev, 1, 64, 8, 32768, None, 23), 0),            # back to the first shape
    ]
    for (q, k, v, sl), splits in problems:
        ref_o, ref_lse = gqa.gqa_attn_decode(q, k, v, sl, 128 ** -0.5, num_splits=splits)
        o = torch.full_like(ref_o, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        gqa.gqa_attn_decode_noalloc(q, k, v, sl, 128 ** -0.5, num_splits=splits, o=o, lse=lse)
        torch.cuda.synchronize()
        compare(o, lse, to_f64(ref_o), to_f64(ref_lse), "noalloc vs workspace decode")
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
