"""GPU parity of the combination of attention states over key shards
(gqa_attn_merge_states), through the C ABI.

Decode over disjoint key shards of a cache, each shard a call of its own, then
merged, must equal the oracle's attention over all keys (the record's
section 4 reduction); random shard states are compared with the oracle's
merge_states.
"""
import math

import numpy as np
import pytest
import torch

import gqa_synth
import oracle
import gqa_attention_decode_gb300 as gqa
from parity import compare

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gqa_attention_decode_gb300 import build
    build.build()
    gqa.load_library()
    torch.cuda.set_device(0)
    yield
    assert gqa.gqa_attn_device_status() == gqa.GQA_OK


def np64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("bounds,seqlens", [
    ([0, 1024, 2600, 4096], [4096, 1500]),   # sequence 1 sees nothing of the last shard
    ([0, 64, 4096], [4096, 64]),            # a one-tile shard; sequence 1 only the first
    ([0, 2048, 2048, 4096], [3000, 2049]),  # an empty shard (no keys at all)
])
def test_sharded_decode_equals_unsplit(bounds, seqlens):
    """Llama3-70B heads: decode over each key shard, merged, against the oracle over
    all keys of each sequence."""
    B, H_q, H_kv, S, d = 2, 64, 8, 4096, 128
    q, k, v, sl = gqa_synth.decode_inputs(B, H_q, H_kv, S, d, seed=81, device=DEV,
                                          seqlens=seqlens)
    scale = 1 / math.sqrt(d)
    o_parts, lse_parts = [], []
    for lo, hi in zip(bounds[:-1], bounds[1:]):
        width = max(hi - lo, 64)                       # a shard cache holds at least one tile
        ks = torch.zeros((B, H_kv, width, d), dtype=k.dtype, device=DEV)
        vs = torch.zeros_like(ks)
        ks[:, :, :hi - lo] = k[:, :, lo:hi]
        vs[:, :, :hi - lo] = v[:, :, lo:hi]
        sl_i = (sl - lo).clamp(0, hi - lo).to(torch.int32)
        o_i, l_i = gqa.gqa_attn_decode(q, ks, vs, sl_i.to(DEV), scale)
        o_parts.append(o_i)
        lse_parts.append(l_i)
    o, lse = gqa.gqa_attn_merge_states(torch.stack(o_parts), torch.stack(lse_parts))
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.decode(np64(q), np64(k), np64(v), sl.numpy(), scale)
    compare(o, lse, o_ref, lse_ref, f"sharded decode {bounds}")


def test_random_states_against_oracle_merge():
    """Random bf16 states with empty shards (lse = -inf) and rows empty in every
    shard."""
    g = torch.Generator(device="cpu").manual_seed(82)
    P, rows, d = 5, 1000, 128
    o_parts = torch.randn((P, rows, d), generator=g).to(torch.bfloat16)
    lse_parts = (torch.randn((P, rows), generator=g) * 6.0).float()
    lse_parts[1, ::3] = float("-inf")
    lse_parts[:, 7] = float("-inf")                   # row 7: nothing visible anywhere
    o, lse = gqa.gqa_attn_merge_states(o_parts.to(DEV), lse_parts.to(DEV))
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.merge_states(np64(o_parts), np64(lse_parts))
    err = np.abs(np64(o) - o_ref)
    assert err.max() <= 2.0 ** -7 * max(1.0, np.abs(o_ref).max())   # bf16 rounding of O
    fin = np.isfinite(lse_ref)
    assert np.abs(lse.cpu().numpy()[fin] - lse_ref[fin]).max() <= 1e-5
    assert lse[7].item() == float("-inf") and torch.all(o[7] == 0)


def test_single_shard_is_identity():
    g = torch.Generator(device="cpu").manual_seed(83)
    o_parts = torch.randn((1, 300, 128), generator=g).to(torch.bfloat16).to(DEV)
    lse_parts = torch.randn((1, 300), generator=g).float().to(DEV)
    o, lse = gqa.gqa_attn_merge_states(o_parts, lse_parts)
    torch.cuda.synchronize()
    assert torch.equal(o, o_parts[0]) and torch.equal(lse, lse_parts[0])


def test_rejects_bad_arguments():
    o_parts = torch.zeros((2, 4, 64), dtype=torch.bfloat16, device=DEV)
    lse_parts = torch.zeros((2, 4), dtype=torch.float32, device=DEV)
    with pytest.raises(gqa.GQAError) as e:
        gqa.gqa_attn_merge_states(o_parts, lse_parts)      # d = 64
    assert e.value.status == gqa.GQA_ERR_UNSUPPORTED
