"""Decode of sequences much shorter than their cache (the device-side chunk).

The host plan knows only S_max, the cache's length; the sequence lengths live
on the device.  The split kernels and the merge derive the keys per split from
the lengths they find there, so a 4K-key sequence in a 128K-key cache is
spread over the SMs instead of over the first few splits of a plan made for
128K keys.  Every case is checked against the oracle on the keys that exist,
and the split and merge entry points called one after the other must agree
with the one-call path bit for bit (both sides derive the same chunk).
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


def oracle_on_present_keys(q, k, v, sl, scale, T_q=None):
    n = int(sl.max())
    kk, vv = np64(k[:, :, :n]), np64(v[:, :, :n])
    if T_q is None:
        return oracle.decode(np64(q), kk, vv, sl.numpy(), scale)
    return oracle.decode_multi(np64(q), kk, vv, sl.numpy(), scale)


@pytest.mark.parametrize("S_max,seqlens", [
    (131072, [4096]),                    # one sequence, 1/32 of its cache
    (65536, [4096, 100, 2048, 1]),       # a ragged batch far below its cache
    (16384, [16384, 3]),                 # one full sequence: the host's chunk
])
def test_short_sequences_in_long_cache(S_max, seqlens):
    B = len(seqlens)
    q, k, v, sl = gqa_synth.decode_inputs(B, 64, 8, S_max, 128, seed=301, device=DEV,
                                          seqlens=seqlens)
    o, lse = gqa.gqa_attn_decode(q, k, v, sl.to(DEV), 1 / math.sqrt(128))
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle_on_present_keys(q, k, v, sl, 1 / math.sqrt(128))
    compare(o, lse, o_ref, lse_ref, f"S_max={S_max} seqlens={seqlens}")


def test_split_and_merge_phases_agree_on_the_device_chunk():
    B, S_max, seqlens = 3, 65536, [5000, 64, 1300]
    q, k, v, sl = gqa_synth.decode_inputs(B, 64, 8, S_max, 128, seed=302, device=DEV,
                                          seqlens=seqlens)
    sl = sl.to(DEV)
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    o1, l1 = gqa.gqa_attn_decode(q, k, v, sl, 0.088)
    ws = torch.empty(gqa.gqa_attn_decode_workspace_size(B, 64, 8, S_max, 128, sms, 0),
                     dtype=torch.uint8, device=DEV)
    o2, l2 = torch.empty_like(o1), torch.empty_like(l1)
    gqa.gqa_attn_decode_split(q, k, v, sl, 0.088, 0, ws)
    gqa.gqa_attn_decode_merge(sl, 8, S_max, 0, o2, l2, ws)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_multi_token_tensor_cores_short_in_long_cache():
    B, T_q, S_max, seqlens = 2, 16, 65536, [3000, 700]
    q = gqa_synth.bf16_normal((B, 64, T_q, 128), 303, DEV)
    _, k, v, sl = gqa_synth.decode_inputs(B, 64, 8, S_max, 128, 304, DEV, seqlens)
    o, lse = gqa.gqa_attn_decode_multi(q, k, v, sl.to(DEV), 1 / math.sqrt(128))
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle_on_present_keys(q, k, v, sl, 1 / math.sqrt(128), T_q)
    compare(o, lse, o_ref, lse_ref, "T_q=16, short sequences in a 64K cache")


def test_paged_short_sequence_in_wide_table():
    """A block table sized for 128K keys holding a 5000-key sequence: equals the
    dense call on the same keys."""
    S_max, L, ps = 131072, 5000, 256
    q, k, v, sl = gqa_synth.decode_inputs(1, 64, 8, S_max, 128, seed=305, device=DEV,
                                          seqlens=[L])
    used = -(-L // ps)
    kp = torch.full((used + 3, 8, ps, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
    vp = torch.full_like(kp, float("nan"))
    perm = torch.randperm(used + 3, generator=torch.Generator().manual_seed(7))
    table = torch.full((1, S_max // ps), -1, dtype=torch.int32)
    for i in range(used):
        pid = int(perm[i])
        table[0, i] = pid
        n = min(ps, L - i * ps)
        kp[pid, :, :n] = k[0, :, i * ps:i * ps + n]
        vp[pid, :, :n] = v[0, :, i * ps:i * ps + n]
    o, lse = gqa.gqa_attn_decode_paged(q, kp, vp, table.to(DEV), sl.to(DEV), 0.088)
    o_d, l_d = gqa.gqa_attn_decode(q, k, v, sl.to(DEV), 0.088)
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all()
    assert torch.equal(o, o_d) and torch.equal(lse, l_d)
