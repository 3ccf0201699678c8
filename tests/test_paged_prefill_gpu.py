"""GPU parity of causal prefill over a paged KV cache (block table), through the C ABI.

The pages are a shuffled pool built from a dense cache; unused pages and the
rows of each sequence's last page past S_kv hold NaN, which must never reach a
result.  Where the paged and the dense call run the same kernel (group sizes
that run one CTA per unit on a dense cache too, and the CTA-pair kernel when
S_kv is a multiple of 128), the paged call must equal the dense call bit for
bit; every case is compared with the oracle.
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


def to_pages(k, v, page_size, extra_pages, seed):
    """Dense [B, H_kv, S, d] -> shuffled pool [num_pages, H_kv, page_size, d] + table;
    slots past S in each sequence's last page and the extra pages hold NaN."""
    B, H_kv, S, d = k.shape
    max_pages = -(-S // page_size)
    num_pages = B * max_pages + extra_pages
    perm = torch.randperm(num_pages, generator=torch.Generator().manual_seed(seed))
    kp = torch.full((num_pages, H_kv, page_size, d), float("nan"), dtype=k.dtype, device=k.device)
    vp = torch.full_like(kp, float("nan"))
    table = torch.empty((B, max_pages), dtype=torch.int32)
    for b in range(B):
        for i in range(max_pages):
            pid = int(perm[b * max_pages + i])
            table[b, i] = pid
            lo, hi = i * page_size, min((i + 1) * page_size, S)
            kp[pid, :, :hi - lo] = k[b, :, lo:hi]
            vp[pid, :, :hi - lo] = v[b, :, lo:hi]
    return kp, vp, table.to(k.device)


@pytest.mark.parametrize("B,H_q,H_kv,T_q,S_kv,q_offset,page_size", [
    (1, 4, 2, 300, 300, 0, 128),       # G = 2, square causal, ragged last page
    (2, 6, 2, 200, 1000, 800, 256),    # G = 3, a chunk after a prefix, two sequences
    (1, 4, 4, 128, 4000, 3872, 512),   # MHA, a short chunk after a long prefix (key split)
    (1, 16, 2, 257, 700, 443, 128),    # G = 8, S_kv not a multiple of 128: one CTA per unit
    (2, 16, 2, 300, 1024, 724, 256),   # G = 8, whole key tiles: CTA pairs
    (1, 64, 8, 256, 4096, 3840, 512),  # the 70B layer's groups, a chunk after a long prefix
    (1, 8, 1, 1, 1, 0, 128),           # one query, one key
])
def test_paged_prefill_against_oracle(B, H_q, H_kv, T_q, S_kv, q_offset, page_size):
    q, k, v = gqa_synth.prefill_inputs(B, H_q, H_kv, T_q, S_kv, 128, seed=95, device=DEV)
    scale = 1 / math.sqrt(128)
    kp, vp, table = to_pages(k, v, page_size, extra_pages=2, seed=S_kv)
    o, lse = gqa.gqa_attn_prefill_causal_paged(q, kp, vp, table, S_kv, scale, q_offset)
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all()
    o_ref, lse_ref = oracle.prefill_causal(np64(q), np64(k), np64(v), q_offset, scale)
    compare(o, lse, o_ref, lse_ref, f"paged prefill {B},{H_q},{H_kv},{T_q},{S_kv},{q_offset}")
    if (H_q // H_kv) % 4 != 0 or S_kv % 128 == 0:   # the dense call runs the same kernel
        o_d, l_d = gqa.gqa_attn_prefill_causal(q, k, v, scale, q_offset)
        torch.cuda.synchronize()
        assert torch.equal(o, o_d) and torch.equal(lse, l_d)


def test_shared_prefix_pages():
    """Two sequences whose tables share their first pages (a common prompt prefix);
    each prefills its own last 200 tokens."""
    B, H_q, H_kv, S, T, ps = 2, 16, 2, 1024, 200, 256
    q, k, v = gqa_synth.prefill_inputs(B, H_q, H_kv, T, S, 128, seed=96, device=DEV)
    kp, vp, table = to_pages(k, v, ps, extra_pages=0, seed=9)
    table[1, :2] = table[0, :2]                     # sequence 1 reuses sequence 0's prefix
    o, lse = gqa.gqa_attn_prefill_causal_paged(q, kp, vp, table, S, 0.1, S - T)
    torch.cuda.synchronize()
    tcpu = table.cpu()
    k_seen = torch.stack([torch.cat([kp[int(p)] for p in tcpu[b]], dim=1) for b in range(B)])
    v_seen = torch.stack([torch.cat([vp[int(p)] for p in tcpu[b]], dim=1) for b in range(B)])
    o_ref, lse_ref = oracle.prefill_causal(np64(q), np64(k_seen), np64(v_seen), S - T, 0.1)
    compare(o, lse, o_ref, lse_ref, "shared prefix pages")


def test_page_id_outside_pool_is_reported():
    B, H_q, H_kv, T, S, ps = 2, 4, 2, 128, 512, 128
    q, k, v = gqa_synth.prefill_inputs(B, H_q, H_kv, T, S, 128, seed=97, device=DEV)
    kp, vp, table = to_pages(k, v, ps, extra_pages=0, seed=5)
    table[0, 1] = kp.shape[0] + 9                   # sequence 0, keys 128..255
    assert gqa.gqa_attn_device_status() == gqa.GQA_OK
    o, lse = gqa.gqa_attn_prefill_causal_paged(q, kp, vp, table, S, 0.1, S - T)
    torch.cuda.synchronize()
    assert gqa.gqa_attn_device_status() == gqa.GQA_ERR_INVALID_ARG
    assert torch.isfinite(o.float()).all()
    o_ref, lse_ref = oracle.prefill_causal(np64(q[1:]), np64(k[1:]), np64(v[1:]), S - T, 0.1)
    compare(o[1:], lse[1:], o_ref, lse_ref, "sequence with valid pages")


def test_rejects_pages_that_split_a_key_tile():
    q, k, v = gqa_synth.prefill_inputs(1, 4, 2, 64, 256, 128, seed=98, device=DEV)
    kp, vp, table = to_pages(k, v, 64, extra_pages=0, seed=1)
    with pytest.raises(gqa.GQAError) as e:
        gqa.gqa_attn_prefill_causal_paged(q, kp, vp, table, 256, 0.1, 192)
    assert e.value.status == gqa.GQA_ERR_UNSUPPORTED
