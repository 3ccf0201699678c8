"""Seeded random decode shapes across the kernel dispatch space, against the oracle.

Each case draws a group size G (1..128), KV heads, batch, new tokens T_q (with
G * T_q within the 128-row limit), cache capacity, ragged sequence lengths
(including 0 and lengths shorter than T_q), a split count (automatic or
forced) and a cache layout (dense, or paged with a page size the chosen path
accepts).  Together they reach the warp-MMA split kernel (one and two
n-tiles), the single-kernel cluster merge, the tcgen05 split kernel, the
paged variants of both, and the split + merge path with many splits.
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


def _cases(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        G = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 12, 16, 24, 32, 64, 128]))
        H_kv = int(rng.choice([1, 2, 3])) if G <= 32 else 1
        max_tq = max(1, min(16, 128 // G))
        T_q = int(rng.integers(1, max_tq + 1))
        B = int(rng.integers(1, 4))
        paged = bool(rng.integers(0, 2))
        tensor_cores = G > 8 or G * T_q > 32
        page = int(rng.choice([128, 256])) if (paged and tensor_cores) else int(rng.choice([64, 128, 256]))
        S_max = page * int(rng.integers(1, 13))
        seqlens = [int(x) for x in rng.integers(0, S_max + 1, B)]
        seqlens[0] = S_max                             # one full sequence
        if B > 1:
            seqlens[1] = int(rng.integers(0, T_q + 1))  # fewer keys than new tokens
        splits = int(rng.choice([0, 0, 1, 3, 40]))
        out.append((G, H_kv, T_q, B, S_max, tuple(seqlens), splits, page if paged else 0))
    return out


@pytest.mark.parametrize("G,H_kv,T_q,B,S_max,seqlens,splits,page", _cases(24, 2026))
def test_random_decode_shapes(G, H_kv, T_q, B, S_max, seqlens, splits, page):
    H_q = G * H_kv
    scale = 1 / math.sqrt(128)
    q = gqa_synth.bf16_normal((B, H_q, T_q, 128), 91, DEV)
    _, k, v, sl = gqa_synth.decode_inputs(B, H_q, H_kv, S_max, 128, 92, DEV, list(seqlens))
    gqa_synth.fill_padding(k, sl, float("nan"))       # cache rows past each length: never read
    gqa_synth.fill_padding(v, sl, float("nan"))
    sld = sl.to(DEV)
    if page:
        mp = S_max // page
        kp = k.view(B, H_kv, mp, page, 128).permute(0, 2, 1, 3, 4).reshape(B * mp, H_kv, page, 128)
        vp = v.view(B, H_kv, mp, page, 128).permute(0, 2, 1, 3, 4).reshape(B * mp, H_kv, page, 128)
        perm = torch.randperm(B * mp, generator=torch.Generator().manual_seed(93))
        inv = torch.argsort(perm)
        kp, vp = kp[perm].contiguous(), vp[perm].contiguous()   # pool order shuffled
        table = inv.view(B, mp).to(torch.int32).to(DEV)
        o, lse = gqa.gqa_attn_decode_paged_multi(q, kp, vp, table, sld, scale, splits)
    else:
        o, lse = gqa.gqa_attn_decode_multi(q, k, v, sld, scale, splits)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.decode_multi(np64(q), np64(k), np64(v), sl.numpy(), scale)
    compare(o, lse, o_ref, lse_ref,
            f"G={G} H_kv={H_kv} T_q={T_q} B={B} S={S_max} splits={splits} page={page}")
