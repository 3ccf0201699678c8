"""GPU parity of multi-token decode (T_q new tokens per sequence) against the oracle.

Token t of sequence b sits at position seqlens[b] - T_q + t and sees keys up to
it; the G * T_q (head, token) rows of one KV head share one pass over K and V.
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


def inputs(B, H_q, H_kv, T_q, S_max, seqlens, seed):
    q = gqa_synth.bf16_normal((B, H_q, T_q, 128), seed, DEV)
    _, k, v, sl = gqa_synth.decode_inputs(B, H_q, H_kv, S_max, 128, seed + 1, DEV, seqlens)
    return q, k, v, sl


@pytest.mark.parametrize("H_q,H_kv,T_q", [(64, 8, 2), (64, 8, 3), (64, 8, 4), (16, 4, 3),
                                          (16, 4, 8), (8, 8, 5), (12, 3, 2)])
@pytest.mark.parametrize("num_splits", [0, 7])
def test_multi_token_decode(H_q, H_kv, T_q, num_splits):
    seqlens = [2000, 1, 700, 3]              # sequences shorter than T_q included
    q, k, v, sl = inputs(4, H_q, H_kv, T_q, 2000, seqlens, 51)
    o, lse = gqa.gqa_attn_decode_multi(q, k, v, sl.to(DEV), 1 / math.sqrt(128), num_splits)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.decode_multi(np64(q), np64(k), np64(v), sl.numpy(),
                                         1 / math.sqrt(128))
    compare(o, lse, o_ref, lse_ref, f"T_q={T_q} G={H_q // H_kv} splits={num_splits}")


def test_single_token_equals_decode():
    q, k, v, sl = inputs(2, 64, 8, 1, 1500, [1500, 333], 52)
    o1, l1 = gqa.gqa_attn_decode_multi(q, k, v, sl.to(DEV), 0.088)
    o2, l2 = gqa.gqa_attn_decode(q[:, :, 0].contiguous(), k, v, sl.to(DEV), 0.088)
    torch.cuda.synchronize()
    assert torch.equal(o1[:, :, 0], o2) and torch.equal(l1[:, :, 0], l2)


def test_llama70b_layer_four_tokens():
    w = gqa_synth.WORKLOADS["llama70b_decode_32k"]
    q, k, v, sl = inputs(1, 64, 8, 4, w.S_max, None, 53)
    o, lse = gqa.gqa_attn_decode_multi(q, k, v, sl.to(DEV), w.scale)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.decode_multi(np64(q), np64(k), np64(v), sl.numpy(), w.scale)
    compare(o, lse, o_ref, lse_ref, "llama70b T_q=4")


def test_nan_padding_multi():
    q, k, v, sl = inputs(2, 32, 8, 4, 640, [577, 100], 54)
    o_ref, l_ref = gqa.gqa_attn_decode_multi(q, k, v, sl.to(DEV), 0.1)
    gqa_synth.fill_padding(k, sl, float("nan"))
    gqa_synth.fill_padding(v, sl, float("nan"))
    o, l = gqa.gqa_attn_decode_multi(q, k, v, sl.to(DEV), 0.1)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(l, l_ref)


def test_too_many_rows_is_unsupported():
    q, k, v, sl = inputs(1, 64, 8, 17, 256, None, 55)         # G * T_q = 136 > 128
    with pytest.raises(gqa.GQAError) as e:
        gqa.gqa_attn_decode_multi(q, k, v, sl.to(DEV), 0.1)
    assert e.value.status == gqa.GQA_ERR_UNSUPPORTED


# ---- more than 32 rows per KV head: the tcgen05 split kernel (128-row tiles) ----

@pytest.mark.parametrize("H_q,H_kv,T_q", [(64, 8, 5), (64, 8, 8), (64, 8, 16), (32, 2, 8),
                                          (96, 8, 10), (48, 1, 2)])
@pytest.mark.parametrize("num_splits", [0, 3])
def test_multi_token_decode_tensor_cores(H_q, H_kv, T_q, num_splits):
    # short sequences (fewer keys than tokens), a tile-exact one, and ragged tails
    seqlens = [2000, 1, 700, 3, 256, 129]
    q, k, v, sl = inputs(6, H_q, H_kv, T_q, 2000, seqlens, 56)
    o, lse = gqa.gqa_attn_decode_multi(q, k, v, sl.to(DEV), 1 / math.sqrt(128), num_splits)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.decode_multi(np64(q), np64(k), np64(v), sl.numpy(),
                                         1 / math.sqrt(128))
    compare(o, lse, o_ref, lse_ref, f"tc T_q={T_q} G={H_q // H_kv} splits={num_splits}")


def test_group_of_16_decode_uses_tensor_cores():
    """gqa_attn_decode with G = 16 (> 8): the tensor-core split kernel."""
    B, H_q, H_kv, S = 3, 64, 4, 1500
    q, k, v, sl = gqa_synth.decode_inputs(B, H_q, H_kv, S, 128, seed=57, device=DEV,
                                          seqlens=[1500, 77, 640])
    o, lse = gqa.gqa_attn_decode(q, k, v, sl.to(DEV), 0.088)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.decode(np64(q), np64(k), np64(v), sl.numpy(), 0.088)
    compare(o, lse, o_ref, lse_ref, "decode G=16")
    assert gqa.gqa_attn_decode_kernel_count(B, H_q, H_kv, S, 128, 0) == 2


def test_llama70b_layer_sixteen_tokens():
    w = gqa_synth.WORKLOADS["llama70b_decode_32k"]
    q, k, v, sl = inputs(1, 64, 8, 16, w.S_max, None, 58)
    o, lse = gqa.gqa_attn_decode_multi(q, k, v, sl.to(DEV), w.scale)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.decode_multi(np64(q), np64(k), np64(v), sl.numpy(), w.scale)
    compare(o, lse, o_ref, lse_ref, "llama70b T_q=16")


def test_nan_padding_tensor_cores():
    """Cache rows past each sequence hold NaN; the V rows of the last tile past
    the sequence are cleared before P V, so nothing changes."""
    q, k, v, sl = inputs(2, 64, 8, 8, 640, [577, 100], 59)
    o_ref, l_ref = gqa.gqa_attn_decode_multi(q, k, v, sl.to(DEV), 0.1)
    gqa_synth.fill_padding(k, sl, float("nan"))
    gqa_synth.fill_padding(v, sl, float("nan"))
    o, l = gqa.gqa_attn_decode_multi(q, k, v, sl.to(DEV), 0.1)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(l, l_ref)


@pytest.mark.parametrize("num_splits", [2, 3, 5, 7, 9, 16])
@pytest.mark.parametrize("G,T_q", [(1, 1), (3, 1), (5, 1), (8, 1), (2, 3), (4, 2)])
def test_cluster_merge_sizes(num_splits, G, T_q):
    """The single-kernel path: each CTA of a cluster of num_splits sends every
    column's partial to the CTA that finalises it (column n to CTA n mod
    num_splits); clusters of 2-16 CTAs against 1-8 (head, token) columns, with a
    sequence that leaves splits empty and one with no keys."""
    H_kv = 2
    S_max = 128 * num_splits
    seqlens = [S_max, S_max // 3 + 1, 0]
    q, k, v, sl = inputs(3, G * H_kv, H_kv, T_q, S_max, seqlens, 60 + num_splits)
    count = gqa.gqa_attn_decode_kernel_count(3, G * H_kv, H_kv, S_max, 128, num_splits)
    if num_splits <= 8:  # portable cluster sizes: always the single kernel
        assert count == 1
    o, lse = gqa.gqa_attn_decode_multi(q, k, v, sl.to(DEV), 1 / math.sqrt(128), num_splits)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.decode_multi(np64(q), np64(k), np64(v), sl.numpy(), 1 / math.sqrt(128))
    compare(o, lse, o_ref, lse_ref, f"cluster of {num_splits}, G={G}, T_q={T_q} ({count} kernel)")


def test_one_split_multi_token_writes_output_directly():
    """T_q = 3 new tokens (24 columns per KV head: two column groups) with one
    split per (sequence, KV head): written by the split kernel itself."""
    B, S = 64, 512
    rng = np.random.default_rng(5)
    seqlens = [0, 2, S] + [int(x) for x in rng.integers(0, S + 1, B - 3)]
    q, k, v, sl = inputs(B, 64, 8, 3, S, seqlens, 70)
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    assert gqa.gqa_attn_decode_plan(B, 8, S, sms, 0)[0] == 1
    o, lse = gqa.gqa_attn_decode_multi(q, k, v, sl.to(DEV), 1 / math.sqrt(128), 0)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.decode_multi(np64(q), np64(k), np64(v), sl.numpy(), 1 / math.sqrt(128))
    compare(o, lse, o_ref, lse_ref, "one split, T_q=3, B=64")


def test_one_split_tensor_core_decode_writes_output_directly():
    """16 new tokens (128 rows per KV head: the tcgen05 kernel) for a batch of
    32 sequences with one split each: the kernel writes o and lse itself; an
    empty sequence and ones shorter than T_q included."""
    B, S, T_q = 32, 1024, 16
    rng = np.random.default_rng(9)
    seqlens = [0, 3, S, 16] + [int(x) for x in rng.integers(0, S + 1, B - 4)]
    q, k, v, sl = inputs(B, 64, 8, T_q, S, seqlens, 80)
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    assert gqa.gqa_attn_decode_plan(B, 8, S, sms, 0)[0] == 1
    o, lse = gqa.gqa_attn_decode_multi(q, k, v, sl.to(DEV), 1 / math.sqrt(128), 0)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.decode_multi(np64(q), np64(k), np64(v), sl.numpy(), 1 / math.sqrt(128))
    compare(o, lse, o_ref, lse_ref, "one split, tcgen05, T_q=16, B=32")


@pytest.mark.parametrize("B,S,T_q", [(12, 4096, 16), (10, 2500, 9)])
def test_tensor_core_plan_of_one_split(B, S, T_q):
    """Batches whose (sequence, KV head) units fill half to all of the SMs, with
    caches past one wave's chunk limit: the tcgen05 path plans one split and
    writes o and lse itself (ragged lengths, an empty sequence)."""
    rng = np.random.default_rng(B)
    seqlens = [0, S] + [int(x) for x in rng.integers(1, S + 1, B - 2)]
    q, k, v, sl = inputs(B, 64, 8, T_q, S, seqlens, 90)
    o, lse = gqa.gqa_attn_decode_multi(q, k, v, sl.to(DEV), 1 / math.sqrt(128), 0)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.decode_multi(np64(q), np64(k), np64(v), sl.numpy(), 1 / math.sqrt(128))
    compare(o, lse, o_ref, lse_ref, f"tcgen05 one-split plan B={B} S={S} T_q={T_q}")
