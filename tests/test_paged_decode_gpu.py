"""GPU parity of decode over a paged KV cache (block table), through the C ABI.

Pages are a random permutation of a dense cache's 64..1024-key slices in a pool
that also holds unused pages filled with NaN; the paged call must equal the
dense call on the same keys bit for bit (same plan) and match the oracle.
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
    """Dense [B, H_kv, S_max, d] -> shuffled pool [num_pages, H_kv, page_size, d] + table."""
    B, H_kv, S_max, d = k.shape
    assert S_max % page_size == 0
    max_pages = S_max // page_size
    num_pages = B * max_pages + extra_pages
    perm = torch.randperm(num_pages, generator=torch.Generator().manual_seed(seed))
    kp = torch.full((num_pages, H_kv, page_size, d), float("nan"), dtype=k.dtype, device=k.device)
    vp = torch.full_like(kp, float("nan"))
    table = torch.empty((B, max_pages), dtype=torch.int32)
    for b in range(B):
        for i in range(max_pages):
            pid = int(perm[b * max_pages + i])
            table[b, i] = pid
            kp[pid] = k[b, :, i * page_size:(i + 1) * page_size]
            vp[pid] = v[b, :, i * page_size:(i + 1) * page_size]
    return kp, vp, table.to(k.device)


@pytest.mark.parametrize("page_size,seqlens,num_splits", [
    (64, [1, 700, 1024], 0),
    (128, [1024, 65, 129], 0),
    (256, [1000, 1024, 3], 5),
    (1024, [1024, 1, 513], 0),
    (256, [256, 512, 1024], 100),      # two-kernel plan
])
def test_paged_equals_dense_and_oracle(page_size, seqlens, num_splits):
    B, H_q, H_kv, S_max, d = 3, 16, 2, 1024, 128
    q, k, v, sl = gqa_synth.decode_inputs(B, H_q, H_kv, S_max, d, seed=41, device=DEV,
                                          seqlens=seqlens)
    sl_dev = sl.to(DEV)
    kp, vp, table = to_pages(k, v, page_size, extra_pages=3, seed=page_size)
    o_p, l_p = gqa.gqa_attn_decode_paged(q, kp, vp, table, sl_dev, 0.088, num_splits)
    o_d, l_d = gqa.gqa_attn_decode(q, k, v, sl_dev, 0.088, num_splits)
    torch.cuda.synchronize()
    assert torch.equal(o_p, o_d) and torch.equal(l_p, l_d)
    o_ref, lse_ref = oracle.decode(np64(q), np64(k), np64(v), sl.numpy(), 0.088)
    compare(o_p, l_p, o_ref, lse_ref, f"paged {page_size}")


def test_paged_llama70b_layer():
    w = gqa_synth.WORKLOADS["llama70b_decode_32k"]
    q, k, v, sl = gqa_synth.workload_decode_inputs(w, DEV)
    kp, vp, table = to_pages(k, v, 256, extra_pages=0, seed=7)
    o_p, l_p = gqa.gqa_attn_decode_paged(q, kp, vp, table, sl.to(DEV), w.scale)
    o_d, l_d = gqa.gqa_attn_decode(q, k, v, sl.to(DEV), w.scale)
    torch.cuda.synchronize()
    assert torch.equal(o_p, o_d) and torch.equal(l_p, l_d)


def test_shared_prefix_pages():
    """Two sequences whose tables share their first pages (a common prompt prefix)."""
    H_q, H_kv, ps, d = 16, 2, 128, 128
    q, k, v, _ = gqa_synth.decode_inputs(2, H_q, H_kv, 512, d, seed=42, device=DEV)
    kp, vp, table = to_pages(k, v, ps, extra_pages=0, seed=1)
    table[1, :2] = table[0, :2]                  # sequence 1 reuses sequence 0's prefix
    sl = torch.tensor([512, 300], dtype=torch.int32)
    o, l = gqa.gqa_attn_decode_paged(q, kp, vp, table, sl.to(DEV), 0.1)
    torch.cuda.synchronize()
    # the dense view each sequence actually sees
    tcpu = table.cpu()
    k_seen = torch.stack([torch.cat([kp[int(p)] for p in tcpu[b]], dim=1) for b in range(2)])
    v_seen = torch.stack([torch.cat([vp[int(p)] for p in tcpu[b]], dim=1) for b in range(2)])
    o_ref, lse_ref = oracle.decode(np64(q), np64(k_seen), np64(v_seen), sl.numpy(), 0.1)
    compare(o, l, o_ref, lse_ref, "shared prefix")


def test_paged_rejects_bad_page_size():
    q, k, v, sl = gqa_synth.decode_inputs(1, 8, 1, 256, 128, seed=43, device=DEV)
    kp = k.view(1, 1, 256, 128).reshape(2, 1, 128, 128)[:, :, :100]
    kp = kp.contiguous()
    table = torch.zeros((1, 3), dtype=torch.int32, device=DEV)
    with pytest.raises(gqa.GQAError) as e:
        gqa.gqa_attn_decode_paged(q, kp, kp, table, sl.to(DEV), 0.1)
    assert e.value.status == gqa.GQA_ERR_UNSUPPORTED


def test_page_id_outside_pool_is_reported():
    """A block-table entry past the pool reads zeros and is reported as
    GQA_ERR_INVALID_ARG through the device status; the other sequence is exact."""
    B, H_q, H_kv, S, ps = 2, 16, 2, 512, 128
    q, k, v, sl = gqa_synth.decode_inputs(B, H_q, H_kv, S, 128, seed=44, device=DEV)
    kp, vp, table = to_pages(k, v, ps, extra_pages=0, seed=3)
    table[0, 1] = kp.shape[0] + 3                     # sequence 0, keys 128..255
    assert gqa.gqa_attn_device_status() == gqa.GQA_OK
    o, l = gqa.gqa_attn_decode_paged(q, kp, vp, table, sl.to(DEV), 0.1)
    torch.cuda.synchronize()
    assert gqa.gqa_attn_device_status() == gqa.GQA_ERR_INVALID_ARG
    tcpu = table.cpu()
    k1 = torch.stack([torch.cat([kp[int(p)] for p in tcpu[1]], dim=1)])
    v1 = torch.stack([torch.cat([vp[int(p)] for p in tcpu[1]], dim=1)])
    o_ref, lse_ref = oracle.decode(np64(q[1:]), np64(k1), np64(v1), sl.numpy()[1:], 0.1)
    compare(o[1:], l[1:], o_ref, lse_ref, "sequence with valid pages")


# ---- paged cache on the tcgen05 split kernel and with T_q new tokens ----

@pytest.mark.parametrize("H_q,H_kv,T_q,page_size,seqlens", [
    (16, 2, 1, 128, [1000, 1024, 3]),     # G = 8 < rows: warp MMAs, one token (plain paged)
    (16, 2, 4, 128, [1000, 130, 1024]),   # G * T_q = 32 rows: warp MMAs, wide variant
    (16, 2, 16, 256, [1000, 17, 768]),    # 128 rows: tcgen05 kernel
    (32, 2, 1, 128, [900, 1024, 5]),      # G = 16: tcgen05 kernel, one token
    (48, 1, 2, 512, [1024, 300, 600]),    # G = 48, 96 rows, a 2-page sequence
])
def test_paged_multi_equals_dense_and_oracle(H_q, H_kv, T_q, page_size, seqlens):
    B, S_max, d = 3, 1024, 128
    q = gqa_synth.bf16_normal((B, H_q, T_q, d), 61, DEV)
    _, k, v, sl = gqa_synth.decode_inputs(B, H_q, H_kv, S_max, d, seed=62, device=DEV,
                                          seqlens=seqlens)
    sl_dev = sl.to(DEV)
    kp, vp, table = to_pages(k, v, page_size, extra_pages=2, seed=page_size + T_q)
    o_p, l_p = gqa.gqa_attn_decode_paged_multi(q, kp, vp, table, sl_dev, 0.088)
    o_d, l_d = gqa.gqa_attn_decode_multi(q, k, v, sl_dev, 0.088)
    torch.cuda.synchronize()
    assert torch.equal(o_p, o_d) and torch.equal(l_p, l_d)
    o_ref, lse_ref = oracle.decode_multi(np64(q), np64(k), np64(v), sl.numpy(), 0.088)
    compare(o_p, l_p, o_ref, lse_ref, f"paged multi G={H_q // H_kv} T_q={T_q} ps={page_size}")
    if T_q == 1:   # the single-token entry point gives the same result
        o1, l1 = gqa.gqa_attn_decode_paged(q[:, :, 0], kp, vp, table, sl_dev, 0.088)
        torch.cuda.synchronize()
        assert torch.equal(o1, o_p[:, :, 0]) and torch.equal(l1, l_p[:, :, 0])


def test_paged_multi_llama70b_layer_16_tokens():
    """Llama3-70B layer, 32K keys in 256-key pages, 16 new tokens (tcgen05 kernel)."""
    w = gqa_synth.WORKLOADS["llama70b_decode_32k"]
    q = gqa_synth.bf16_normal((1, w.H_q, 16, w.d), 63, DEV)
    _, k, v, sl = gqa_synth.workload_decode_inputs(w, DEV)
    kp, vp, table = to_pages(k, v, 256, extra_pages=0, seed=8)
    o_p, l_p = gqa.gqa_attn_decode_paged_multi(q, kp, vp, table, sl.to(DEV), w.scale)
    o_d, l_d = gqa.gqa_attn_decode_multi(q, k, v, sl.to(DEV), w.scale)
    torch.cuda.synchronize()
    assert torch.equal(o_p, o_d) and torch.equal(l_p, l_d)


def test_paged_tensor_core_path_needs_128_key_pages():
    """The tcgen05 kernel's 128-key tiles must not straddle pages: 64-key pages are
    refused there (and still served by the warp-MMA kernel)."""
    B, H_q, H_kv, T_q, S = 1, 16, 2, 16, 256
    q = gqa_synth.bf16_normal((B, H_q, T_q, 128), 64, DEV)
    _, k, v, sl = gqa_synth.decode_inputs(B, H_q, H_kv, S, 128, seed=65, device=DEV)
    kp, vp, table = to_pages(k, v, 64, extra_pages=0, seed=2)
    with pytest.raises(gqa.GQAError) as e:
        gqa.gqa_attn_decode_paged_multi(q, kp, vp, table, sl.to(DEV), 0.1)
    assert e.value.status == gqa.GQA_ERR_UNSUPPORTED
    o, l = gqa.gqa_attn_decode_paged_multi(q[:, :, :4].contiguous(), kp, vp, table, sl.to(DEV),
                                           0.1)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.decode_multi(np64(q[:, :, :4]), np64(k), np64(v), sl.numpy(), 0.1)
    compare(o, l, o_ref, lse_ref, "64-key pages, 32 rows")


def test_page_id_outside_pool_is_reported_tensor_core_path():
    B, H_q, H_kv, T_q, S, ps = 2, 16, 2, 16, 512, 128
    q = gqa_synth.bf16_normal((B, H_q, T_q, 128), 66, DEV)
    _, k, v, sl = gqa_synth.decode_inputs(B, H_q, H_kv, S, 128, seed=67, device=DEV)
    kp, vp, table = to_pages(k, v, ps, extra_pages=0, seed=4)
    table[0, 2] = -7                                   # sequence 0, keys 256..383
    assert gqa.gqa_attn_device_status() == gqa.GQA_OK
    o, l = gqa.gqa_attn_decode_paged_multi(q, kp, vp, table, sl.to(DEV), 0.1)
    torch.cuda.synchronize()
    assert gqa.gqa_attn_device_status() == gqa.GQA_ERR_INVALID_ARG
    assert torch.isfinite(o.float()).all()
    tcpu = table.cpu()
    k1 = torch.stack([torch.cat([kp[int(p)] for p in tcpu[1]], dim=1)])
    v1 = torch.stack([torch.cat([vp[int(p)] for p in tcpu[1]], dim=1)])
    o_ref, lse_ref = oracle.decode_multi(np64(q[1:]), np64(k1), np64(v1), sl.numpy()[1:], 0.1)
    compare(o[1:], l[1:], o_ref, lse_ref, "sequence with valid pages (tensor cores)")


def test_l2_prefetch_reads_the_block_table_the_preceding_grid_writes():
    """A one-wave decode reads the block-table entries of its first tiles before
    its grid-dependency wait (an L2 prefetch hint) while the preceding grid may
    still be writing the table.  Here the preceding grid (a merge of shard
    states, which lets its dependents launch at its start) writes the table
    over one that points at NaN pages: the decode must read the new table.
    The table's int32 ids are written as the bf16 halves of one merge row
    (ids 128..191: every half is a normal bf16 or +0, copied exactly)."""
    B, H_q, H_kv, S, d, ps = 2, 64, 8, 8192, 128, 256
    splits, _ = gqa.gqa_attn_decode_plan(B, H_kv, S, torch.cuda.get_device_properties(0)
                                         .multi_processor_count)
    assert splits * H_kv * B <= torch.cuda.get_device_properties(0).multi_processor_count
    q, k, v, sl = gqa_synth.decode_inputs(B, H_q, H_kv, S, d, seed=79, device=DEV)
    q16 = gqa_synth.bf16_normal((B, H_q, 16, d), 80, DEV)
    mp = S // ps
    perm = torch.randperm(B * mp, generator=torch.Generator().manual_seed(81))
    true_table = (128 + perm).to(torch.int32).view(B, mp)
    kp = torch.full((128 + B * mp, H_kv, ps, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    vp = torch.full_like(kp, float("nan"))
    for b in range(B):
        for i in range(mp):
            kp[int(true_table[b, i])] = k[b, :, i * ps:(i + 1) * ps]
            vp[int(true_table[b, i])] = v[b, :, i * ps:(i + 1) * ps]
    parts = true_table.to(DEV).view(torch.bfloat16).reshape(1, 1, d)
    assert parts.shape[-1] == d
    lse_parts = torch.zeros((1, 1), dtype=torch.float32, device=DEV)
    table = torch.empty((B, mp), dtype=torch.int32, device=DEV)
    stale = torch.arange(B * mp, dtype=torch.int32, device=DEV).view(B, mp)   # NaN pages
    lse_out = torch.empty((1,), dtype=torch.float32, device=DEV)
    sl_d = sl.to(DEV)
    torch.cuda.synchronize()
    for _ in range(3):
        for qq in (q, q16):
            table.copy_(stale)
            gqa.gqa_attn_merge_states(parts, lse_parts, table.view(torch.bfloat16).view(1, d),
                                      lse_out)
            if qq.dim() == 3:
                o, lse = gqa.gqa_attn_decode_paged(qq, kp, vp, table, sl_d, 1 / math.sqrt(d))
            else:
                o16, lse16 = gqa.gqa_attn_decode_paged_multi(qq, kp, vp, table, sl_d,
                                                             1 / math.sqrt(d))
            torch.cuda.synchronize()
            assert torch.equal(table.cpu(), true_table)
    assert torch.isfinite(o.float()).all() and torch.isfinite(o16.float()).all()
    o_ref, lse_ref = oracle.decode(np64(q), np64(k), np64(v), sl.numpy(), 1 / math.sqrt(d))
    compare(o, lse, o_ref, lse_ref, "paged decode after a grid writing its block table")
    o_ref, lse_ref = oracle.decode_multi(np64(q16), np64(k), np64(v), sl.numpy(),
                                         1 / math.sqrt(d))
    compare(o16, lse16, o_ref, lse_ref, "paged 16-token decode after a grid writing its table")
