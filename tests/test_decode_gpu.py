"""GPU parity of split-KV GQA decode against the fp64 oracle, through the C ABI.

Covers the three decode workloads (tiny, one Llama3-70B layer at 32K, the
ragged batch of 16 in a 128K cache), each compared in full, and
edge cases: ragged tails, seqlen 0 and 1, more splits than keys, G < 8, MHA,
NaN in the padding, scale 0 and negative, determinism, host buffers.
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


def run_decode(q, k, v, seqlens, scale, num_splits=0):
    o, lse = gqa.gqa_attn_decode(q, k, v, seqlens.to(DEV), scale, num_splits=num_splits)
    torch.cuda.synchronize()
    return o, lse


def check_full(q, k, v, seqlens, scale, num_splits=0, what=""):
    o, lse = run_decode(q, k, v, seqlens, scale, num_splits)
    o_ref, lse_ref = oracle.decode(np64(q), np64(k), np64(v), seqlens.cpu().numpy(), scale)
    return compare(o, lse, o_ref, lse_ref, what)


def test_tiny_decode_workload():
    w = gqa_synth.WORKLOADS["tiny_decode"]
    q, k, v, seqlens = gqa_synth.workload_decode_inputs(w, DEV)
    check_full(q, k, v, seqlens, w.scale, w.num_splits, "tiny")


def test_llama70b_decode_32k_workload():
    w = gqa_synth.WORKLOADS["llama70b_decode_32k"]
    q, k, v, seqlens = gqa_synth.workload_decode_inputs(w, DEV)
    check_full(q, k, v, seqlens, w.scale, 0, "llama70b 32k")


def test_ragged_decode_b16_workload_full():
    """Full-size ragged batch, every (sequence, query head) against the oracle;
    padding past each seqlen holds NaN."""
    w = gqa_synth.WORKLOADS["ragged_decode_b16"]
    q, k, v, seqlens = gqa_synth.workload_decode_inputs(w, DEV)
    gqa_synth.fill_padding(k, seqlens, float("nan"))
    gqa_synth.fill_padding(v, seqlens, float("nan"))
    o, lse = run_decode(q, k, v, seqlens, w.scale)
    ref_o = np.zeros((w.B, w.H_q, w.d))
    ref_lse = np.zeros((w.B, w.H_q))
    for b in range(w.B):       # one sequence at a time: only its valid keys leave the GPU
        n = int(seqlens[b])
        ref_o[b:b + 1], ref_lse[b:b + 1] = oracle.decode(
            np64(q[b:b + 1]), k[b:b + 1, :, :n].float().cpu().numpy(),
            v[b:b + 1, :, :n].float().cpu().numpy(), [n], w.scale)
    compare(o, lse, ref_o, ref_lse, "ragged_decode_b16", max_escape_frac=1e-5)


@pytest.mark.parametrize("seqlens,num_splits", [
    ([1, 333, 1000], 0),        # ragged tails, one single-key sequence
    ([1000, 64, 65], 7),        # tile-exact and one-past-tile lengths
    ([0, 5, 1000], 0),          # an empty sequence: O = 0, lse = -inf
    ([3, 2, 1], 100),           # more splits than keys
    ([1000, 1000, 999], 1),     # one split per sequence (no real merge)
])
def test_ragged_edge_cases(seqlens, num_splits):
    B, H_q, H_kv, S_max, d = 3, 16, 2, 1000, 128
    q, k, v, sl = gqa_synth.decode_inputs(B, H_q, H_kv, S_max, d, seed=11, device=DEV,
                                          seqlens=seqlens)
    check_full(q, k, v, sl, 1 / math.sqrt(d), num_splits, f"edge {seqlens}/{num_splits}")


@pytest.mark.parametrize("H_q,H_kv", [(12, 3), (8, 8), (14, 2), (5, 5)])
def test_group_sizes_below_eight(H_q, H_kv):
    q, k, v, sl = gqa_synth.decode_inputs(2, H_q, H_kv, 700, 128, seed=12, device=DEV,
                                          seqlens=[700, 259])
    check_full(q, k, v, sl, 1 / math.sqrt(128), 0, f"G={H_q // H_kv}")


@pytest.mark.parametrize("num_splits", [1, 2, 5])
def test_single_kernel_path_matches_two_phase_path(num_splits):
    """Plans whose clusters all fit in one wave run as one cluster kernel; the
    explicit split and merge calls always run the two-kernel path.  Both must
    agree."""
    q, k, v, sl = gqa_synth.decode_inputs(3, 64, 8, 2000, 128, seed=18, device=DEV,
                                          seqlens=[2000, 1, 640])
    sl = sl.to(DEV)
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    assert gqa.gqa_attn_decode_kernel_count(3, 64, 8, 2000, 128, num_splits) == 1
    o1, l1 = gqa.gqa_attn_decode(q, k, v, sl, 0.088, num_splits=num_splits)
    ws = torch.empty(gqa.gqa_attn_decode_workspace_size(3, 64, 8, 2000, 128, sms, num_splits),
                     dtype=torch.uint8, device=DEV)
    o2 = torch.empty_like(o1)
    l2 = torch.empty_like(l1)
    gqa.gqa_attn_decode_split(q, k, v, sl, 0.088, num_splits, ws)
    gqa.gqa_attn_decode_merge(sl, 8, 2000, num_splits, o2, l2, ws)
    torch.cuda.synchronize()
    compare(o1, l1, np64(o2), np64(l2), f"single kernel vs split+merge ({num_splits})")
    o_ref, lse_ref = oracle.decode(np64(q), np64(k), np64(v), sl.cpu().numpy(), 0.088)
    compare(o1, l1, o_ref, lse_ref, "single kernel vs oracle")


@pytest.mark.parametrize("B,S,num_splits", [(64, 1024, 0), (40, 700, 1)])
def test_one_split_writes_output_directly(B, S, num_splits):
    """A plan with one split per (sequence, KV head) and too many of them for one
    wave of clusters: the split kernel writes o and lse itself (one launch, no
    merge); empty sequences get O = 0, lse = -inf."""
    rng = np.random.default_rng(B)
    seqlens = [0, 1, S] + [int(x) for x in rng.integers(0, S + 1, B - 3)]
    q, k, v, sl = gqa_synth.decode_inputs(B, 64, 8, S, 128, seed=19, device=DEV, seqlens=seqlens)
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    assert gqa.gqa_attn_decode_plan(B, 8, S, sms, num_splits)[0] == 1
    assert gqa.gqa_attn_decode_kernel_count(B, 64, 8, S, 128, num_splits) == 1
    check_full(q, k, v, sl, 1 / math.sqrt(128), num_splits, f"one split, B={B}")


def test_two_kernel_path_for_many_splits():
    assert gqa.gqa_attn_decode_kernel_count(1, 64, 8, 32768, 128, 37) == 2
    assert gqa.gqa_attn_decode_kernel_count(1, 8, 1, 256, 128, 4) == 1     # tiny: one cluster


def test_nan_padding_is_never_read():
    q, k, v, sl = gqa_synth.decode_inputs(2, 16, 2, 640, 128, seed=13, device=DEV,
                                          seqlens=[577, 100])
    o_ref, lse_ref = run_decode(q, k, v, sl, 0.088)
    gqa_synth.fill_padding(k, sl, float("nan"))
    gqa_synth.fill_padding(v, sl, float("nan"))
    o, lse = run_decode(q, k, v, sl, 0.088)
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


@pytest.mark.parametrize("scale", [0.0, -0.2, 0.5])
def test_scale_values(scale):
    q, k, v, sl = gqa_synth.decode_inputs(1, 16, 2, 300, 128, seed=14, device=DEV,
                                          seqlens=[300])
    check_full(q, k, v, sl, scale, 0, f"scale={scale}")


def test_deterministic_bitwise():
    w = gqa_synth.WORKLOADS["llama70b_decode_32k"]
    q, k, v, seqlens = gqa_synth.workload_decode_inputs(w, DEV)
    o1, l1 = run_decode(q, k, v, seqlens, w.scale)
    o2, l2 = run_decode(q, k, v, seqlens, w.scale)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_host_buffer_variant_matches_device_call():
    q, k, v, sl = gqa_synth.decode_inputs(2, 16, 2, 1500, 128, seed=15, device="cpu",
                                          seqlens=[1500, 777])
    o_dev, lse_dev = run_decode(q.to(DEV), k.to(DEV), v.to(DEV), sl, 0.088)
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    nbytes = gqa.gqa_attn_decode_from_host_arena_size(2, 16, 2, 1500, 128, sms, 0)
    arena = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    pin = lambda t: t.pin_memory()
    o_h = torch.empty((2, 16, 128), dtype=torch.bfloat16).pin_memory()
    lse_h = torch.empty((2, 16), dtype=torch.float32).pin_memory()
    gqa.gqa_attn_decode_from_host(pin(q), pin(k), pin(v), pin(sl), 0.088, 0, o_h, lse_h, arena)
    torch.cuda.synchronize()
    assert torch.equal(o_h, o_dev.cpu()) and torch.equal(lse_h, lse_dev.cpu())


def test_workspace_too_small_is_rejected():
    q, k, v, sl = gqa_synth.decode_inputs(1, 8, 1, 256, 128, seed=16, device=DEV)
    ws = torch.empty(64, dtype=torch.uint8, device=DEV)
    with pytest.raises(gqa.GQAError) as e:
        gqa.gqa_attn_decode(q, k, v, sl.to(DEV), 0.1, workspace=ws)
    assert e.value.status == gqa.GQA_ERR_WORKSPACE


def test_misaligned_device_pointer_is_rejected():
    q, k, v, sl = gqa_synth.decode_inputs(1, 8, 1, 256, 128, seed=17, device=DEV)
    flat = torch.empty(k.numel() + 8, dtype=torch.bfloat16, device=DEV)
    k_off = flat[1:1 + k.numel()].view(k.shape)           # 2-byte offset
    with pytest.raises(gqa.GQAError) as e:
        gqa.gqa_attn_decode(q, k_off, v, sl.to(DEV), 0.1)
    assert e.value.status == gqa.GQA_ERR_INVALID_ARG


def test_bounded_wait_reports_timeout_without_hanging():
    assert gqa.gqa_attn_device_status() == gqa.GQA_OK
    gqa.gqa_attn_selftest_bounded_wait(20000)        # 20 ms wait on a barrier nobody hits
    assert gqa.gqa_attn_device_status() == gqa.GQA_ERR_TIMEOUT
    assert gqa.gqa_attn_device_status() == gqa.GQA_OK   # cleared by the read
    # the context is still usable afterwards
    test_tiny_decode_workload()


def test_out_of_range_seqlens_are_clamped_and_reported():
    """seqlens outside [0, S_max]: used clamped (0 -> no key, S_max -> all
    keys) and reported as GQA_ERR_INVALID_ARG through the device status."""
    B, H_q, H_kv, S = 2, 16, 2, 500
    q, k, v, _ = gqa_synth.decode_inputs(B, H_q, H_kv, S, 128, seed=22, device=DEV)
    bad = torch.tensor([-7, S + 100], dtype=torch.int32)
    assert gqa.gqa_attn_device_status() == gqa.GQA_OK
    o, lse = run_decode(q, k, v, bad, 0.088)
    assert gqa.gqa_attn_device_status() == gqa.GQA_ERR_INVALID_ARG
    o_ref, lse_ref = oracle.decode(np64(q), np64(k), np64(v), np.array([0, S]), 0.088)
    compare(o, lse, o_ref, lse_ref, "clamped seqlens")
    assert gqa.gqa_attn_device_status() == gqa.GQA_OK      # cleared by the read


def test_one_million_keys_full():
    """One sequence of 2^20 - 37 keys in a 2^20-key cache (Llama3-70B heads): each
    of K and V is 2 GiB, so element offsets pass 2^31.  Run on the automatic plan
    (one wave: 19 splits of ~55K keys) and on 512 requested splits that the merge
    combines.  Every head against the oracle (one KV head at a time)."""
    B, H_q, H_kv, S = 1, 64, 8, 1 << 20
    n = S - 37
    q, k, v, sl = gqa_synth.decode_inputs(B, H_q, H_kv, S, 128, seed=71, device=DEV,
                                          seqlens=[n])
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    splits, chunk = gqa.gqa_attn_decode_plan(B, H_kv, S, sms, 0)
    assert splits * chunk >= S and splits * H_kv <= sms
    splits, chunk = gqa.gqa_attn_decode_plan(B, H_kv, S, sms, 512)
    assert splits == 512 and splits * chunk >= S
    runs = [run_decode(q, k, v, sl, 1 / math.sqrt(128)),
            run_decode(q, k, v, sl, 1 / math.sqrt(128), num_splits=512)]
    G = H_q // H_kv
    ref_o = np.zeros((B, H_q, 128))
    ref_lse = np.zeros((B, H_q))
    for kv in range(H_kv):
        heads = slice(kv * G, (kv + 1) * G)
        ref_o[:, heads], ref_lse[:, heads] = oracle.decode(
            np64(q[:, heads]), k[:, kv:kv + 1, :n].float().cpu().numpy(),
            v[:, kv:kv + 1, :n].float().cpu().numpy(), [n], 1 / math.sqrt(128))
    for (o, lse), what in zip(runs, ("one wave", "512 splits")):
        compare(o, lse, ref_o, ref_lse, f"2^20 keys, {what}")


def test_l2_prefetch_sees_the_preceding_grids_writes():
    """A one-wave decode prefetches its first K/V tiles into L2 before its
    grid-dependency wait, while the preceding grid may still be writing.  Here
    the preceding grid (a merge of shard states, which lets its dependents
    launch at its start) writes the very K cache the decode reads, over a
    buffer that held NaN: the decode must see the new keys."""
    H_q, H_kv, S, d = 64, 8, 8192, 128
    # 19 splits x 8 KV heads = one wave of split CTAs (the prefetching path), then the merge
    assert gqa.gqa_attn_decode_kernel_count(1, H_q, H_kv, S, d, 0, DEV) == 2
    g = torch.Generator(device="cpu").manual_seed(77)
    parts = torch.randn((1, H_kv * S, d), generator=g).to(torch.bfloat16).to(DEV)
    lse_parts = torch.zeros((1, H_kv * S), dtype=torch.float32, device=DEV)
    q, _, v, sl = gqa_synth.decode_inputs(1, H_q, H_kv, S, d, seed=78, device=DEV)
    k_buf = torch.full((H_kv * S, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse_out = torch.empty((H_kv * S,), dtype=torch.float32, device=DEV)
    torch.cuda.synchronize()
    for _ in range(3):
        k_buf.fill_(float("nan"))
        # merge of a single shard: writes parts[0] into k_buf (the identity)
        gqa.gqa_attn_merge_states(parts, lse_parts, k_buf, lse_out)
        o, lse = gqa.gqa_attn_decode(q, k_buf.view(1, H_kv, S, d), v, sl.to(DEV),
                                     1 / math.sqrt(d))
        torch.cuda.synchronize()
        assert torch.equal(k_buf, parts[0])
        assert torch.isfinite(o.float()).all()
    o_ref, lse_ref = oracle.decode(np64(q), np64(parts[0].view(1, H_kv, S, d)), np64(v),
                                   sl.numpy(), 1 / math.sqrt(d))
    compare(o, lse, o_ref, lse_ref, "decode after a grid writing its K cache")


@pytest.mark.parametrize("B,S", [(10, 4096), (12, 3000)])
def test_plan_of_few_splits(B, S):
    """Batches whose units fill at least half the SMs take only as many splits as
    the 2048-key chunk cap needs (two here: one-wave clusters)."""
    rng = np.random.default_rng(B + 100)
    seqlens = [0, S] + [int(x) for x in rng.integers(1, S + 1, B - 2)]
    q, k, v, sl = gqa_synth.decode_inputs(B, 64, 8, S, 128, seed=23, device=DEV, seqlens=seqlens)
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    if sms >= 152:
        assert gqa.gqa_attn_decode_plan(B, 8, S, sms, 0)[0] == 2
    check_full(q, k, v, sl, 1 / math.sqrt(128), 0, f"few splits B={B} S={S}")
