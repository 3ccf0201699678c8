"""Randomized sweep: many more seeded shapes from the parity tests' own generators.

The decode, prefill and paged-prefill parity tests each draw a few dozen shapes
from seeded generators.  This test keeps drawing from the same generators with
fresh seeds (GQA_SWEEP_SEED, default 5000, then 5001, ...) and compares every
case against the oracle: a fixed number of seeds by default (so the GPU suite
is short and always runs the same cases), or for GQA_SWEEP_SECONDS seconds
when that is set (a long sweep only needs the variable).  Per seed: 16 decode
shapes (every decode path, dense and paged, ragged lengths, forced split
counts), 4 prefill shapes with ragged query tiles, every third seed one wide
prefill (several rounds of units, key-range pieces, rows past the last key),
one paged prefill over a shuffled page pool, and one merge of random attention
states (1 to 70 shards, some empty).  The device status word is checked after
every seed, so a bounds violation reported by the bounds-checked build
(GQA_ATTN_LIB set to libgqa_attn_debug.so) fails the sweep too.

A second sweep (20 seeds, or GQA_SWEEP_LARGE_SECONDS) draws larger decode
problems — batches up to 24, caches up to 64K keys, up to 2M cached rows —
which reach the planner's multi-wave, few-split, one-split and cluster plans.
A third (100 seeds, or GQA_SWEEP_PREFILL_SECONDS) runs causal prefills of up to
8K query rows after up to 32K keys, dense or paged, and checks sampled rows
(tile edges and random ones) against the oracle and every output for
finiteness.
"""
import os
import time

import numpy as np
import pytest
import torch

import gqa_synth
import gqa_attention_decode_gb300 as gqa
import oracle
import test_decode_random_gpu as decode_tests
import test_paged_prefill_gpu as paged_prefill_tests
import test_prefill_gpu as prefill_tests
from parity import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gqa_attention_decode_gb300 import build
    build.build()
    gqa.load_library()
    torch.cuda.set_device(0)
    yield


def _paged_prefill_case(seed):
    """One paged prefill shape: group sizes for one CTA per unit and for CTA
    pairs, page sizes of 128 to 512 keys, key counts on and off whole tiles."""
    rng = np.random.default_rng(seed)
    G = int(rng.choice([1, 2, 3, 4, 8]))
    H_kv = int(rng.choice([1, 2]))
    B = int(rng.integers(1, 3))
    page = int(rng.choice([128, 256, 512]))
    T_q = int(rng.integers(1, 600))
    q_offset = int(rng.integers(0, 2500))
    S_kv = q_offset + T_q
    if rng.random() < 0.5:
        S_kv = -(-S_kv // 128) * 128  # whole key tiles: the CTA-pair kernel reads pages
    return (B, G * H_kv, H_kv, T_q, S_kv, q_offset, page)


def _merge_states_case(seed):
    """Random shard states: n_parts 1..70, rows 0..3000, lse spread over +-18,
    whole shards, single entries and whole rows with no visible key (-inf);
    against the oracle's merge within the bf16 rounding of O."""
    rng = np.random.default_rng(seed)
    P = int(rng.integers(1, 71))
    rows = int(rng.integers(0, 3001))
    g = torch.Generator(device="cpu").manual_seed(seed)
    o_parts = torch.randn((P, rows, 128), generator=g).to(torch.bfloat16)
    lse_parts = (torch.randn((P, rows), generator=g) * 6.0).float()
    if rows:
        lse_parts[torch.rand((P, rows), generator=g) < 0.2] = float("-inf")
        lse_parts[int(rng.integers(0, P))] = float("-inf")       # an empty shard
        lse_parts[:, int(rng.integers(0, rows))] = float("-inf")  # a row empty everywhere
    dev = torch.device("cuda", 0)
    o, lse = gqa.gqa_attn_merge_states(o_parts.to(dev), lse_parts.to(dev))
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.merge_states(o_parts.double().numpy(), lse_parts.double().numpy())
    if rows == 0:
        return
    err = np.abs(o.double().cpu().numpy() - o_ref)
    assert err.max() <= 2.0 ** -7 * max(1.0, np.abs(o_ref).max()), f"merge seed {seed}"
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse.cpu().numpy()), fin), f"merge seed {seed}"
    if fin.any():
        assert np.abs(lse.cpu().numpy()[fin] - lse_ref[fin]).max() <= 1e-5, f"merge seed {seed}"
    assert torch.all(o[torch.from_numpy(~fin).to(o.device)] == 0), f"merge seed {seed}"


def _sweep_limits(var, default_seeds):
    """(seconds, seeds): a time budget when the variable is set, else a seed count."""
    if os.environ.get(var):
        return float(os.environ[var]), None
    return None, default_seeds


def _done(t0, budget, seed, first, n_seeds):
    if n_seeds is not None:
        return seed - first >= n_seeds
    return time.time() - t0 >= budget


def test_random_sweep():
    budget, n_seeds = _sweep_limits("GQA_SWEEP_SECONDS", 12)
    t0 = time.time()
    seed = first = int(os.environ.get("GQA_SWEEP_SEED", "5000"))
    counts = dict(decode=0, prefill=0, wide=0, paged=0, merge=0)
    while True:
        for c in decode_tests._cases(16, seed):
            decode_tests.test_random_decode_shapes(*c)
            counts["decode"] += 1
        for c in prefill_tests._seeded_configs(4, seed):
            prefill_tests.test_seeded_random_shapes(*c)
            counts["prefill"] += 1
        if seed % 3 == 0:
            for c in prefill_tests._seeded_wide_configs(1, seed):
                prefill_tests.test_seeded_random_shapes_wide(*c)
                counts["wide"] += 1
        paged_prefill_tests.test_paged_prefill_against_oracle(*_paged_prefill_case(seed))
        counts["paged"] += 1
        _merge_states_case(seed)
        counts["merge"] += 1
        assert gqa.gqa_attn_device_status() == gqa.GQA_OK, f"device status after seed {seed}"
        seed += 1
        if _done(t0, budget, seed, first, n_seeds):
            break
    print(f"random sweep: seeds {first}..{seed - 1}, cases {counts}")


def _large_decode_case(seed):
    """A decode problem large enough for multi-wave plans: (G, H_kv, T_q, B,
    S_max, seqlens, splits, page) as the decode parity test takes them, with at
    most 2M cached rows and 2^27 (row, key) pairs for the oracle."""
    rng = np.random.default_rng(seed)
    G = int(rng.choice([1, 2, 4, 5, 8, 16]))
    H_kv = int(rng.choice([1, 2, 4, 8])) if G <= 8 else int(rng.choice([1, 2, 4]))
    T_q = int(rng.integers(1, max(1, min(16, 128 // G)) + 1))
    B = int(rng.integers(1, 25))
    tensor_cores = G > 8 or G * T_q > 32
    paged = bool(rng.random() < 0.4)
    page = (int(rng.choice([128, 256])) if tensor_cores else int(rng.choice([64, 128, 256]))) if paged else 0
    unit = page or 64
    cap = min((1 << 21) // (B * H_kv), (1 << 27) // (B * H_kv * G * T_q))
    S_max = int(rng.integers(1, 65536 // unit + 1)) * unit
    S_max = max(unit, min(S_max, cap // unit * unit))
    kind = rng.random()
    if kind < 0.4:
        seqlens = [S_max] * B                                    # every sequence full
    elif kind < 0.8:
        seqlens = [int(x) for x in rng.integers(0, S_max + 1, B)]  # ragged
    else:
        seqlens = [int(x) for x in rng.integers(0, min(S_max, 600) + 1, B)]  # short in a long cache
    splits = int(rng.choice([0, 0, 0, 1, 2, 7, 33]))
    return (G, H_kv, T_q, B, S_max, tuple(seqlens), splits, page)


def test_random_sweep_large_decode():
    budget, n_seeds = _sweep_limits("GQA_SWEEP_LARGE_SECONDS", 20)
    t0 = time.time()
    seed = first = int(os.environ.get("GQA_SWEEP_SEED", "5000"))
    while True:
        decode_tests.test_random_decode_shapes(*_large_decode_case(seed))
        assert gqa.gqa_attn_device_status() == gqa.GQA_OK, f"device status after seed {seed}"
        seed += 1
        torch.cuda.empty_cache()
        if _done(t0, budget, seed, first, n_seeds):
            break
    print(f"large decode sweep: seeds {first}..{seed - 1}")


def _large_prefill_case(seed):
    """(B, H_q, H_kv, T_q, S_kv, q_offset, page): up to 8K query rows after up to
    32K keys, at most 2^22 query rows and 2^21 cached rows in all; sometimes
    rows past the last key; page 0 for a dense cache."""
    rng = np.random.default_rng(seed)
    G = int(rng.choice([1, 2, 3, 4, 5, 8, 16]))
    H_kv = int(rng.choice([1, 2, 4, 8]))
    B = int(rng.integers(1, 5))
    T_q = int(rng.integers(1, 8193))
    T_q = max(1, min(T_q, (1 << 22) // (B * G * H_kv)))
    q_offset = int(rng.integers(0, 32769 - T_q)) if rng.random() < 0.7 else 0
    S_kv = q_offset + T_q
    if rng.random() < 0.2:
        S_kv = max(1, S_kv - int(rng.integers(0, min(T_q, 300) + 1)))  # rows past the last key
    if B * H_kv * S_kv > (1 << 21):
        return _large_prefill_case(seed + 100000)
    page = 0
    if rng.random() < 0.3 and q_offset + T_q <= S_kv:
        page = int(rng.choice([128, 256, 512]))
        if rng.random() < 0.5:
            S_kv = -(-S_kv // 128) * 128  # whole key tiles: the CTA-pair kernel reads pages
    return (B, G * H_kv, H_kv, T_q, S_kv, q_offset, page)


def test_random_sweep_large_prefill():
    budget, n_seeds = _sweep_limits("GQA_SWEEP_PREFILL_SECONDS", 100)
    t0 = time.time()
    seed = first = int(os.environ.get("GQA_SWEEP_SEED", "5000"))
    dev = torch.device("cuda", 0)
    scale = 0.088
    while True:
        B, H_q, H_kv, T_q, S_kv, q_offset, page = _large_prefill_case(seed)
        G = H_q // H_kv
        q, k, v = gqa_synth.prefill_inputs(B, H_q, H_kv, T_q, S_kv, 128, seed=seed, device=dev)
        if page:
            kp, vp, table = paged_prefill_tests.to_pages(k, v, page, extra_pages=1, seed=seed)
            o, lse = gqa.gqa_attn_prefill_causal_paged(q, kp, vp, table, S_kv, scale, q_offset)
            del kp, vp
        else:
            o, lse = gqa.gqa_attn_prefill_causal(q, k, v, scale, q_offset)
        torch.cuda.synchronize()
        what = f"seed {seed}: B={B} H_q={H_q} H_kv={H_kv} T_q={T_q} S_kv={S_kv} q_offset={q_offset} page={page}"
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all(), what
        rng = np.random.default_rng(seed)
        edges = {0, T_q - 1} | {min(T_q - 1, t) for t in (127, 128, 255, 256)}
        rows = sorted(edges | set(int(x) for x in rng.integers(0, T_q, 40)))
        picks = [(int(rng.integers(0, B)), int(rng.integers(0, H_q)), i) for i in rows]
        qs = q[[b for b, _, _ in picks], [h for _, h, _ in picks], rows]
        ref_o = np.zeros((len(picks), 128))
        ref_lse = np.zeros(len(picks))
        for r, (b, h, i) in enumerate(picks):
            n = min(q_offset + i + 1, S_kv)
            ro, rl = oracle.attend_rows(qs[r:r + 1].float().cpu().numpy().astype(np.float64),
                                        k[b, h // G, :n].float().cpu().numpy().astype(np.float64),
                                        v[b, h // G, :n].float().cpu().numpy().astype(np.float64),
                                        scale, [n])
            ref_o[r], ref_lse[r] = ro[0], rl[0]
        compare(torch.stack([o[b, h, i] for b, h, i in picks]),
                torch.stack([lse[b, h, i] for b, h, i in picks]), ref_o, ref_lse, what)
        del q, k, v, o, lse
        assert gqa.gqa_attn_device_status() == gqa.GQA_OK, f"device status after seed {seed}"
        seed += 1
        torch.cuda.empty_cache()
        if _done(t0, budget, seed, first, n_seeds):
            break
    print(f"large prefill sweep: seeds {first}..{seed - 1}")
