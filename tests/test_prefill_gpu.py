"""GPU parity of the causal GQA prefill against the fp64 oracle, through the C ABI.

Small cases span several 128-row and 128-key tiles with ragged tails and are
compared in full; so are the two prefill workloads (8K causal, and the last
2K chunk of a 32K prompt with q_offset = 30720), at full size.  Longer
problems outside the workload list (a 32K square prompt, 256 tokens after
128K keys, G = 16) are compared on sampled rows: the first rows (few visible
keys), rows around tile boundaries and the last rows.
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


def run(q, k, v, q_offset, scale):
    o, lse = gqa.gqa_attn_prefill_causal(q, k, v, scale, q_offset)
    torch.cuda.synchronize()
    return o, lse


@pytest.mark.parametrize("B,H_q,H_kv,T_q,S_kv,q_offset", [
    (1, 8, 1, 300, 300, 0),       # square causal, ragged last tile
    (2, 16, 2, 200, 264, 64),     # chunk after a 64-token prefix
    (1, 8, 2, 257, 300, 43),      # q_offset not tile aligned, one row past a tile
    (1, 6, 2, 130, 130, 0),       # G = 3: the last head pair holds a single head
    (1, 4, 4, 129, 200, 71),      # G = 1 (MHA)
    (1, 8, 1, 1, 1, 0),           # one query, one key
    (1, 8, 1, 1, 517, 516),       # one query at the end of a long prefix
    (1, 16, 2, 384, 384, 0),      # exact multiple of the tile
    (2, 8, 2, 300, 1000, 700),    # G = 4: one head quad per KV head, two sequences
    (1, 12, 1, 200, 200, 0),      # G = 12: three head quads
    (1, 10, 2, 520, 600, 80),     # G = 5: the last head of a group over query tiles 4+3, 2+1, 0
    (2, 7, 1, 384, 384, 0),       # G = 7, three query tiles: last head over tiles 2+1, then 0
    (1, 3, 3, 257, 257, 0),       # G = 1 (MHA), query tiles 2+1, then 0 (ragged)
])
def test_small_cases_full_compare(B, H_q, H_kv, T_q, S_kv, q_offset):
    q, k, v = gqa_synth.prefill_inputs(B, H_q, H_kv, T_q, S_kv, 128, seed=31, device=DEV)
    scale = 1 / math.sqrt(128)
    o, lse = run(q, k, v, q_offset, scale)
    o_ref, lse_ref = oracle.prefill_causal(np64(q), np64(k), np64(v), q_offset, scale)
    compare(o, lse, o_ref, lse_ref, f"prefill {B},{H_q},{H_kv},{T_q},{S_kv},{q_offset}")


@pytest.mark.parametrize("name", ["causal_prefill_8k", "chunked_prefill_32k"])
def test_prefill_workloads_full(name):
    """Both prefill workloads at full size, every (head, row) against the oracle
    (the oracle runs in parallel processes over (KV head, row range) pieces)."""
    from oracle_pool import prefill_causal_parallel
    w = gqa_synth.WORKLOADS[name]
    q, k, v = gqa_synth.workload_prefill_inputs(w, DEV)
    o, lse = run(q, k, v, w.q_offset, w.scale)
    qn, kn, vn = (t.float().cpu().numpy() for t in (q, k, v))
    o_ref, lse_ref = prefill_causal_parallel(qn, kn, vn, w.q_offset, w.scale)
    compare(o, lse, o_ref, lse_ref, name, max_escape_frac=1e-5)


def _seeded_configs(n, seed):
    """Random shapes: group sizes that use CTA pairs (4, 8, 12, 16) and one CTA
    per unit (1, 2, 3, 6), ragged query tiles, q_offset anywhere in a tile."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        G = int(rng.choice([1, 2, 3, 4, 6, 8, 12, 16]))
        H_kv = int(rng.integers(1, 3))
        B = int(rng.integers(1, 3))
        T_q = int(rng.integers(1, 400))
        q_offset = int(rng.integers(0, 300))
        out.append((B, G * H_kv, H_kv, T_q, q_offset + T_q, q_offset))
    return out


@pytest.mark.parametrize("B,H_q,H_kv,T_q,S_kv,q_offset", _seeded_configs(10, 2024))
def test_seeded_random_shapes(B, H_q, H_kv, T_q, S_kv, q_offset):
    q, k, v = gqa_synth.prefill_inputs(B, H_q, H_kv, T_q, S_kv, 128, seed=37, device=DEV)
    o, lse = run(q, k, v, q_offset, 0.09)
    o_ref, lse_ref = oracle.prefill_causal(np64(q), np64(k), np64(v), q_offset, 0.09)
    compare(o, lse, o_ref, lse_ref, f"random {B},{H_q},{H_kv},{T_q},{S_kv},{q_offset}")


def _seeded_wide_configs(n, seed):
    """Larger random shapes: several rounds of work units, key-range pieces,
    and query rows past the last key (S_kv < q_offset + T_q)."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        G = int(rng.choice([1, 2, 4, 5, 8, 16]))
        H_kv = int(rng.choice([1, 2, 4]))
        B = int(rng.integers(1, 3))
        T_q = int(rng.integers(100, 1500))
        q_offset = int(rng.integers(0, 3000))
        short = int(rng.integers(0, min(T_q, 200))) if rng.random() < 0.4 else 0
        out.append((B, G * H_kv, H_kv, T_q, max(1, q_offset + T_q - short), q_offset))
    return out


@pytest.mark.parametrize("B,H_q,H_kv,T_q,S_kv,q_offset", _seeded_wide_configs(8, 2026))
def test_seeded_random_shapes_wide(B, H_q, H_kv, T_q, S_kv, q_offset):
    q, k, v = gqa_synth.prefill_inputs(B, H_q, H_kv, T_q, S_kv, 128, seed=41, device=DEV)
    o, lse = run(q, k, v, q_offset, 0.09)
    o_ref, lse_ref = oracle.prefill_causal(np64(q), np64(k), np64(v), q_offset, 0.09)
    compare(o, lse, o_ref, lse_ref, f"random wide {B},{H_q},{H_kv},{T_q},{S_kv},{q_offset}")


def test_group_of_16_full():
    """G = 16 (four head quads per KV head), 4K causal, every row."""
    from oracle_pool import prefill_causal_parallel
    B, H_q, H_kv, T = 1, 32, 2, 4096
    q, k, v = gqa_synth.prefill_inputs(B, H_q, H_kv, T, T, 128, seed=38, device=DEV)
    o, lse = run(q, k, v, 0, 1 / math.sqrt(128))
    o_ref, lse_ref = prefill_causal_parallel(*(t.float().cpu().numpy() for t in (q, k, v)), 0,
                                             1 / math.sqrt(128))
    compare(o, lse, o_ref, lse_ref, "G = 16, 4K causal", max_escape_frac=1e-5)


@pytest.mark.parametrize("H_q,H_kv", [(8, 2), (4, 2)])   # G = 4 (CTA pairs), G = 2 (one CTA)
def test_running_max_paths(H_q, H_kv):
    """Scores chosen in log2 units (scale = ln 2, q = e_0): key tile 0 scores 0,
    tile 1 scores 7 (every exp is 2^7, the tile sum far above 2^8, yet the max
    stays within 8 of the reference: no rescale), tile 2 scores 20 (the max
    jumps by more than 8: O and the sum are rescaled and the tile redone)."""
    T = 384
    q, k, v = gqa_synth.prefill_inputs(1, H_q, H_kv, T, T, 128, seed=33, device=DEV)
    q.zero_()
    q[..., 0] = 1.0
    k.zero_()
    k[:, :, 128:256, 0] = 7.0
    k[:, :, 256:, 0] = 20.0
    scale = math.log(2.0)
    o, lse = run(q, k, v, 0, scale)
    o_ref, lse_ref = oracle.prefill_causal(np64(q), np64(k), np64(v), 0, scale)
    compare(o, lse, o_ref, lse_ref, f"running max paths G={H_q // H_kv}")


# Shapes whose last round of units is split by key range (76 CTA pairs or 152
# CTAs on a GB300): (B, H_q, H_kv, T_q, S_kv, q_offset).
SPLIT_CASES = [
    (1, 8, 2, 128, 4096, 3968),     # 2 units, 4 pieces each (fewer units than pairs)
    (1, 16, 2, 200, 3000, 2800),    # G = 8, 8 units, ragged second query tile
    (1, 8, 1, 300, 4300, 4000),     # 6 units, 4 pieces each, q_offset not tile aligned
    (1, 32, 8, 1280, 3328, 2048),   # 80 units: one full round, the 4 left cut in 2
    (2, 16, 2, 256, 2304, 2048),    # two sequences
    # one CTA per unit (G not a multiple of 4)
    (1, 6, 2, 128, 4096, 3968),     # G = 3: 4 units, 4 pieces each
    (1, 4, 4, 300, 3000, 2700),     # MHA: last-head units over query tiles 2+1 and 0, cut in 2
    (1, 10, 2, 256, 2560, 2304),    # G = 5
    (2, 8, 4, 200, 2200, 2000),     # G = 2, two sequences, ragged second query tile
]


def _run_ws(q, k, v, q_offset, scale, ws):
    o, lse = gqa.gqa_attn_prefill_causal(q, k, v, scale, q_offset, workspace=ws)
    torch.cuda.synchronize()
    return o, lse


@pytest.mark.parametrize("B,H_q,H_kv,T_q,S_kv,q_offset", SPLIT_CASES)
def test_key_split_full_compare(B, H_q, H_kv, T_q, S_kv, q_offset):
    """Pieces of the last round's units write partial (O, m, l); the merge
    kernel combines them; compared in full with the oracle."""
    nb = gqa.gqa_attn_prefill_causal_workspace_size(B, H_q, H_kv, T_q, S_kv, 128, q_offset,
                                                    torch.cuda.get_device_properties(0).multi_processor_count)
    assert gqa.gqa_attn_prefill_causal_kernel_count(B, H_q, H_kv, T_q, S_kv, 128, q_offset,
                                                    nb, DEV) == 2
    q, k, v = gqa_synth.prefill_inputs(B, H_q, H_kv, T_q, S_kv, 128, seed=41, device=DEV)
    scale = 1 / math.sqrt(128)
    ws = torch.empty(nb, dtype=torch.uint8, device=DEV)
    ws.fill_(0xFF)                     # contents on entry must not matter (NaN bit patterns)
    o, lse = _run_ws(q, k, v, q_offset, scale, ws)
    o_ref, lse_ref = oracle.prefill_causal(np64(q), np64(k), np64(v), q_offset, scale)
    compare(o, lse, o_ref, lse_ref, f"split {B},{H_q},{H_kv},{T_q},{S_kv},{q_offset}")
    # the same call without a workspace runs whole units: equal within rounding
    o1, l1 = _run_ws(q, k, v, q_offset, scale, torch.empty(0, dtype=torch.uint8, device=DEV))
    assert (o.float() - o1.float()).abs().max().item() <= 2 ** -7
    assert (lse - l1).abs().max().item() <= 1e-5
    # deterministic with the split
    o2, l2 = _run_ws(q, k, v, q_offset, scale, ws)
    assert torch.equal(o, o2) and torch.equal(lse, l2)


def test_key_split_scores_jump_between_pieces():
    """Keys of the second half score 20 (log2 units) above the first: the pieces'
    reference maxima differ by 20 and the merge's weights 2^(m_i - M) carry it."""
    B, H_q, H_kv, T_q, S_kv, q_offset = SPLIT_CASES[0]
    q, k, v = gqa_synth.prefill_inputs(B, H_q, H_kv, T_q, S_kv, 128, seed=42, device=DEV)
    q.zero_()
    q[..., 0] = 1.0
    k.zero_()
    k[:, :, 2048:, 0] = 20.0
    k[:, :, 3000:, 0] = -30.0
    scale = math.log(2.0)
    o, lse = gqa.gqa_attn_prefill_causal(q, k, v, scale, q_offset)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.prefill_causal(np64(q), np64(k), np64(v), q_offset, scale)
    compare(o, lse, o_ref, lse_ref, "split, scores jump between pieces")


def test_short_chunk_after_long_prefix_full():
    """A 128-token chunk after 32K keys (Llama3-70B layer): 16 units on 76 pairs,
    each cut in 4 pieces; every row against the oracle."""
    from oracle_pool import prefill_causal_parallel
    B, H_q, H_kv, T_q, S_kv = 1, 64, 8, 128, 32768
    q_offset = S_kv - T_q
    q, k, v = gqa_synth.prefill_inputs(B, H_q, H_kv, T_q, S_kv, 128, seed=43, device=DEV)
    o, lse = gqa.gqa_attn_prefill_causal(q, k, v, 1 / math.sqrt(128), q_offset)
    torch.cuda.synchronize()
    o_ref, lse_ref = prefill_causal_parallel(*(t.float().cpu().numpy() for t in (q, k, v)),
                                             q_offset, 1 / math.sqrt(128))
    compare(o, lse, o_ref, lse_ref, "128 after 32K")


@pytest.mark.parametrize("scale", [0.0, -0.15, 0.3])
def test_scale_values(scale):
    q, k, v = gqa_synth.prefill_inputs(1, 8, 1, 200, 260, 128, seed=32, device=DEV)
    o, lse = run(q, k, v, 60, scale)
    o_ref, lse_ref = oracle.prefill_causal(np64(q), np64(k), np64(v), 60, scale)
    compare(o, lse, o_ref, lse_ref, f"scale={scale}")


def test_deterministic_bitwise():
    q, k, v = gqa_synth.prefill_inputs(1, 64, 8, 1024, 1024, 128, seed=33, device=DEV)
    o1, l1 = run(q, k, v, 0, 0.088)
    o2, l2 = run(q, k, v, 0, 0.088)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_causal_skip_never_reads_future_keys():
    """Keys after the last query's position are never loaded: NaN there changes nothing."""
    q, k, v = gqa_synth.prefill_inputs(1, 8, 1, 256, 1024, 128, seed=34, device=DEV)
    o_ref, l_ref = run(q, k, v, 100, 0.088)     # last query at position 355
    k2, v2 = k.clone(), v.clone()
    k2[:, :, 384:] = float("nan")                # tiles starting at 384 are all future
    v2[:, :, 384:] = float("nan")
    o, l = run(q, k2, v2, 100, 0.088)
    assert torch.equal(o, o_ref) and torch.equal(l, l_ref)


def test_host_buffer_variant_matches_device_call():
    q, k, v = gqa_synth.prefill_inputs(1, 16, 2, 300, 400, 128, seed=35, device="cpu")
    o_dev, l_dev = run(q.to(DEV), k.to(DEV), v.to(DEV), 100, 0.088)
    nbytes = gqa.gqa_attn_prefill_causal_from_host_arena_size(1, 16, 2, 300, 400, 128)
    arena = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    o_h = torch.empty_like(q).pin_memory()
    l_h = torch.empty((1, 16, 300), dtype=torch.float32).pin_memory()
    gqa.gqa_attn_prefill_causal_from_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), 0.088,
                                          100, o_h, l_h, arena)
    torch.cuda.synchronize()
    assert torch.equal(o_h, o_dev.cpu()) and torch.equal(l_h, l_dev.cpu())


def test_rejects_bad_q_offset_and_misalignment():
    q, k, v = gqa_synth.prefill_inputs(1, 8, 1, 64, 64, 128, seed=36, device=DEV)
    with pytest.raises(gqa.GQAError) as e:
        gqa.gqa_attn_prefill_causal(q, k, v, 0.1, q_offset=-1)
    assert e.value.status == gqa.GQA_ERR_INVALID_ARG
    flat = torch.empty(k.numel() + 8, dtype=torch.bfloat16, device=DEV)
    k_off = flat[4:4 + k.numel()].view(k.shape)                # 8-byte offset
    with pytest.raises(gqa.GQAError) as e:
        gqa.gqa_attn_prefill_causal(q, k_off, v, 0.1)
    assert e.value.status == gqa.GQA_ERR_INVALID_ARG


@pytest.mark.parametrize("B,H_q,H_kv,T_q,S_kv,q_offset", [
    (1, 16, 2, 300, 256, 256),     # every row past the keys: unmasked (G = 8, CTA pairs)
    (1, 16, 2, 300, 256, 100),     # rows 0..155 causal, the rest see every key
    (2, 6, 2, 200, 130, 1000),     # G = 3 (one CTA per unit), a ragged key tile
    (1, 4, 4, 129, 385, 300),      # MHA, the boundary inside a query tile
    (1, 64, 8, 512, 1024, 4096),   # a ring step's whole-past block (Llama3-70B heads)
    (1, 32, 8, 256, 4096, 3968),   # G = 4, one query tile straddling the last key
])
def test_rows_past_the_last_key(B, H_q, H_kv, T_q, S_kv, q_offset):
    """Rows at or past the last key see every key (q_offset + T_q > S_kv): the
    whole-past blocks of a ring prefill, through the causal prefill call."""
    q, k, v = gqa_synth.prefill_inputs(B, H_q, H_kv, T_q, S_kv, 128, seed=44, device=DEV)
    o, lse = run(q, k, v, q_offset, 1 / math.sqrt(128))
    o_ref, lse_ref = oracle.prefill_causal(np64(q), np64(k), np64(v), q_offset,
                                           1 / math.sqrt(128))
    compare(o, lse, o_ref, lse_ref, f"past the keys {B},{H_q},{H_kv},{T_q},{S_kv},{q_offset}")


def test_chunk_after_128k_keys_full():
    """A 256-token chunk after 128K keys: 32 units on the CTA pairs, each split by
    key range; every row against the oracle."""
    from oracle_pool import prefill_causal_parallel
    B, H_q, H_kv, T_q, S_kv = 1, 64, 8, 256, 131072
    q_offset = S_kv - T_q
    q, k, v = gqa_synth.prefill_inputs(B, H_q, H_kv, T_q, S_kv, 128, seed=72, device=DEV)
    o, lse = run(q, k, v, q_offset, 1 / math.sqrt(128))
    o_ref, lse_ref = prefill_causal_parallel(*(t.float().cpu().numpy() for t in (q, k, v)),
                                             q_offset, 1 / math.sqrt(128))
    compare(o, lse, o_ref, lse_ref, "256 after 128K", max_escape_frac=1e-5)


def test_long_context_sampled():
    """A 32K square causal prefill (too long for the oracle in full); sampled rows
    against the oracle."""
    T_q = S_kv = 32768
    B, H_q, H_kv = 1, 64, 8
    q_offset = S_kv - T_q
    q, k, v = gqa_synth.prefill_inputs(B, H_q, H_kv, T_q, S_kv, 128, seed=72, device=DEV)
    o, lse = run(q, k, v, q_offset, 1 / math.sqrt(128))
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    rng = np.random.default_rng(10)
    rows = sorted({0, 127, 128, T_q - 1} | set(int(x) for x in rng.integers(0, T_q, 40)))
    picks = [(0, int(rng.integers(0, H_q)), i) for i in rows]
    ref_o = np.zeros((len(picks), 128))
    ref_lse = np.zeros(len(picks))
    for r, (b, h, i) in enumerate(picks):
        n = q_offset + i + 1
        ro, rl = oracle.attend_rows(np64(q[b, h, i])[None], np64(k[b, h // 8, :n]),
                                    np64(v[b, h // 8, :n]), 1 / math.sqrt(128), [n])
        ref_o[r], ref_lse[r] = ro[0], rl[0]
    compare(torch.stack([o[b, h, i] for b, h, i in picks]),
            torch.stack([lse[b, h, i] for b, h, i in picks]), ref_o, ref_lse,
            f"T_q={T_q} after {q_offset}")
