"""Pins for the fp64 oracle against facts other than its own code.

Each test ties the oracle to something the design record "ADR-0060: AHBM GQA
Fused Attention Kernel (Llama3-70B)" or plain mathematics fixes:

* hand-worked cases with exact softmax weights (tests/golden);
* brute force on tiny inputs written from the textbook (un-stabilised)
  softmax definition with Python floats;
* torch's scaled_dot_product_attention in fp64 with the KV heads repeated
  (a library routine) for GQA head sharing and causal masks;
* closed forms (uniform scores give the mean of V and lse = ln n; causal
  row 0 is V[0]; a single key returns its V row);
* the record's own claims: the log-sum-exp merge of any key split, empty
  shards included, equals the unsplit result (section 4), and the per-tile
  online softmax (section 3) equals it for any tile size;
* invariants: convexity, key-permutation invariance, the causal boundary
  including the diagonal (section 5.4), padding past seqlen ignored.

``test_planted_mistakes_are_caught`` plants plausible mistakes in copies of
the oracle and checks that these pins catch every one.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as A

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# independent references used by the pins
# ---------------------------------------------------------------------------

def brute_row(q, keys, vals, scale):
    """Textbook softmax without max subtraction, pure Python floats."""
    s = [scale * sum(a * b for a, b in zip(q, k)) for k in keys]
    w = [math.exp(x) for x in s]
    z = sum(w)
    o = [sum(wj * vj[c] for wj, vj in zip(w, vals)) / z for c in range(len(vals[0]))]
    return o, math.log(z)


def brute_decode(q, k, v, seqlens, scale):
    B, H_q, d = q.shape
    H_kv = k.shape[1]
    G = H_q // H_kv
    o = np.zeros((B, H_q, d))
    lse = np.zeros((B, H_q))
    for b in range(B):
        n = int(seqlens[b])
        for h in range(H_q):
            if n == 0:
                lse[b, h] = -math.inf
                continue
            keys = k[b, h // G, :n].tolist()
            vals = v[b, h // G, :n].tolist()
            oo, ll = brute_row(q[b, h].tolist(), keys, vals, scale)
            o[b, h], lse[b, h] = oo, ll
    return o, lse


def brute_prefill(q, k, v, q_offset, scale):
    B, H_q, T_q, d = q.shape
    G = H_q // k.shape[1]
    o = np.zeros((B, H_q, T_q, d))
    lse = np.zeros((B, H_q, T_q))
    for b in range(B):
        for h in range(H_q):
            for i in range(T_q):
                n = q_offset + i + 1
                oo, ll = brute_row(q[b, h, i].tolist(), k[b, h // G, :n].tolist(),
                                   v[b, h // G, :n].tolist(), scale)
                o[b, h, i], lse[b, h, i] = oo, ll
    return o, lse


def sdpa_prefill(q, k, v, q_offset, scale):
    """torch SDPA (fp64, CPU) with KV repeated G times and an explicit causal mask."""
    qt = torch.from_numpy(np.asarray(q, dtype=np.float64))
    kt = torch.from_numpy(np.asarray(k, dtype=np.float64))
    vt = torch.from_numpy(np.asarray(v, dtype=np.float64))
    G = qt.shape[1] // kt.shape[1]
    kt = kt.repeat_interleave(G, dim=1)
    vt = vt.repeat_interleave(G, dim=1)
    T_q, S_kv = qt.shape[2], kt.shape[2]
    pos = torch.arange(T_q)[:, None] + q_offset
    mask = torch.arange(S_kv)[None, :] <= pos
    return torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, attn_mask=mask, scale=scale).numpy()


def rng_inputs(seed, *shapes):
    r = np.random.default_rng(seed)
    return [r.standard_normal(s) for s in shapes]


# ---------------------------------------------------------------------------
# pins
# ---------------------------------------------------------------------------

def test_hand_worked_golden():
    with open(os.path.join(GOLDEN, "hand_worked_softmax.json")) as f:
        g = json.load(f)
    dec = g["decode"]
    q = np.array(dec["q"])[None]                       # [1, H_q, d]
    k = np.array(dec["k"])[None, None]                 # [1, 1, S, d]
    v = np.array(dec["v"])[None, None]
    o, lse = oracle.decode(q, k, v, [dec["seqlen"]], g["scale"])
    np.testing.assert_allclose(o[0], dec["expect_o"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse[0], dec["expect_lse"], rtol=0, atol=1e-13)

    pf = g["prefill"]
    q = np.array(pf["q"])[None, None]                  # [1, 1, T_q, d]
    k = np.array(pf["k"])[None, None]
    v = np.array(pf["v"])[None, None]
    o, lse = oracle.prefill_causal(q, k, v, pf["q_offset"], g["scale"])
    np.testing.assert_allclose(o[0, 0], pf["expect_o"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse[0, 0], pf["expect_lse"], rtol=0, atol=1e-13)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_decode_matches_brute_force(seed):
    B, H_q, H_kv, S, d = 3, 4, 2, 5, 4
    q, k, v = rng_inputs(seed, (B, H_q, d), (B, H_kv, S, d), (B, H_kv, S, d))
    seqlens = [1, 3, 5]
    scale = 0.37
    o, lse = oracle.decode(q, k, v, seqlens, scale)
    bo, blse = brute_decode(q, k, v, seqlens, scale)
    np.testing.assert_allclose(o, bo, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, blse, rtol=0, atol=1e-12)


@pytest.mark.parametrize("q_offset", [0, 1, 3])
def test_prefill_matches_brute_force(q_offset):
    B, H_q, H_kv, T_q, d = 2, 4, 2, 3, 4
    S_kv = q_offset + T_q
    q, k, v = rng_inputs(10 + q_offset, (B, H_q, T_q, d), (B, H_kv, S_kv, d), (B, H_kv, S_kv, d))
    scale = 0.61
    o, lse = oracle.prefill_causal(q, k, v, q_offset, scale)
    bo, blse = brute_prefill(q, k, v, q_offset, scale)
    np.testing.assert_allclose(o, bo, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, blse, rtol=0, atol=1e-12)


@pytest.mark.parametrize("q_offset,T_q,S_kv", [(0, 16, 16), (5, 11, 16), (9, 7, 20)])
def test_prefill_matches_torch_sdpa_gqa(q_offset, T_q, S_kv):
    B, H_q, H_kv, d = 2, 8, 2, 16
    q, k, v = rng_inputs(20 + q_offset, (B, H_q, T_q, d), (B, H_kv, S_kv, d), (B, H_kv, S_kv, d))
    scale = 1 / math.sqrt(d)
    o, _ = oracle.prefill_causal(q, k, v, q_offset, scale, row_block=4)
    ref = sdpa_prefill(q, k, v, q_offset, scale)
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("q_offset,T_q,S_kv", [(3, 4, 5), (5, 3, 5), (9, 2, 4)])
def test_prefill_rows_past_the_keys_match_brute_force(q_offset, T_q, S_kv):
    """Rows at or past the last key see every key (the ring's whole-past blocks)."""
    B, H_q, H_kv, d = 2, 4, 2, 4
    q, k, v = rng_inputs(30 + q_offset, (B, H_q, T_q, d), (B, H_kv, S_kv, d), (B, H_kv, S_kv, d))
    o, lse = oracle.prefill_causal(q, k, v, q_offset, 0.53)
    bo, blse = brute_prefill(q, k, v, q_offset, 0.53)
    np.testing.assert_allclose(o, bo, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, blse, rtol=0, atol=1e-12)


def test_rows_wholly_past_the_keys_equal_unmasked_attention():
    """q_offset >= S_kv - 1: every row sees the whole block, i.e. plain (unmasked)
    attention -- torch SDPA without a mask, KV heads repeated."""
    B, H_q, H_kv, T_q, S_kv, d = 2, 8, 2, 6, 9, 16
    q, k, v = rng_inputs(41, (B, H_q, T_q, d), (B, H_kv, S_kv, d), (B, H_kv, S_kv, d))
    o, _ = oracle.prefill_causal(q, k, v, S_kv + 3, 0.2, row_block=4)
    qt, kt, vt = (torch.from_numpy(x) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(
        qt, kt.repeat_interleave(4, dim=1), vt.repeat_interleave(4, dim=1), scale=0.2).numpy()
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)
    o2, _ = oracle.prefill_causal(q, k, v, S_kv - 1, 0.2)     # the last key is row 0's own
    np.testing.assert_allclose(o2, ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("n_ranks", [2, 3, 4])
def test_ring_steps_merge_to_the_causal_prefill(n_ranks):
    """The record's section 5.5 ring: a causal prefill whose sequence is cut into
    n chunks equals, for query chunk r, the log-sum-exp merge over the KV chunks
    src <= r of attention over chunk src -- causal on the diagonal (src = r),
    unmasked for whole-past chunks (src < r) -- with whole-future chunks skipped."""
    B, H_q, H_kv, C, d = 1, 4, 2, 5, 8
    S = n_ranks * C
    q, k, v = rng_inputs(50 + n_ranks, (B, H_q, S, d), (B, H_kv, S, d), (B, H_kv, S, d))
    o_ref, lse_ref = oracle.prefill_causal(q, k, v, 0, 0.3)
    for r in range(n_ranks):
        qc = q[:, :, r * C:(r + 1) * C]
        parts_o, parts_l = [], []
        for src in range(n_ranks):
            if src > r:
                continue                                      # whole-future block: skipped
            kc, vc = k[:, :, src * C:(src + 1) * C], v[:, :, src * C:(src + 1) * C]
            po, pl = oracle.prefill_causal(qc, kc, vc, (r - src) * C, 0.3)
            parts_o.append(po)
            parts_l.append(pl)
        o, lse = oracle.merge_states(np.stack(parts_o).reshape(len(parts_o), -1, d),
                                     np.stack(parts_l).reshape(len(parts_l), -1))
        np.testing.assert_allclose(o.reshape(B, H_q, C, d), o_ref[:, :, r * C:(r + 1) * C],
                                   rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse.reshape(B, H_q, C), lse_ref[:, :, r * C:(r + 1) * C],
                                   rtol=0, atol=1e-12)


def test_decode_matches_torch_sdpa_gqa():
    B, H_q, H_kv, S, d = 2, 8, 2, 40, 16
    q, k, v = rng_inputs(30, (B, H_q, d), (B, H_kv, S, d), (B, H_kv, S, d))
    scale = 1 / math.sqrt(d)
    o, _ = oracle.decode(q, k, v, [S, S], scale)
    # decode is the last causal row of a prefill whose query sits at position S-1
    ref = sdpa_prefill(q[:, :, None, :], k, v, S - 1, scale)[:, :, 0]
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)


def test_decode_multi_pins():
    """T_q new tokens: T_q = 1 is decode; equal lengths make it the causal prefill
    of the last T_q rows (q_offset = S - T_q); brute force on a tiny case; tokens
    at negative positions see nothing."""
    B, H_q, H_kv, S, d, T_q = 2, 4, 2, 9, 8, 3
    q, k, v = rng_inputs(120, (B, H_q, T_q, d), (B, H_kv, S, d), (B, H_kv, S, d))
    o1, l1 = oracle.decode_multi(q[:, :, :1], k, v, [S, 5], 0.4)
    od, ld = oracle.decode(q[:, :, 0], k, v, [S, 5], 0.4)
    np.testing.assert_allclose(o1[:, :, 0], od, rtol=0, atol=1e-14)
    np.testing.assert_allclose(l1[:, :, 0], ld, rtol=0, atol=1e-14)
    om, lm = oracle.decode_multi(q, k, v, [S, S], 0.4)
    op, lp = oracle.prefill_causal(q, k, v, S - T_q, 0.4)
    np.testing.assert_allclose(om, op, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lm, lp, rtol=0, atol=1e-13)
    om, lm = oracle.decode_multi(q, k, v, [6, 2], 0.4)
    for b, n in enumerate([6, 2]):
        for h in range(H_q):
            for t in range(T_q):
                pos = n - T_q + t
                if pos < 0:
                    assert np.all(om[b, h, t] == 0) and np.isneginf(lm[b, h, t])
                    continue
                bo, bl = brute_row(q[b, h, t].tolist(), k[b, h // 2, :pos + 1].tolist(),
                                   v[b, h // 2, :pos + 1].tolist(), 0.4)
                np.testing.assert_allclose(om[b, h, t], bo, rtol=0, atol=1e-12)
                assert lm[b, h, t] == pytest.approx(bl, abs=1e-12)


def test_uniform_scores_give_mean_of_v():
    B, H_q, H_kv, S, d = 2, 4, 1, 9, 8
    _, k, v = rng_inputs(40, (1,), (B, H_kv, S, d), (B, H_kv, S, d))
    q = np.zeros((B, H_q, d))
    seqlens = [4, 9]
    o, lse = oracle.decode(q, k, v, seqlens, 0.5)
    for b, n in enumerate(seqlens):
        np.testing.assert_allclose(o[b], np.broadcast_to(v[b, 0, :n].mean(0), (H_q, d)),
                                   rtol=0, atol=1e-14)
        np.testing.assert_allclose(lse[b], math.log(n), rtol=0, atol=1e-14)
    # scale = 0 gives the same closed form with any q
    qr, = rng_inputs(41, (B, H_q, d))
    o0, lse0 = oracle.decode(qr, k, v, seqlens, 0.0)
    np.testing.assert_allclose(o0, o, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse0, lse, rtol=0, atol=1e-14)


def test_causal_row0_is_v0_and_single_key():
    B, H_q, H_kv, T_q, d = 1, 4, 2, 5, 8
    q, k, v = rng_inputs(50, (B, H_q, T_q, d), (B, H_kv, T_q, d), (B, H_kv, T_q, d))
    scale = 0.3
    o, lse = oracle.prefill_causal(q, k, v, 0, scale)
    for h in range(H_q):
        np.testing.assert_array_equal(o[0, h, 0], v[0, h // 2, 0])
        assert lse[0, h, 0] == pytest.approx(scale * float(q[0, h, 0] @ k[0, h // 2, 0]),
                                             abs=1e-14)
    # a decode that sees one key returns that key's V row
    od, lsed = oracle.decode(q[:, :, 0], k, v, [1], scale)
    for h in range(H_q):
        np.testing.assert_array_equal(od[0, h], v[0, h // 2, 0])


def test_empty_visible_set():
    q, k, v = rng_inputs(60, (2, 2, 4), (2, 1, 3, 4), (2, 1, 3, 4))
    o, lse = oracle.decode(q, k, v, [0, 3], 1.0)
    assert np.all(o[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))


@pytest.mark.parametrize("seed", [0, 1])
def test_split_merge_equals_unsplit(seed):
    r = np.random.default_rng(seed)
    R, N, d = 6, 37, 8
    q, k, v = r.standard_normal((R, d)), r.standard_normal((N, d)), r.standard_normal((N, d))
    scale = 0.4
    ref_o, ref_lse = A.attend_rows(q, k, v, scale, np.full(R, N))
    for trial in range(5):
        cuts = np.sort(r.integers(0, N + 1, size=r.integers(1, 6)))
        bounds = [0, *cuts.tolist(), N]                   # repeated cuts = empty shards
        parts = [A.partial_triplet(q, k, v, scale, lo, hi)
                 for lo, hi in zip(bounds[:-1], bounds[1:])]
        order = r.permutation(len(parts))                 # commutative: any order
        acc = parts[order[0]]
        for i in order[1:]:
            acc = A.merge_triplets(acc, parts[i])
        o, lse = A.finalize_triplet(acc)
        np.testing.assert_allclose(o, ref_o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_merge_states_of_shards_equals_unsplit(seed):
    """Attention over disjoint key shards, each finalised to (O_i, lse_i), then
    combined by merge_states, equals attention over all keys (the record's
    section 4 associativity); empty shards (lse = -inf) change nothing."""
    r = np.random.default_rng(100 + seed)
    R, N, d = 5, 41, 8
    q, k, v = r.standard_normal((R, d)), r.standard_normal((N, d)), r.standard_normal((N, d))
    scale = 0.35
    ref_o, ref_lse = A.attend_rows(q, k, v, scale, np.full(R, N))
    cuts = np.sort(r.integers(0, N + 1, size=4))
    bounds = [0, *cuts.tolist(), N]
    o_p, l_p = [], []
    for lo, hi in zip(bounds[:-1], bounds[1:]):
        o_i, l_i = A.finalize_triplet(A.partial_triplet(q, k, v, scale, lo, hi))
        o_p.append(o_i)
        l_p.append(l_i)
    o, lse = A.merge_states(np.stack(o_p), np.stack(l_p))
    np.testing.assert_allclose(o, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_merge_states_closed_forms():
    """Two states with equal lse average their outputs and add ln 2; a single
    state is returned unchanged; all-empty rows give (0, -inf)."""
    o = np.array([[[1.0, -2.0]], [[3.0, 4.0]]])
    lse = np.array([[0.5], [0.5]])
    out, l = A.merge_states(o, lse)
    np.testing.assert_allclose(out, [[2.0, 1.0]], rtol=0, atol=1e-15)
    np.testing.assert_allclose(l, [0.5 + np.log(2.0)], rtol=0, atol=1e-15)
    out, l = A.merge_states(o[:1], lse[:1])
    np.testing.assert_array_equal(out, o[0])
    np.testing.assert_array_equal(l, lse[0])
    out, l = A.merge_states(o, np.full((2, 1), -np.inf))
    np.testing.assert_array_equal(out, [[0.0, 0.0]])
    assert l[0] == -np.inf


@pytest.mark.parametrize("tile", [1, 3, 7, 64])
def test_online_softmax_tiles_equal_definition(tile):
    r = np.random.default_rng(tile)
    R, N, d = 5, 50, 8
    q, k, v = r.standard_normal((R, d)), r.standard_normal((N, d)), r.standard_normal((N, d))
    n_visible = np.array([0, 1, 17, 49, 50])
    o, lse = A.online_softmax_tiles(q, k, v, 0.7, n_visible, tile)
    ref_o, ref_lse = A.attend_rows(q, k, v, 0.7, n_visible)
    np.testing.assert_allclose(o, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_convexity_and_permutation_invariance():
    B, H_q, H_kv, S, d = 1, 4, 1, 30, 8
    q, k, v = rng_inputs(70, (B, H_q, d), (B, H_kv, S, d), (B, H_kv, S, d))
    q *= 3.0
    o, lse = oracle.decode(q, k, v, [S], 0.5)
    lo, hi = v[0, 0].min(0), v[0, 0].max(0)
    assert np.all(o[0] >= lo - 1e-12) and np.all(o[0] <= hi + 1e-12)
    perm = np.random.default_rng(71).permutation(S)
    op, lsep = oracle.decode(q, k[:, :, perm], v[:, :, perm], [S], 0.5)
    np.testing.assert_allclose(op, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lsep, lse, rtol=0, atol=1e-12)


def test_gqa_head_mapping_is_h_div_G():
    B, H_q, H_kv, S, d = 1, 6, 3, 7, 4
    q, k, v = rng_inputs(80, (B, H_q, d), (B, H_kv, S, d), (B, H_kv, S, d))
    o, _ = oracle.decode(q, k, v, [S], 0.5)
    # G = 2: heads 0,1 -> kv 0; 2,3 -> kv 1; 4,5 -> kv 2 (MHA with repeated KV)
    k_rep = np.repeat(k, 2, axis=1)
    v_rep = np.repeat(v, 2, axis=1)
    o_mha, _ = oracle.decode(q, k_rep, v_rep, [S], 0.5)
    np.testing.assert_allclose(o, o_mha, rtol=0, atol=1e-14)
    for h in range(H_q):
        single, _ = A.attend_rows(q[0, h][None], k[0, h // 2], v[0, h // 2], 0.5, [S])
        np.testing.assert_allclose(o[0, h], single[0], rtol=0, atol=1e-14)


def test_causal_boundary_includes_diagonal():
    B, H_q, H_kv, T_q, d, q_offset = 1, 2, 1, 6, 4, 3
    S_kv = q_offset + T_q
    q, k, v = rng_inputs(90, (B, H_q, T_q, d), (B, H_kv, S_kv, d), (B, H_kv, S_kv, d))
    o, _ = oracle.prefill_causal(q, k, v, q_offset, 0.5)
    for i in range(T_q):
        pos = q_offset + i
        if pos + 1 < S_kv:            # the next key is invisible to row i
            v2 = v.copy(); v2[0, 0, pos + 1] += 100.0
            o2, _ = oracle.prefill_causal(q, k, v2, q_offset, 0.5)
            np.testing.assert_array_equal(o2[0, :, i], o[0, :, i])
        v3 = v.copy(); v3[0, 0, pos] += 100.0      # the diagonal key is visible
        o3, _ = oracle.prefill_causal(q, k, v3, q_offset, 0.5)
        assert np.all(np.abs(o3[0, :, i] - o[0, :, i]) > 1e-6)


def test_decode_ignores_padding_past_seqlen():
    B, H_q, H_kv, S, d = 2, 4, 2, 12, 8
    q, k, v = rng_inputs(100, (B, H_q, d), (B, H_kv, S, d), (B, H_kv, S, d))
    seqlens = [5, 12]
    o, lse = oracle.decode(q, k, v, seqlens, 0.5)
    k2, v2 = k.copy(), v.copy()
    k2[0, :, 5:] = np.nan
    v2[0, :, 5:] = np.nan
    o2, lse2 = oracle.decode(q, k2, v2, seqlens, 0.5)
    np.testing.assert_array_equal(o2, o)
    np.testing.assert_array_equal(lse2, lse)


def test_sampled_rows_match_full():
    B, H_q, H_kv, T_q, d, q_offset = 2, 4, 2, 9, 8, 4
    S_kv = q_offset + T_q
    q, k, v = rng_inputs(110, (B, H_q, T_q, d), (B, H_kv, S_kv, d), (B, H_kv, S_kv, d))
    o, lse = oracle.prefill_causal(q, k, v, q_offset, 0.3, row_block=4)
    picks = [(0, 0, 0), (1, 3, 8), (0, 2, 5), (1, 1, 4)]
    so, slse = oracle.prefill_causal_rows(q, k, v, q_offset, 0.3, picks)
    for r, (b, h, i) in enumerate(picks):     # equal up to BLAS summation order
        np.testing.assert_allclose(so[r], o[b, h, i], rtol=0, atol=1e-14)
        assert slse[r] == pytest.approx(lse[b, h, i], abs=1e-14)
    qd = q[:, :, 0]
    od, lsed = oracle.decode(qd, k, v, [3, 13], 0.3)
    pairs = [(0, 1), (1, 3)]
    po, plse = oracle.decode_pairs(qd, k, v, [3, 13], 0.3, pairs)
    for r, (b, h) in enumerate(pairs):
        np.testing.assert_allclose(po[r], od[b, h], rtol=0, atol=1e-14)


def test_bf16_inputs_are_read_exactly():
    """The oracle sees bf16 inputs as exact fp64 values (no re-rounding)."""
    import gqa_synth
    t = gqa_synth.bf16_normal((4, 8), seed=5)
    as64 = A._f64(t.float().numpy())
    np.testing.assert_array_equal(as64, t.double().numpy())


# ---------------------------------------------------------------------------
# planted mistakes: each mutant oracle must fail at least one pin above
# ---------------------------------------------------------------------------

def _mutant_attend(kind):
    def attend(q_rows, k, v, scale, n_visible):
        q_rows, k, v = A._f64(q_rows), A._f64(k), A._f64(v)
        n_visible = np.asarray(n_visible, dtype=np.int64).reshape(-1)
        if kind == "dropped_scale":
            scale = 1.0
        if kind == "swapped_kv":
            k, v = v, k
        N = k.shape[0]
        s = float(scale) * (q_rows @ k.T)
        if kind == "wrong_sign":
            s = -s
        limit = n_visible - 1 if kind == "causal_off_by_one" else n_visible
        vis = np.arange(N)[None, :] < limit[:, None]
        s = np.where(vis, s, -np.inf)
        m = s.max(axis=1, initial=-np.inf)
        m = np.where(np.isfinite(m), m, 0.0)
        e = np.where(vis, np.exp(s - m[:, None]), 0.0)
        l = e.sum(1)
        o = np.zeros((q_rows.shape[0], v.shape[1]))
        ok = l > 0
        o[ok] = (e[ok] @ v) / l[ok, None]
        lse = np.full(len(l), -np.inf)
        lse[ok] = (np.log2(l[ok]) if kind == "lse_log2" else np.log(l[ok])) + m[ok]
        return o, lse
    return attend


@pytest.mark.parametrize("kind", ["dropped_scale", "swapped_kv", "wrong_sign",
                                  "causal_off_by_one", "lse_log2", "head_mod"])
def test_planted_mistakes_are_caught(kind, monkeypatch):
    if kind == "head_mod":
        # query head h mapped to KV head h % H_kv instead of h // G
        orig_decode = A.decode

        def decode(q, k_cache, v_cache, seqlens, scale):
            H_kv = k_cache.shape[1]
            o = np.zeros(q.shape); lse = np.zeros(q.shape[:2])
            for b in range(q.shape[0]):
                for h in range(q.shape[1]):
                    n = int(seqlens[b])
                    oo, ll = A.attend_rows(A._f64(q[b, h])[None], k_cache[b, h % H_kv, :n],
                                           v_cache[b, h % H_kv, :n], scale, [n])
                    o[b, h], lse[b, h] = oo[0], ll[0]
            return o, lse
        monkeypatch.setattr(oracle, "decode", decode)
        with pytest.raises(AssertionError):
            test_decode_matches_torch_sdpa_gqa()
        monkeypatch.setattr(oracle, "decode", orig_decode)
        return
    monkeypatch.setattr(A, "attend_rows", _mutant_attend(kind))
    failed = []
    for name, fn in [("golden", test_hand_worked_golden),
                     ("brute_decode", lambda: test_decode_matches_brute_force(0)),
                     ("brute_prefill", lambda: test_prefill_matches_brute_force(1)),
                     ("sdpa", lambda: test_prefill_matches_torch_sdpa_gqa(5, 11, 16))]:
        try:
            fn()
        except AssertionError:
            failed.append(name)
    assert failed, f"planted mistake {kind!r} was not caught by any pin"
