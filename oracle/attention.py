"""fp64 reference for GQA decode and causal prefill (test infrastructure only).

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT: only the tests, the smoke check
and the bench's CPU-baseline leg use this module.  It shares no code with the
CUDA library.

Source: "ADR-0060: AHBM GQA Fused Attention Kernel (Llama3-70B)" (kernbench2,
revision 5a76ed4).  Its "Algorithm lineage" paragraph states that the kernels
are FlashAttention (online softmax), FlashDecoding (split-KV with a
log-sum-exp merge) and Ring Attention, and that no new math is introduced.
All of them reach the same result as plain scaled softmax attention, so that
definition is what ``attend_rows``/``decode``/``prefill_causal`` write out:

    s_j  = scale * <q, k_j>                   for visible keys j
    m    = max_j s_j
    l    = sum_j exp(s_j - m)
    O    = sum_j exp(s_j - m) * v_j / l
    lse  = m + ln l                            (natural log of the scaled scores)

Conventions taken from the record:
  * GQA head sharing: query head h uses KV head h // G, G = H_q / H_kv
    (section 0 "Reference dimensions"; section 0.5.3 "INPUTS": the G query
    rows of one KV head form the group).
  * Decode (T_q = 1) sees every cached key 0..seqlen-1 (section 5.2: no
    future tiles, only the last ragged tile is bounded).
  * Causal prefill: query row i sits at absolute position q_offset + i and
    sees keys 0..q_offset+i inclusive; keys after it are masked (section 5.4
    "PREFILL, no SP": all-past tiles unmasked, all-future tiles skipped,
    boundary tiles masked).  A row at or past the last key sees every key:
    the steps of section 5.5's ring where a KV block lies wholly before the
    query block attend to the whole block.
  * An empty visible set gives O = 0 and lse = -inf (the record is silent;
    this is the reading the merge needs so that an empty split is the
    identity of the log-sum-exp merge).

``partial_triplet``/``merge_triplets``/``finalize_triplet`` restate the
split-and-combine of section 4 ("Reduction ... 2-level reduce-to-root": the
unnormalised (m, l, O) of a key shard and its associative merge), and
``online_softmax_tiles`` restates the per-tile steps of section 3 ("Per-tile
op sequence").  They are not used to produce expected values for the CUDA
path; the tests use them to pin the definition against the record's own
algorithms (any split and any tiling must give the same answer).

All inputs are converted to float64 exactly (bf16 and fp32 values are exact
in fp64) and every step runs in float64.
"""
from __future__ import annotations

import numpy as np

NEG_INF = -np.inf


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


# ---------------------------------------------------------------------------
# The definition
# ---------------------------------------------------------------------------

def attend_rows(q_rows, k, v, scale, n_visible):
    """Scaled softmax attention of each query row over a prefix of the keys.

    q_rows [R, d]; k, v [N, d]; n_visible [R] -- row r sees keys
    0 .. n_visible[r]-1 of k and v.  Returns (O [R, d], lse [R]) in float64.
    A row with n_visible = 0 gets O = 0 and lse = -inf.
    """
    q_rows, k, v = _f64(q_rows), _f64(k), _f64(v)
    n_visible = np.asarray(n_visible, dtype=np.int64).reshape(-1)
    R, N = q_rows.shape[0], k.shape[0]
    s = float(scale) * (q_rows @ k.T)                          # [R, N]
    visible = np.arange(N)[None, :] < n_visible[:, None]        # [R, N]
    s = np.where(visible, s, NEG_INF)
    has_keys = n_visible > 0
    m = np.where(has_keys, s.max(axis=1, initial=NEG_INF), 0.0)   # 0 only as a dummy
    e = np.where(visible, np.exp(s - m[:, None]), 0.0)
    l = e.sum(axis=1)
    o = np.zeros((R, v.shape[1]), dtype=np.float64)
    o[has_keys] = (e[has_keys] @ v) / l[has_keys, None]
    lse = np.full(R, NEG_INF)
    lse[has_keys] = m[has_keys] + np.log(l[has_keys])
    return o, lse


def _group_size(H_q: int, H_kv: int) -> int:
    if H_kv <= 0 or H_q % H_kv != 0:
        raise ValueError(f"H_q={H_q} must be a positive multiple of H_kv={H_kv}")
    return H_q // H_kv


def decode(q, k_cache, v_cache, seqlens, scale):
    """Decode (T_q = 1) for every (b, h_q).

    q [B, H_q, d]; k_cache, v_cache [B, H_kv, S_max, d]; seqlens [B].
    Query head h uses KV head h // G and sees cached keys 0..seqlens[b]-1.
    Returns O [B, H_q, d] and lse [B, H_q] in float64.
    """
    q = _f64(q)
    B, H_q, d = q.shape
    H_kv = k_cache.shape[1]
    G = _group_size(H_q, H_kv)
    seqlens = np.asarray(seqlens, dtype=np.int64).reshape(-1)
    o = np.zeros((B, H_q, d))
    lse = np.zeros((B, H_q))
    for b in range(B):
        n = int(seqlens[b])
        for kv in range(H_kv):
            heads = slice(kv * G, (kv + 1) * G)
            k = _f64(k_cache[b, kv, :n])
            v = _f64(v_cache[b, kv, :n])
            o[b, heads], lse[b, heads] = attend_rows(q[b, heads], k, v, scale, np.full(G, n))
    return o, lse


def decode_multi(q, k_cache, v_cache, seqlens, scale):
    """Decode of T_q new tokens per sequence (speculative / multi-token decode).

    q [B, H_q, T_q, d]; k_cache, v_cache [B, H_kv, S_max, d]; seqlens[b] counts
    every cached key of sequence b, the T_q new ones included.  New token t
    sits at absolute position seqlens[b] - T_q + t and sees keys 0..that
    position (causal among the new tokens; the record's T_q of section 0.5.2
    and its G*T_q folded rows of section 5.2).  A token whose position is
    negative sees nothing: O = 0, lse = -inf.
    Returns O [B, H_q, T_q, d] and lse [B, H_q, T_q] in float64.
    """
    B, H_q, T_q, d = q.shape
    H_kv = k_cache.shape[1]
    G = _group_size(H_q, H_kv)
    seqlens = np.asarray(seqlens, dtype=np.int64).reshape(-1)
    o = np.zeros((B, H_q, T_q, d))
    lse = np.zeros((B, H_q, T_q))
    for b in range(B):
        n = int(seqlens[b])
        n_visible = np.clip(n - T_q + np.arange(T_q) + 1, 0, None)
        for kv in range(H_kv):
            k = _f64(k_cache[b, kv, :n])
            v = _f64(v_cache[b, kv, :n])
            for h in range(kv * G, (kv + 1) * G):
                o[b, h], lse[b, h] = attend_rows(_f64(q[b, h]), k, v, scale, n_visible)
    return o, lse


def decode_pairs(q, k_cache, v_cache, seqlens, scale, pairs):
    """Decode for a sample of (b, h_q) pairs only; returns O [P, d], lse [P]."""
    B, H_q, d = q.shape
    G = _group_size(H_q, k_cache.shape[1])
    seqlens = np.asarray(seqlens, dtype=np.int64).reshape(-1)
    o = np.zeros((len(pairs), d))
    lse = np.zeros(len(pairs))
    for i, (b, h) in enumerate(pairs):
        n = int(seqlens[b])
        k = _f64(k_cache[b, h // G, :n])
        v = _f64(v_cache[b, h // G, :n])
        o[i:i + 1], lse[i:i + 1] = attend_rows(_f64(q[b, h])[None, :], k, v, scale, [n])
    return o, lse


def prefill_causal(q, k, v, q_offset, scale, row_block: int = 512):
    """Causal prefill for every (b, h_q, i).

    q [B, H_q, T_q, d]; k, v [B, H_kv, S_kv, d].  Row i is at absolute
    position q_offset + i and sees keys 0..min(q_offset+i, S_kv-1) (rows at or
    past the last key see every key).  Rows are processed in blocks of
    `row_block` only to bound memory; each row is independent.
    Returns O [B, H_q, T_q, d] and lse [B, H_q, T_q] in float64.
    """
    B, H_q, T_q, d = q.shape
    H_kv, S_kv = k.shape[1], k.shape[2]
    G = _group_size(H_q, H_kv)
    if q_offset < 0 or (T_q > 0 and S_kv == 0):
        raise ValueError("need 0 <= q_offset and, with queries, at least one key")
    o = np.zeros((B, H_q, T_q, d))
    lse = np.zeros((B, H_q, T_q))
    for b in range(B):
        for kv in range(H_kv):
            for r0 in range(0, T_q, row_block):
                r1 = min(T_q, r0 + row_block)
                n_keys = min(q_offset + r1, S_kv)  # keys the last row of the block sees
                kb = _f64(k[b, kv, :n_keys])
                vb = _f64(v[b, kv, :n_keys])
                n_visible = np.minimum(q_offset + np.arange(r0, r1) + 1, S_kv)
                for h in range(kv * G, (kv + 1) * G):
                    o[b, h, r0:r1], lse[b, h, r0:r1] = attend_rows(
                        _f64(q[b, h, r0:r1]), kb, vb, scale, n_visible)
    return o, lse


def prefill_causal_rows(q, k, v, q_offset, scale, picks):
    """Causal prefill for a sample of (b, h_q, i) rows; returns O [P, d], lse [P]."""
    B, H_q, T_q, d = q.shape
    G = _group_size(H_q, k.shape[1])
    o = np.zeros((len(picks), d))
    lse = np.zeros(len(picks))
    for r, (b, h, i) in enumerate(picks):
        n = min(q_offset + int(i) + 1, k.shape[2])
        kb = _f64(k[b, h // G, :n])
        vb = _f64(v[b, h // G, :n])
        o[r:r + 1], lse[r:r + 1] = attend_rows(_f64(q[b, h, i])[None, :], kb, vb, scale, [n])
    return o, lse


# ---------------------------------------------------------------------------
# The record's split-and-combine (section 4) and per-tile loop (section 3).
# Used only to pin the definition above; never as an expected value.
# ---------------------------------------------------------------------------

def partial_triplet(q_rows, k, v, scale, lo, hi):
    """Unnormalised (m, l, O) of query rows over the key shard [lo, hi).

    m = max_j s_j, l = sum_j exp(s_j - m), O = sum_j exp(s_j - m) v_j with
    s_j = scale <q, k_j>.  An empty shard is (-inf, 0, 0).
    """
    q_rows = _f64(q_rows)
    R, d = q_rows.shape
    if hi <= lo:
        return np.full(R, NEG_INF), np.zeros(R), np.zeros((R, d))
    kk, vv = _f64(k[lo:hi]), _f64(v[lo:hi])
    s = float(scale) * (q_rows @ kk.T)
    m = s.max(axis=1)
    e = np.exp(s - m[:, None])
    return m, e.sum(axis=1), e @ vv


def merge_triplets(a, b):
    """The record's associative log-sum-exp merge of two (m, l, O) partials.

    m = max(m_a, m_b); l = l_a e^(m_a-m) + l_b e^(m_b-m); O likewise.
    A partial with m = -inf (empty shard) is the identity.
    """
    m_a, l_a, o_a = a
    m_b, l_b, o_b = b
    m = np.maximum(m_a, m_b)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w_a = np.where(np.isfinite(m_a), np.exp(np.where(np.isfinite(m_a), m_a, 0.0) - m_safe), 0.0)
    w_b = np.where(np.isfinite(m_b), np.exp(np.where(np.isfinite(m_b), m_b, 0.0) - m_safe), 0.0)
    return m, l_a * w_a + l_b * w_b, o_a * w_a[:, None] + o_b * w_b[:, None]


def finalize_triplet(t):
    """Normalise once: O / l and lse = m + ln l; an empty partial gives (0, -inf)."""
    m, l, o = t
    ok = l > 0
    out = np.zeros_like(o)
    out[ok] = o[ok] / l[ok, None]
    lse = np.full(m.shape, NEG_INF)
    lse[ok] = m[ok] + np.log(l[ok])
    return out, lse


def merge_states(o_parts, lse_parts):
    """Combine finalised attention states of disjoint key shards.

    The record's section 4 reduction applied to normalised partials: a shard's
    (O_i, lse_i) is its (m, l, O) triplet after ``finalize_triplet``, so with
    lse = ln sum_i exp(lse_i) the combined output is
    O = sum_i exp(lse_i - lse) O_i.  o_parts [P, R, d], lse_parts [P, R]; a
    shard with lse_i = -inf (no visible key) contributes nothing; a row whose
    shards are all empty gives O = 0, lse = -inf.
    """
    o_parts = _f64(o_parts)
    lse_parts = _f64(lse_parts)
    m = lse_parts.max(axis=0)
    ok = np.isfinite(m)
    m_safe = np.where(ok, m, 0.0)
    w = np.where(np.isfinite(lse_parts), np.exp(np.where(np.isfinite(lse_parts), lse_parts, 0.0)
                                                 - m_safe[None, :]), 0.0)
    total = w.sum(axis=0)
    out = np.zeros(o_parts.shape[1:])
    out[ok] = (w[:, ok, None] * o_parts[:, ok]).sum(axis=0) / total[ok, None]
    lse = np.full(m.shape, NEG_INF)
    lse[ok] = m[ok] + np.log(total[ok])
    return out, lse


def online_softmax_tiles(q_rows, k, v, scale, n_visible, tile):
    """The per-tile online-softmax loop of section 3, in float64.

    Running state m = -inf, l = 0, O = 0.  For each key tile: S = scale Q K^T,
    keys a row may not see are set to -inf, m' = max(m, rowmax S),
    P = exp(S - m'), corr = exp(m - m'), l = l corr + rowsum P,
    O = O corr + P V, m = m'.  Finally O / l and lse = m + ln l.
    """
    q_rows, k, v = _f64(q_rows), _f64(k), _f64(v)
    n_visible = np.asarray(n_visible, dtype=np.int64).reshape(-1)
    R, d = q_rows.shape
    N = k.shape[0]
    m = np.full(R, NEG_INF)
    l = np.zeros(R)
    o = np.zeros((R, d))
    for t0 in range(0, N, tile):
        t1 = min(N, t0 + tile)
        s = float(scale) * (q_rows @ k[t0:t1].T)
        keys = np.arange(t0, t1)
        s = np.where(keys[None, :] < n_visible[:, None], s, NEG_INF)
        m_new = np.maximum(m, s.max(axis=1))
        live = np.isfinite(m_new)                 # rows that have seen a key so far
        m_ref = np.where(live, m_new, 0.0)
        p = np.where(live[:, None], np.exp(s - m_ref[:, None]), 0.0)
        corr = np.where(np.isfinite(m), np.exp(np.where(np.isfinite(m), m, 0.0) - m_ref), 0.0)
        l = l * corr + p.sum(axis=1)
        o = o * corr[:, None] + p @ v[t0:t1]
        m = m_new
    return finalize_triplet((m, l, o))
