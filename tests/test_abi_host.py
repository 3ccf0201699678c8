"""Host-side checks of the C ABI that need no GPU.

* the library builds for sm_103a and loads without a CUDA driver;
* it exports every function include/gqa_attn.h declares;
* the decode split planner and workspace sizing (pure host functions);
* argument rejection happens before any CUDA call.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import gqa_attention_decode_gb300 as gqa
from gqa_attention_decode_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gqa_attn.h")


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return gqa.load_library()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"GQA_API\s+[\w\s\*]+?\b(gqa_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ("gqa_attn_decode", "gqa_attn_prefill_causal", "gqa_attn_decode_plan",
                 "gqa_attn_decode_workspace_size", "gqa_status_string",
                 "gqa_attn_device_status"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(gqa.lib_path())
    missing = [n for n in declared_functions() if not hasattr(raw, n)]
    assert not missing, f"symbols declared in gqa_attn.h but not exported: {missing}"


def test_abi_version_and_status_strings(lib):
    assert gqa.gqa_attn_abi_version() == 1
    for code in range(6):
        assert gqa.gqa_status_string(code).startswith("GQA_")
    assert "unknown" in gqa.gqa_status_string(99)


@pytest.mark.parametrize("B,H_kv,S_max,sms,req,expect", [
    # one 32K sequence, 8 KV heads, 152 SMs: one wave of 19 splits x 8 heads
    (1, 8, 32768, 152, 0, (19, 1728)),
    # 128K keys, one sequence: still one wave of 19 splits (at least 16 per KV
    # head spread it over the GPU), chunks of 108 tiles
    (1, 8, 131072, 152, 0, (19, 6912)),
    # two sequences of 64K keys: 9 splits each, chunks capped at 2048 keys,
    # several waves of 2 CTAs/SM
    (2, 8, 65536, 152, 0, (32, 2048)),
    # tiny decode with 4 requested splits of one 64-key tile each
    (1, 1, 256, 152, 4, (4, 64)),
    # ragged batch: chunks capped at 2048 keys
    (16, 8, 131072, 152, 0, (64, 2048)),
    # requested splits above the tile count are clamped
    (1, 1, 100, 152, 50, (2, 64)),
    # empty cache
    (2, 8, 0, 152, 0, (1, 64)),
])
def test_decode_plan(lib, B, H_kv, S_max, sms, req, expect):
    assert gqa.gqa_attn_decode_plan(B, H_kv, S_max, sms, req) == expect


@pytest.mark.parametrize("B,H_kv,S_max,sms", [(1, 8, 32768, 152), (3, 2, 1000, 20),
                                               (16, 8, 131072, 152), (1, 1, 1, 152),
                                               (7, 3, 4097, 152),
                                               # one-wave plans with uncapped chunks
                                               (1, 8, 1 << 20, 152), (1, 1, 1 << 22, 152)])
def test_decode_plan_covers_every_key_once(lib, B, H_kv, S_max, sms):
    for req in (0, 1, 3, 1000):
        splits, chunk = gqa.gqa_attn_decode_plan(B, H_kv, S_max, sms, req)
        assert chunk % 64 == 0 and chunk > 0 and splits >= 1
        assert splits * chunk >= S_max          # the splits cover the cache
        assert (splits - 1) * chunk < S_max     # and no split starts past it


def _tc_splits(S_max, chunk):
    """The tcgen05 kernel's plan: the chunk rounded up to whole 128-key tiles."""
    c = -(-chunk // 128) * 128
    return -(-S_max // c), c


@pytest.mark.parametrize("B,H_kv,S_max", [(1, 8, (1 << 31) - 1), (1, 1, (1 << 31) - 64),
                                          (2, 8, (1 << 31) - 1000), (1, 8, 1 << 30)])
@pytest.mark.parametrize("req", [0, 100000])
def test_decode_plan_split_cap_near_int_max(lib, B, H_kv, S_max, req):
    """Splits run along the grid's z dimension (at most 65535): caches near 2^31
    keys get longer chunks instead, on both decode kernels."""
    splits, chunk = gqa.gqa_attn_decode_plan(B, H_kv, S_max, 152, req)
    assert 1 <= splits <= 65535 and chunk % 64 == 0
    assert splits * chunk >= S_max and (splits - 1) * chunk < S_max
    # the tensor-core path (G > 8, or G * T_q > 32 rows) rounds chunks to 128 keys
    tc_splits, tc_chunk = _tc_splits(S_max, chunk)
    assert 1 <= tc_splits <= splits <= 65535
    assert tc_splits * tc_chunk >= S_max and (tc_splits - 1) * tc_chunk < S_max
    H_q = 16 * H_kv                                            # G = 16
    assert gqa.gqa_attn_decode_workspace_size(B, H_q, H_kv, S_max, 128, 152, req) == \
        -(-(B * H_q * tc_splits * 129 * 4) // 256) * 256
    assert gqa.gqa_attn_decode_multi_workspace_size(B, 8 * H_kv, H_kv, 16, S_max, 128, 152,
                                                    req) == \
        -(-(B * 8 * H_kv * 16 * tc_splits * 129 * 4) // 256) * 256


def _device_chunk(seqlen, B, S_max, chunk, splits, H_kv, num_sms, tile):
    """The kernels' per-sequence chunk rule, restated with exact integer division:
    the sequence's tiles spread as if the batch held B like it, at most the
    host's chunk, at least what fits the sequence into the grid's splits."""
    if seqlen >= S_max:
        return chunk
    t = -(-seqlen // tile)
    chunk_tiles = chunk // tile
    work = t * H_kv * B
    c = chunk_tiles if work >= (1 << 20) else -(-work // num_sms)
    c = min(c, chunk_tiles)
    c = max(c, -(-t // splits) if t < (1 << 20) else chunk_tiles)
    return max(c, 1) * tile


@pytest.mark.parametrize("B,H_kv,S_max", [(1, 8, 32768), (16, 8, 131072), (1, 8, 1 << 20),
                                          (1, 1, 1 << 22), (4, 8, 65536), (3, 2, 1000)])
@pytest.mark.parametrize("req", [0, 7, 1000])
def test_device_chunk_fits_the_grid(lib, B, H_kv, S_max, req):
    """For any length in [0, S_max] the device-side chunk never exceeds the host's
    and fits the sequence into the grid's splits, so every key is covered."""
    splits, chunk = gqa.gqa_attn_decode_plan(B, H_kv, S_max, 152, req)
    rng = np.random.default_rng(S_max + req)
    lens = {0, 1, 63, 64, 65, S_max - 1, S_max} | set(int(x) for x in
                                                       rng.integers(0, S_max + 1, 300))
    for tile, (sp, ch) in ((64, (splits, chunk)), (128, _tc_splits(S_max, chunk))):
        for n in sorted(x for x in lens if 0 <= x <= S_max):
            c = _device_chunk(n, B, S_max, ch, sp, H_kv, 152, tile)
            assert c % tile == 0 and 0 < c <= ch
            assert -(-n // c) <= sp


def test_workspace_size(lib):
    splits, _ = gqa.gqa_attn_decode_plan(1, 8, 32768, 152, 0)
    ws = gqa.gqa_attn_decode_workspace_size(1, 64, 8, 32768, 128, 152, 0)
    assert ws >= 64 * splits * 129 * 4 and ws % 256 == 0
    assert gqa.gqa_attn_decode_workspace_size(1, 64, 8, 32768, 128, 0, 0) == 0  # bad num_sms


PIECE_BYTES = 4 * 128 * 130 * 4   # per piece, CTA pairs: 4 heads x 128 rows x (O[128], m, l) fp32
PIECE_BYTES_1 = 2 * 128 * 130 * 4  # per piece, one CTA: 2 slots x 128 rows


def _split_rule(units, workers, n_kv_min, piece_bytes, ws_bytes):
    """The planner's choice restated: the r = units % workers units of the last
    round are cut into the s pieces (2..min(32, n_kv_min // 8)) that minimise
    ceil(r s / workers) * (n_kv_min / s + 3), at most 4 rounds of pieces and
    within the workspace, if that beats n_kv_min (the units run whole)."""
    r = units % workers
    best, best_s = float(n_kv_min), 1
    if r:
        for s in range(2, min(32, n_kv_min // 8) + 1):
            pieces = r * s
            rounds = -(-pieces // workers)
            if rounds > 4 or pieces * piece_bytes > ws_bytes:
                break
            span = rounds * (n_kv_min / s + 3)
            if span < best:
                best, best_s = span, s
    return (units, r if best_s > 1 else 0, best_s)


@pytest.mark.parametrize("shape,sms,expect", [
    # chunked 32K (last 2K): 256 units on 76 pairs, the 28 of the fourth round cut
    # in 8 (224 pieces: three rounds of pieces of ~30 tiles instead of one of ~120)
    ((1, 64, 8, 2048, 32768, 30720), 152, (256, 28, 8)),
    # 8K causal: the last round's units are 1-3 key tiles long, nothing to split
    ((1, 64, 8, 8192, 8192, 0), 152, (1024, 0, 1)),
    # a 128-token chunk after 32K keys: 16 units, each cut in 9 (two rounds)
    ((1, 64, 8, 128, 32768, 32640), 152, (16, 16, 9)),
    # two units of 32 tiles: at most 32 // 8 = 4 pieces each
    ((1, 8, 2, 128, 4096, 3968), 152, (2, 2, 4)),
    # units fill whole rounds: no split
    ((1, 64, 8, 2048, 32768, 30720), 128, (256, 0, 1)),
    # one unit, 300 pairs: capped at 32 pieces
    ((1, 4, 1, 100, 65536, 65436), 600, (1, 1, 32)),
    # G = 3 (one CTA per unit): 16 query tiles x 2 KV heads head-pair units plus
    # 8 x 2 last-head units over two query tiles = 48 units on 152 CTAs, cut in 3
    ((1, 6, 2, 2048, 32768, 30720), 152, (48, 48, 3)),
    # G = 2, 8K causal: 2048 units, nothing to split
    ((1, 64, 32, 8192, 8192, 0), 152, (2048, 0, 1)),
    # MHA, a 256-token chunk after 128K keys: 64 heads x 1 two-tile unit on 152
    # CTAs, cut in 7 (three rounds of pieces of ~146 tiles)
    ((1, 64, 64, 256, 131072, 130816), 152, (64, 64, 7)),
    # G = 3 over 16 KV heads: 384 units on 152 CTAs, the 80 of the last round cut in 7
    ((1, 48, 16, 2048, 32768, 30720), 152, (384, 80, 7)),
])
def test_prefill_split_plan(lib, shape, sms, expect):
    B, H_q, H_kv, T_q, S_kv, q_off = shape
    got = gqa.gqa_attn_prefill_causal_plan(B, H_q, H_kv, T_q, S_kv, 128, q_off, sms, 1 << 30)
    assert got == expect
    units, split_units, s = got
    piece = PIECE_BYTES if (H_q // H_kv) % 4 == 0 else PIECE_BYTES_1
    workers = sms // 2 if (H_q // H_kv) % 4 == 0 else sms
    n_kv_min = min((q_off + min(T_q, 128) - 1) // 128 + 1, -(-S_kv // 128))
    assert got == _split_rule(units, workers, n_kv_min, piece, 1 << 30)
    if split_units:
        # the workspace the plan needs is within the size query's bound
        bound = gqa.gqa_attn_prefill_causal_workspace_size(B, H_q, H_kv, T_q, S_kv, 128, q_off,
                                                           sms)
        assert split_units * s * piece <= bound
        # a workspace one byte short: fewer pieces that fit (or none), never an error
        small = split_units * s * piece - 1
        _, su2, s2 = gqa.gqa_attn_prefill_causal_plan(B, H_q, H_kv, T_q, S_kv, 128, q_off, sms,
                                                      small)
        assert s2 < s and su2 * s2 * piece <= small
        assert (units, su2, s2) == _split_rule(units, workers, n_kv_min, piece, small)
        # no workspace: no split
        assert gqa.gqa_attn_prefill_causal_plan(B, H_q, H_kv, T_q, S_kv, 128, q_off, sms,
                                                0)[1] == 0


@pytest.mark.parametrize("q_off,T_q,s", [(30720, 2048, 2), (32640, 128, 4), (3968, 128, 4),
                                         (1000, 300, 3), (65436, 100, 32)])
def test_prefill_pieces_cover_the_key_range(q_off, T_q, s):
    """Piece i of s covers key tiles [i*n/s, (i+1)*n/s) of a unit with n tiles:
    together exactly [0, n), each at least 8 tiles when s <= n // 8, and every
    piece but the first starts at or before the tile of the unit's first query
    row, so each piece's first tile has a visible key in every row."""
    for qt in range((T_q + 127) // 128):
        q0 = q_off + 128 * qt
        qe = min(128 * (qt + 1), T_q)
        n = (q_off + qe - 1) // 128 + 1
        if s > n // 8:
            continue
        starts = [i * n // s for i in range(s + 1)]
        assert starts[0] == 0 and starts[-1] == n
        assert all(b - a >= 8 for a, b in zip(starts, starts[1:]))
        assert all(starts[i] * 128 <= q0 for i in range(s))


def test_prefill_workspace_size(lib):
    # four rounds of pieces at most: 4 x 76 pairs on 152 SMs
    assert gqa.gqa_attn_prefill_causal_workspace_size(1, 64, 8, 2048, 32768, 128, 30720,
                                                      152) == 304 * PIECE_BYTES
    # few units: up to 32 pieces per unit
    assert gqa.gqa_attn_prefill_causal_workspace_size(1, 8, 2, 128, 4096, 128, 3968,
                                                      152) == 64 * PIECE_BYTES
    assert gqa.gqa_attn_prefill_causal_workspace_size(1, 4, 1, 100, 4096, 128, 3996,
                                                      152) == 32 * PIECE_BYTES
    # one CTA per unit (G = 3): 2 head-pair + 2 last-head units, 32 pieces each at most
    assert gqa.gqa_attn_prefill_causal_workspace_size(1, 6, 2, 128, 4096, 128, 3968,
                                                      152) == 128 * PIECE_BYTES_1
    assert gqa.gqa_attn_prefill_causal_workspace_size(1, 6, 2, 2048, 32768, 128, 30720,
                                                      152) == 608 * PIECE_BYTES_1
    assert gqa.gqa_attn_prefill_causal_workspace_size(1, 64, 8, 128, 0, 128, 0, 152) == 0
    # rows past the last key are valid: 8 units on 76 pairs, each cut by key range
    assert gqa.gqa_attn_prefill_causal_workspace_size(1, 64, 8, 128, 100, 128, 0, 152) > 0
    assert gqa.gqa_attn_prefill_causal_workspace_size(1, 64, 8, 128, 256, 128, 0, 0) == 0


def test_plan_rejects_bad_arguments(lib):
    with pytest.raises(gqa.GQAError) as e:
        gqa.gqa_attn_decode_plan(-1, 8, 100, 152, 0)
    assert e.value.status == gqa.GQA_ERR_INVALID_ARG
    with pytest.raises(gqa.GQAError):
        gqa.gqa_attn_decode_plan(1, 8, 100, 0, 0)


def _raw_decode(lib, **kw):
    args = dict(q=1 << 20, k=1 << 20, v=1 << 20, seqlens=1 << 20, B=1, H_q=64, H_kv=8,
                S_max=1024, d=128, scale=0.088, num_splits=0, o=1 << 20, lse=1 << 20,
                ws=1 << 20, ws_bytes=1 << 30, stream=0)
    args.update(kw)
    v = ctypes.c_void_p
    return lib.gqa_attn_decode(v(args["q"]), v(args["k"]), v(args["v"]), v(args["seqlens"]),
                               args["B"], args["H_q"], args["H_kv"], args["S_max"], args["d"],
                               args["scale"], args["num_splits"], v(args["o"]), v(args["lse"]),
                               v(args["ws"]), args["ws_bytes"], v(args["stream"]))


@pytest.mark.parametrize("kw,expect", [
    (dict(q=0), gqa.GQA_ERR_INVALID_ARG),                      # null pointer
    (dict(k=(1 << 20) + 2), gqa.GQA_ERR_INVALID_ARG),          # misaligned pointer
    (dict(H_q=60), gqa.GQA_ERR_INVALID_ARG),                   # H_q % H_kv != 0
    (dict(d=64), gqa.GQA_ERR_UNSUPPORTED),                     # only d = 128
    (dict(H_q=576, H_kv=4), gqa.GQA_ERR_UNSUPPORTED),          # G = 144 > 128 rows
    (dict(num_splits=-1), gqa.GQA_ERR_INVALID_ARG),
    (dict(S_max=-5), gqa.GQA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), gqa.GQA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), gqa.GQA_ERR_INVALID_ARG),
    (dict(B=0), gqa.GQA_OK),                                   # empty batch: nothing to do
])
def test_decode_rejects_before_any_cuda_call(lib, kw, expect):
    assert _raw_decode(lib, **kw) == expect


def _raw_prefill(lib, **kw):
    args = dict(q=1 << 20, k=1 << 20, v=1 << 20, B=1, H_q=64, H_kv=8, T_q=128, S_kv=256,
                d=128, q_offset=0, scale=0.088, o=1 << 20, lse=1 << 20, stream=0)
    args.update(kw)
    v = ctypes.c_void_p
    return lib.gqa_attn_prefill_causal(v(args["q"]), v(args["k"]), v(args["v"]), args["B"],
                                       args["H_q"], args["H_kv"], args["T_q"], args["S_kv"],
                                       args["d"], args["q_offset"], args["scale"], v(args["o"]),
                                       v(args["lse"]), v(args["stream"]))


@pytest.mark.parametrize("kw,expect", [
    (dict(v=0), gqa.GQA_ERR_INVALID_ARG),
    (dict(o=(1 << 20) + 8), gqa.GQA_ERR_INVALID_ARG),
    (dict(q_offset=-1), gqa.GQA_ERR_INVALID_ARG),
    (dict(S_kv=0), gqa.GQA_ERR_INVALID_ARG),                   # queries but no key
    (dict(S_kv=0, T_q=0), gqa.GQA_OK),
    (dict(H_kv=7), gqa.GQA_ERR_INVALID_ARG),
    (dict(d=96), gqa.GQA_ERR_UNSUPPORTED),
    (dict(T_q=0), gqa.GQA_OK),
    (dict(B=0), gqa.GQA_OK),
])
def test_prefill_rejects_before_any_cuda_call(lib, kw, expect):
    assert _raw_prefill(lib, **kw) == expect


def test_binding_refuses_cpu_tensors(lib):
    import torch
    q = torch.zeros((1, 8, 128), dtype=torch.bfloat16)
    k = torch.zeros((1, 1, 64, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        gqa.gqa_attn_decode(q, k, k, torch.zeros(1, dtype=torch.int32), 0.1)


def _raw_paged(lib, **kw):
    args = dict(q=1 << 20, k=1 << 20, v=1 << 20, table=1 << 20, seqlens=1 << 20, B=2, H_q=64,
                H_kv=8, num_pages=10, page_size=256, max_pages=4, d=128, scale=0.088,
                num_splits=0, o=1 << 20, lse=1 << 20, ws=1 << 20, ws_bytes=1 << 30, stream=0)
    args.update(kw)
    v = ctypes.c_void_p
    return lib.gqa_attn_decode_paged(v(args["q"]), v(args["k"]), v(args["v"]), v(args["table"]),
                                     v(args["seqlens"]), args["B"], args["H_q"], args["H_kv"],
                                     args["num_pages"], args["page_size"], args["max_pages"],
                                     args["d"], args["scale"], args["num_splits"], v(args["o"]),
                                     v(args["lse"]), v(args["ws"]), args["ws_bytes"],
                                     v(args["stream"]))


@pytest.mark.parametrize("kw,expect", [
    (dict(page_size=100), gqa.GQA_ERR_UNSUPPORTED),           # not a multiple of 64
    (dict(page_size=0), gqa.GQA_ERR_INVALID_ARG),
    (dict(table=0), gqa.GQA_ERR_INVALID_ARG),                 # no block table
    (dict(table=(1 << 20) + 4), gqa.GQA_ERR_INVALID_ARG),     # misaligned table
    (dict(num_pages=0), gqa.GQA_ERR_INVALID_ARG),
    (dict(max_pages=-1), gqa.GQA_ERR_INVALID_ARG),
    (dict(d=64), gqa.GQA_ERR_UNSUPPORTED),
    (dict(H_q=128, H_kv=8, page_size=64), gqa.GQA_ERR_UNSUPPORTED),  # G = 16 (tensor cores): 128-key pages
    (dict(H_q=8, H_kv=8, num_pages=1 << 28), gqa.GQA_ERR_UNSUPPORTED),  # pool blocks >= 2^31
    (dict(B=0), gqa.GQA_OK),
])
def test_paged_rejects_before_any_cuda_call(lib, kw, expect):
    assert _raw_paged(lib, **kw) == expect


def test_paged_multi_rejections(lib):
    v = ctypes.c_void_p
    p = 1 << 20
    call = lambda H_q, H_kv, T_q, page_size, B=1: lib.gqa_attn_decode_paged_multi(
        v(p), v(p), v(p), v(p), v(p), B, H_q, H_kv, T_q, 64, page_size, 8, 128, 0.088, 0, v(p),
        v(p), v(p), 1 << 30, v(0))
    assert call(64, 8, 17, 256) == gqa.GQA_ERR_UNSUPPORTED   # G * T_q = 136 > 128
    assert call(64, 8, 16, 64) == gqa.GQA_ERR_UNSUPPORTED    # tensor cores: 128-key pages
    assert call(64, 8, 0, 256) == gqa.GQA_ERR_INVALID_ARG
    assert call(64, 8, 16, 256, B=0) == gqa.GQA_OK


def test_release_build_carries_no_bounds_checks(lib):
    """The release library compiles the store checks away; its bounds self-test
    refuses before any CUDA call (the bounds-checked build is libgqa_attn_debug.so)."""
    assert gqa.gqa_attn_bounds_checked() is False
    assert lib.gqa_attn_selftest_bounds(ctypes.c_void_p(0)) == gqa.GQA_ERR_UNSUPPORTED
    assert "OUT_OF_BOUNDS" in gqa.gqa_status_string(gqa.GQA_ERR_OUT_OF_BOUNDS)


def test_paged_prefill_rejects_before_any_cuda_call(lib):
    v = ctypes.c_void_p
    p = 1 << 20
    def call(table=p, S_kv=1024, num_pages=8, page_size=256, max_pages=4, d=128, B=1):
        return lib.gqa_attn_prefill_causal_paged(v(p), v(p), v(p), v(table), B, 8, 2, 128, S_kv,
                                                 num_pages, page_size, max_pages, d, S_kv - 128,
                                                 0.088, v(p), v(p), v(0), 0, v(0))
    assert call(table=0) == gqa.GQA_ERR_INVALID_ARG
    assert call(S_kv=2048) == gqa.GQA_ERR_INVALID_ARG            # past max_pages * page_size
    assert call(num_pages=0) == gqa.GQA_ERR_INVALID_ARG
    assert call(page_size=64, max_pages=16) == gqa.GQA_ERR_UNSUPPORTED  # tiles straddle pages
    assert call(d=64) == gqa.GQA_ERR_UNSUPPORTED
    assert call(B=0) == gqa.GQA_OK


def test_merge_states_rejects_before_any_cuda_call(lib):
    v = ctypes.c_void_p
    p = 1 << 20
    call = lambda o_parts=p, lse_parts=p, n=2, rows=10, d=128, o=p, lse=p: \
        lib.gqa_attn_merge_states(v(o_parts), v(lse_parts), n, rows, d, v(o), v(lse), v(0))
    assert call(n=0) == gqa.GQA_ERR_INVALID_ARG
    assert call(rows=-1) == gqa.GQA_ERR_INVALID_ARG
    assert call(o=0) == gqa.GQA_ERR_INVALID_ARG
    assert call(lse_parts=p + 4) == gqa.GQA_ERR_INVALID_ARG    # misaligned
    assert call(d=64) == gqa.GQA_ERR_UNSUPPORTED
    assert call(rows=0) == gqa.GQA_OK                          # nothing to do


def test_multi_token_rejections(lib):
    v = ctypes.c_void_p
    p = 1 << 20
    call = lambda B, H_q, H_kv, T_q, d=128: lib.gqa_attn_decode_multi(
        v(p), v(p), v(p), v(p), B, H_q, H_kv, T_q, 1024, d, 0.088, 0, v(p), v(p), v(p), 1 << 30,
        v(0))
    assert call(1, 64, 8, 17) == gqa.GQA_ERR_UNSUPPORTED     # G * T_q = 136 > 128
    assert call(1, 64, 8, 0) == gqa.GQA_ERR_INVALID_ARG
    assert call(1, 64, 8, 2, d=64) == gqa.GQA_ERR_UNSUPPORTED
    assert call(65535, 65536, 8192, 1) == gqa.GQA_ERR_UNSUPPORTED  # > 2^31 output rows
    assert call(0, 64, 8, 2) == gqa.GQA_OK
    # workspace: per (row, split) O[128] and lse in fp32, rounded up to 256 bytes
    ws_bytes = lambda rows, splits: (rows * splits * 129 * 4 + 255) // 256 * 256
    assert gqa.gqa_attn_decode_workspace_size(1, 64, 8, 32768, 128, 152) == ws_bytes(64, 19)
    assert gqa.gqa_attn_decode_multi_workspace_size(1, 64, 8, 4, 32768, 128, 152) == \
        ws_bytes(64 * 4, 19)
    # more than 32 rows per KV head: tensor-core split kernel, chunks of whole
    # 128-key tiles (1728 keys -> 1792, still 19 splits for 32K keys)
    assert gqa.gqa_attn_decode_multi_workspace_size(1, 64, 8, 16, 32768, 128, 152) == \
        ws_bytes(64 * 16, 19)


def test_device_chunk_ceil_division_is_exact():
    """The device-side split planner divides with the approximate hardware
    reciprocal, then corrects the quotient once each way with integer compares
    (ceil_div_small in csrc/device_common.cuh).  The same steps in float32 here,
    with the reciprocal anywhere within 4 ulp of 1/d, must give ceil(n / d)
    exactly for every n < 2^20 it is used on."""
    rng = np.random.default_rng(11)

    def ceil_div(n, d, r):
        q = np.floor((n.astype(np.float32) * np.float32(r)).astype(np.float32)).astype(np.uint64)
        dd = np.uint64(d)
        q = np.where(q * dd > n, q - 1, np.where((q + 1) * dd <= n, q + 1, q))
        return q + (q * dd != n)

    for d in list(range(1, 160)) + [255, 1000, 4096, 65535, (1 << 20) - 1]:
        n = np.concatenate([np.arange(0, 4096, dtype=np.uint64),
                            rng.integers(0, 1 << 20, 20000).astype(np.uint64),
                            np.array([(1 << 20) - 1, d - 1, d, d + 1, 2 * d], dtype=np.uint64)])
        n = n[n < (1 << 20)]
        exact = (n + np.uint64(d - 1)) // np.uint64(d)
        r = np.float32(1) / np.float32(d)
        lo = hi = r
        for _ in range(5):
            assert np.array_equal(ceil_div(n, d, lo), exact), (d, lo)
            assert np.array_equal(ceil_div(n, d, hi), exact), (d, hi)
            lo = np.nextafter(lo, np.float32(0))
            hi = np.nextafter(hi, np.float32(np.inf))


def test_cluster_merge_slots_fit_the_receive_area():
    """Host restatement of the single-kernel decode's cluster merge: in a cluster
    of cs CTAs, column n (n < n_cols <= 8) is finalised by CTA n mod cs, which
    receives it from every CTA c of the cluster into slot c * per_rank + n / cs
    (per_rank = ceil(n_cols / cs)), with n / cs taken as (n >= cs) + (n >= 2 cs)
    + (n >= 3 cs).  Every finaliser's slots are distinct and below 16, and its
    expected byte count (columns it owns x cs senders x (128 + 1) floats)
    matches what the senders send it."""
    kRecvSlots, kD = 16, 128
    for cs in range(2, 17):
        for n_cols in range(1, 9):
            per_rank = (n_cols + cs - 1) // cs
            assert cs * per_rank <= kRecvSlots
            received = {r: [] for r in range(cs)}
            for c in range(cs):                       # sender
                for n in range(n_cols):
                    quo = (n >= cs) + (n >= 2 * cs) + (n >= 3 * cs)
                    assert quo == n // cs
                    dst = n - quo * cs
                    received[dst].append(c * per_rank + quo)
            for r in range(cs):
                n_mine = (n_cols - r + cs - 1) // cs if r < n_cols else 0
                slots = received[r]
                assert len(slots) == len(set(slots)) and all(0 <= x < kRecvSlots for x in slots)
                assert len(slots) * (kD + 1) * 4 == n_mine * cs * (kD + 1) * 4
