"""Every kernel path under the bounds-checked build (libgqa_attn_debug.so).

That build checks, in every kernel, the index of each global store against the
extent the kernel derives from its arguments and records a violation as
GQA_ERR_OUT_OF_BOUNDS in the device status word (the store is skipped): a
stand-in for a memory checker.  The calls below reach the warp-MMA and
tcgen05 decode kernels (dense and paged, one and many tokens, the
single-kernel cluster merge and split + merge), both causal prefill kernels
with and without the key-range split, and the merge of shard states; none may
record a violation, and the results must match the oracle.  The same build
counts the S = Q K^T tile products the prefill kernels issue, which must equal
the causal (lower-triangular) count of the design record's verification plan.  The library
is loaded in a child process (one library per process).
"""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = textwrap.dedent("""
    import math, sys
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import numpy as np, torch
    import gqa_synth, oracle
    import gqa_attention_decode_gb300 as gqa
    from parity import compare

    gqa.load_library()
    assert gqa.gqa_attn_bounds_checked(), "not the bounds-checked build"
    dev = torch.device("cuda", 0)
    np64 = lambda t: t.detach().float().cpu().numpy().astype(np.float64)

    def ok(what):
        st = gqa.gqa_attn_device_status()
        assert st == gqa.GQA_OK, (what, st)

    # decode: cluster-merged single kernel, split + merge, T_q = 4, T_q = 16 (tcgen05)
    for (B, H_q, H_kv, S, T_q, splits) in [(1, 8, 1, 256, 1, 4), (2, 64, 8, 4096, 1, 0),
                                            (2, 64, 8, 4096, 4, 0), (1, 64, 8, 4096, 16, 0),
                                            (3, 32, 2, 2048, 1, 40)]:
        q = gqa_synth.bf16_normal((B, H_q, T_q, 128), 1, dev)
        _, k, v, sl = gqa_synth.decode_inputs(B, H_q, H_kv, S, 128, 2, dev,
                                              [S] + [S // 3] * (B - 1))
        o, lse = gqa.gqa_attn_decode_multi(q, k, v, sl.to(dev), 0.088, splits)
        torch.cuda.synchronize()
        ok(("decode", B, H_q, H_kv, S, T_q, splits))
        o_ref, l_ref = oracle.decode_multi(np64(q), np64(k), np64(v), sl.numpy(), 0.088)
        compare(o, lse, o_ref, l_ref, "debug decode")
        # the same cache, paged (256-key pages in pool order)
        mp = S // 256
        kp = k.view(B, H_kv, mp, 256, 128).permute(0, 2, 1, 3, 4).reshape(B * mp, H_kv, 256, 128).contiguous()
        vp = v.view(B, H_kv, mp, 256, 128).permute(0, 2, 1, 3, 4).reshape(B * mp, H_kv, 256, 128).contiguous()
        table = torch.arange(B * mp, dtype=torch.int32, device=dev).view(B, mp)
        o2, l2 = gqa.gqa_attn_decode_paged_multi(q, kp, vp, table, sl.to(dev), 0.088, splits)
        torch.cuda.synchronize()
        ok(("paged decode", B, H_q, H_kv, S, T_q, splits))
        assert torch.equal(o2, o) and torch.equal(l2, lse)

    # short sequences in a long cache (the device-side chunk), T_q = 1 and 16
    for T_q in (1, 16):
        q = gqa_synth.bf16_normal((2, 64, T_q, 128), 6, dev)
        _, k, v, sl = gqa_synth.decode_inputs(2, 64, 8, 32768, 128, 7, dev, [3000, 17])
        o, lse = gqa.gqa_attn_decode_multi(q, k, v, sl.to(dev), 0.088)
        torch.cuda.synchronize()
        ok(("short in long cache", T_q))
        o_ref, l_ref = oracle.decode_multi(np64(q), np64(k[:, :, :3000]), np64(v[:, :, :3000]),
                                           sl.numpy(), 0.088)
        compare(o, lse, o_ref, l_ref, "debug short in long cache")

    # The record's causal tile count (section 11): query tile t of a head sees key
    # tiles 0 .. (q_offset + min(128 t + 128, T_q) - 1) // 128; the kernels must
    # issue exactly that many S products per head and tile -- plus, for odd group
    # sizes, the known extra of the group's last head, which runs query tiles t
    # and t - 1 together over tile t's key range (a lone tile 0 with a discarded
    # copy of itself).
    def n_kv(t, T_q, q_offset, S):
        return min((q_offset + min(128 * t + 128, T_q) - 1) // 128 + 1, -(-S // 128))

    def causal_s_tiles(B, H_q, T_q, q_offset, S):
        return B * H_q * sum(n_kv(t, T_q, q_offset, S) for t in range(-(-T_q // 128)))

    def issued_s_tiles(B, H_q, H_kv, T_q, q_offset, S):
        G, n_qt = H_q // H_kv, -(-T_q // 128)
        extra = 0
        if G % 2 == 1:
            for r in range(0, n_qt, 2):
                t0 = n_qt - 1 - r
                extra += (n_kv(t0, T_q, q_offset, S) - n_kv(t0 - 1, T_q, q_offset, S) if t0 > 0
                          else n_kv(0, T_q, q_offset, S))
        return causal_s_tiles(B, H_q, T_q, q_offset, S) + B * H_kv * extra

    gqa.gqa_attn_debug_s_tile_count()          # start from zero
    # prefill: CTA pairs (G = 8, 4) and one CTA per unit (G = 3, 1, 2), whole and split
    # (the last cases put rows past the last key: every key tile, none beyond)
    for (B, H_q, H_kv, T, S, qo) in [(1, 16, 2, 300, 300, 0), (1, 8, 2, 128, 4096, 3968),
                                     (1, 6, 2, 200, 200, 0), (1, 6, 2, 128, 4096, 3968),
                                     (1, 4, 4, 256, 2304, 2048), (1, 16, 2, 200, 3000, 2800),
                                     (2, 16, 2, 1024, 1024, 0), (1, 8, 4, 1000, 1000, 0),
                                     (1, 3, 3, 640, 700, 60), (1, 64, 8, 2048, 2048, 0),
                                     (1, 64, 8, 512, 8192, 7680), (1, 16, 2, 300, 256, 100),
                                     (1, 6, 2, 400, 300, 1000), (1, 64, 8, 256, 1024, 4096)]:
        q, k, v = gqa_synth.prefill_inputs(B, H_q, H_kv, T, S, 128, seed=3, device=dev)
        o, lse = gqa.gqa_attn_prefill_causal(q, k, v, 0.088, qo)
        torch.cuda.synchronize()
        ok(("prefill", B, H_q, H_kv, T, S))
        got = gqa.gqa_attn_debug_s_tile_count()
        want = issued_s_tiles(B, H_q, H_kv, T, qo, S)
        assert got == want, ("S tile count", B, H_q, H_kv, T, S, got, want)
        if (H_q // H_kv) % 2 == 0:   # no odd-group extra: exactly the lower triangle
            assert got == causal_s_tiles(B, H_q, T, qo, S)
        print("S tiles", (B, H_q, H_kv, T, S), got, "causal", causal_s_tiles(B, H_q, T, qo, S),
              "square", B * H_q * (-(-T // 128)) * (-(-S // 128)))
        o_ref, l_ref = oracle.prefill_causal(np64(q), np64(k), np64(v), qo, 0.088)
        compare(o, lse, o_ref, l_ref, "debug prefill")

    # prefill over a paged cache (pool in order, 256-key pages, a ragged last page)
    q, k, v = gqa_synth.prefill_inputs(1, 6, 2, 200, 1000, 128, seed=4, device=dev)
    kp = torch.zeros((4, 2, 256, 128), dtype=k.dtype, device=dev)
    vp = torch.zeros_like(kp)
    for i in range(4):
        n = min(256, 1000 - 256 * i)
        kp[i, :, :n] = k[0, :, 256 * i:256 * i + n]
        vp[i, :, :n] = v[0, :, 256 * i:256 * i + n]
    table = torch.arange(4, dtype=torch.int32, device=dev).view(1, 4)
    o, lse = gqa.gqa_attn_prefill_causal_paged(q, kp, vp, table, 1000, 0.088, 800)
    torch.cuda.synchronize()
    ok("paged prefill")
    o_ref, l_ref = oracle.prefill_causal(np64(q), np64(k), np64(v), 800, 0.088)
    compare(o, lse, o_ref, l_ref, "debug paged prefill")

    # the same on CTA pairs (G = 8, whole key tiles)
    q, k, v = gqa_synth.prefill_inputs(1, 16, 2, 300, 1024, 128, seed=5, device=dev)
    kp = k[0].view(2, 4, 256, 128).permute(1, 0, 2, 3).contiguous()
    vp = v[0].view(2, 4, 256, 128).permute(1, 0, 2, 3).contiguous()
    table = torch.arange(4, dtype=torch.int32, device=dev).view(1, 4)
    o, lse = gqa.gqa_attn_prefill_causal_paged(q, kp, vp, table, 1024, 0.088, 724)
    torch.cuda.synchronize()
    ok("paged prefill, CTA pairs")
    o_ref, l_ref = oracle.prefill_causal(np64(q), np64(k), np64(v), 724, 0.088)
    compare(o, lse, o_ref, l_ref, "debug paged prefill, CTA pairs")

    # merge of shard states
    parts = torch.randn((3, 1000, 128), device=dev).to(torch.bfloat16)
    lses = torch.randn((3, 1000), device=dev)
    gqa.gqa_attn_merge_states(parts, lses)
    torch.cuda.synchronize()
    ok("merge states")

    # the check itself: one store one element past its range is recorded
    gqa.gqa_attn_selftest_bounds()
    assert gqa.gqa_attn_device_status() == gqa.GQA_ERR_OUT_OF_BOUNDS
    assert gqa.gqa_attn_device_status() == gqa.GQA_OK     # read and cleared
    print("debug-bounds ok")
""")


def test_every_path_under_the_bounds_checked_build():
    sys.path.insert(0, ROOT)
    from gqa_attention_decode_gb300 import build
    lib = build.build(debug_bounds=True)
    env = dict(os.environ, GQA_ATTN_LIB=lib)
    r = subprocess.run([sys.executable, "-c", f"import os\nROOT = {ROOT!r}\n" + SCRIPT],
                       env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "debug-bounds ok" in r.stdout
