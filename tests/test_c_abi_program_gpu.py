"""The library from a plain C program: no Python, no torch, only the C ABI.

tests/c_abi_program.c is compiled against include/gqa_attn.h and linked with
libgqa_attn.so; it allocates device buffers with cudaMalloc, runs one decode
(Llama3-70B heads, three ragged sequences) and one chunked causal prefill, and
writes the outputs to files, which are compared here with the fp64 oracle on
the same seeded inputs.
"""
import math
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import gqa_synth
import oracle
from parity import compare

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "gqa_attention_decode_gb300")


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().tobytes()


def test_c_program_decode_and_prefill(tmp_path):
    from gqa_attention_decode_gb300 import build
    build.build()
    nvcc = build.nvcc_path()
    exe = str(tmp_path / "c_abi_program")
    subprocess.run([nvcc, "-o", exe, os.path.join(ROOT, "tests", "c_abi_program.c"),
                    "-I", os.path.join(ROOT, "include"), "-L", PKG, "-lgqa_attn",
                    "-Xlinker", "-rpath", "-Xlinker", PKG], check=True, capture_output=True)
    B, H_q, H_kv, S_max = 3, 64, 8, 3000
    T_q, S_kv, q_offset = 300, 1000, 700
    scale = 1 / math.sqrt(128)
    q, k, v, sl = gqa_synth.decode_inputs(B, H_q, H_kv, S_max, 128, seed=61,
                                          seqlens=[3000, 1, 1777])
    pq, pk, pv = gqa_synth.prefill_inputs(1, H_q, H_kv, T_q, S_kv, 128, seed=62)
    d = tmp_path
    (d / "shapes.txt").write_text(f"{B} {H_q} {H_kv} {S_max} {T_q} {S_kv} {q_offset} {scale!r}\n")
    for name, t in (("q", q), ("k", k), ("v", v), ("pq", pq), ("pk", pk), ("pv", pv)):
        (d / f"{name}.bin").write_bytes(_bits(t))
    (d / "seqlens.bin").write_bytes(sl.numpy().astype("<i4").tobytes())
    r = subprocess.run([exe, str(d)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c abi program ok" in r.stdout

    def bf16_file(name, shape):
        raw = np.frombuffer((d / name).read_bytes(), dtype="<u2").astype(np.uint32) << 16
        return raw.view(np.float32).reshape(shape).astype(np.float64)

    o = bf16_file("o.bin", (B, H_q, 128))
    lse = np.frombuffer((d / "lse.bin").read_bytes(), dtype="<f4").reshape(B, H_q)
    o_ref, lse_ref = oracle.decode(q.float().numpy(), k.float().numpy(), v.float().numpy(),
                                   sl.numpy(), scale)
    compare(o, lse, o_ref, lse_ref, "C program: decode")
    po = bf16_file("po.bin", (1, H_q, T_q, 128))
    plse = np.frombuffer((d / "plse.bin").read_bytes(), dtype="<f4").reshape(1, H_q, T_q)
    po_ref, plse_ref = oracle.prefill_causal(pq.float().numpy(), pk.float().numpy(),
                                             pv.float().numpy(), q_offset, scale)
    compare(po, plse, po_ref, plse_ref, "C program: chunked prefill")
