"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module only draws random numbers and fixes shapes; it holds none of the
attention arithmetic, so both the CUDA path and the CPU oracle can be fed from
it without sharing any computation.

Workload shapes follow the Llama3-70B attention layer of the design record
"ADR-0060: AHBM GQA Fused Attention Kernel (Llama3-70B)", section 0 (Reference
dimensions: H_q=64, H_kv=8, G=8, d=128).  Values are bf16 rounded (round to
nearest even) from fp32 N(0,1) draws; sequence lengths of the ragged batch are
uniform integers.  The pages fix no data, so N(0,1) stands in for real
activations.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

__all__ = [
    "DecodeWorkload",
    "PrefillWorkload",
    "WORKLOADS",
    "bf16_normal",
    "ragged_seqlens",
    "decode_inputs",
    "prefill_inputs",
    "fill_padding",
]


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    B: int
    H_q: int
    H_kv: int
    d: int
    S_max: int
    seed: int
    num_splits: int = 0            # 0 = let the library's planner choose
    seqlen_lo: int | None = None   # ragged batch: U[seqlen_lo, seqlen_hi]
    seqlen_hi: int | None = None
    seqlen_seed: int | None = None

    @property
    def G(self) -> int:
        return self.H_q // self.H_kv

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


@dataclass(frozen=True)
class PrefillWorkload:
    name: str
    B: int
    H_q: int
    H_kv: int
    d: int
    T_q: int
    S_kv: int
    q_offset: int
    seed: int

    @property
    def G(self) -> int:
        return self.H_q // self.H_kv

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


WORKLOADS = {
    # small decode the oracle finishes instantly: one KV head, 4 splits
    "tiny_decode": DecodeWorkload("tiny_decode", B=1, H_q=8, H_kv=1, d=128, S_max=256,
                                  seed=0, num_splits=4),
    # one Llama3-70B layer, one 32K-token sequence
    "llama70b_decode_32k": DecodeWorkload("llama70b_decode_32k", B=1, H_q=64, H_kv=8, d=128,
                                          S_max=32768, seed=1),
    # 16 sequences of ragged length in a padded 128K-token cache
    "ragged_decode_b16": DecodeWorkload("ragged_decode_b16", B=16, H_q=64, H_kv=8, d=128,
                                        S_max=131072, seed=2, seqlen_lo=1024,
                                        seqlen_hi=131072, seqlen_seed=1002),
    # full causal prefill of an 8K prompt
    "causal_prefill_8k": PrefillWorkload("causal_prefill_8k", B=1, H_q=64, H_kv=8, d=128,
                                         T_q=8192, S_kv=8192, q_offset=0, seed=3),
    # last 2K-token chunk of a 32K prompt against the cached keys
    "chunked_prefill_32k": PrefillWorkload("chunked_prefill_32k", B=1, H_q=64, H_kv=8, d=128,
                                           T_q=2048, S_kv=32768, q_offset=30720, seed=4),
}


def _generator(seed: int, device) -> torch.Generator:
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))
    return g


def bf16_normal(shape, seed: int, device="cpu", *, chunk_elems: int = 1 << 28) -> torch.Tensor:
    """N(0,1) fp32 draws rounded to bf16, deterministic for (shape, seed, device type).

    Large tensors are drawn in slabs along dim 0 so the fp32 temporary stays
    bounded; the slab size only depends on the shape, so the values are
    reproducible.
    """
    shape = tuple(int(s) for s in shape)
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    numel = out.numel()
    if numel == 0:
        return out
    g = _generator(seed, device)
    if numel <= chunk_elems or len(shape) == 0:
        out.copy_(torch.randn(shape, generator=g, device=device, dtype=torch.float32))
        return out
    flat = out.view(-1)
    for start in range(0, numel, chunk_elems):
        n = min(chunk_elems, numel - start)
        flat[start:start + n].copy_(
            torch.randn((n,), generator=g, device=device, dtype=torch.float32))
    return out


def ragged_seqlens(B: int, lo: int, hi: int, seed: int) -> torch.Tensor:
    """B int32 lengths, uniform on [lo, hi] inclusive, drawn on the CPU."""
    g = _generator(seed, "cpu")
    return torch.randint(int(lo), int(hi) + 1, (int(B),), generator=g, dtype=torch.int64).to(
        torch.int32)


def fill_padding(cache: torch.Tensor, seqlens: torch.Tensor, value: float) -> None:
    """Overwrite cache[b, :, seqlens[b]:, :] with `value` (e.g. NaN) in place."""
    for b, n in enumerate(seqlens.tolist()):
        cache[b, :, int(n):, :] = value


def decode_inputs(B: int, H_q: int, H_kv: int, S_max: int, d: int, seed: int,
                  device="cpu", seqlens=None):
    """q [B,H_q,d], k_cache/v_cache [B,H_kv,S_max,d] (bf16), seqlens [B] int32 (CPU).

    q, k_cache and v_cache use the seeds seed, seed+1 and seed+2.  When
    `seqlens` is None every sequence fills the cache (seqlen = S_max).
    """
    q = bf16_normal((B, H_q, d), seed, device)
    k = bf16_normal((B, H_kv, S_max, d), seed + 1, device)
    v = bf16_normal((B, H_kv, S_max, d), seed + 2, device)
    if seqlens is None:
        seqlens = torch.full((B,), S_max, dtype=torch.int32)
    else:
        seqlens = torch.as_tensor(seqlens, dtype=torch.int32).cpu()
    return q, k, v, seqlens


def prefill_inputs(B: int, H_q: int, H_kv: int, T_q: int, S_kv: int, d: int, seed: int,
                   device="cpu"):
    """q [B,H_q,T_q,d], k/v [B,H_kv,S_kv,d] (bf16) with seeds seed, seed+1, seed+2."""
    q = bf16_normal((B, H_q, T_q, d), seed, device)
    k = bf16_normal((B, H_kv, S_kv, d), seed + 1, device)
    v = bf16_normal((B, H_kv, S_kv, d), seed + 2, device)
    return q, k, v


def workload_decode_inputs(w: DecodeWorkload, device="cpu"):
    seqlens = None
    if w.seqlen_lo is not None:
        seqlens = ragged_seqlens(w.B, w.seqlen_lo, w.seqlen_hi, w.seqlen_seed)
    return decode_inputs(w.B, w.H_q, w.H_kv, w.S_max, w.d, w.seed, device, seqlens)


def workload_prefill_inputs(w: PrefillWorkload, device="cpu"):
    return prefill_inputs(w.B, w.H_q, w.H_kv, w.T_q, w.S_kv, w.d, w.seed, device)
