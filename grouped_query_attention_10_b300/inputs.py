"""Seeded synthetic inputs for grouped-query attention workloads.

This module only draws random numbers; it holds none of the attention
arithmetic, so both the CUDA path and the CPU oracle can consume its output.

Recipe: a ``torch.Generator`` seeded with the workload's seed, on the device
the tensors are created on; draws in the order Q, K, V, then the per-sequence
cache lengths. Values are i.i.d. N(0, 1) drawn in fp32 and rounded to bf16
(round to nearest even), so the library and the oracle read the very same
bf16 bits. The CPU and CUDA generators produce different streams for the same
seed; every comparison copies the device inputs to the host, never re-draws.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch


@dataclass(frozen=True)
class PrefillWorkload:
    name: str
    B: int
    L: int
    h_q: int
    g: int
    d: int
    causal: bool
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / (self.d ** 0.5)


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    B: int
    h_q: int
    g: int
    d: int
    S_max: int
    len_lo: int
    len_hi: int
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / (self.d ** 0.5)


# The five workloads the library is specified against.
TINY_CAUSAL_PREFILL = PrefillWorkload(
    "tiny_causal_prefill_b1_l128_hq8_g2_d64", B=1, L=128, h_q=8, g=2, d=64,
    causal=True, seed=1001)
NONCAUSAL_PREFILL = PrefillWorkload(
    "noncausal_prefill_b32_l1024_hq8_g4_d64", B=32, L=1024, h_q=8, g=4, d=64,
    causal=False, seed=1002)
LLAMA_CAUSAL_PREFILL = PrefillWorkload(
    "causal_prefill_b4_l4096_hq32_g8_d128", B=4, L=4096, h_q=32, g=8, d=128,
    causal=True, seed=1003)
DECODE_RAGGED = DecodeWorkload(
    "decode_b64_hq32_g8_d128_s8192_ragged", B=64, h_q=32, g=8, d=128,
    S_max=8192, len_lo=1024, len_hi=8192, seed=1004)
DECODE_SWEEP_G = (1, 2, 4, 8, 16, 32)


def decode_sweep(g: int) -> DecodeWorkload:
    """Long-context decode, every sequence full at 32768 cached tokens."""
    return DecodeWorkload(
        f"decode_sweep_b16_hq32_g{g}_d128_s32768", B=16, h_q=32, g=g, d=128,
        S_max=32768, len_lo=32768, len_hi=32768, seed=1005)


def _gen(seed: int, device) -> torch.Generator:
    return torch.Generator(device=device).manual_seed(seed)


def normal_bf16(shape, gen: torch.Generator, device, chunk_elems: int = 1 << 28):
    """i.i.d. N(0,1) drawn in fp32, rounded to bf16; drawn in chunks so the
    fp32 staging buffer stays bounded for multi-GB caches."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    n = flat.numel()
    pos = 0
    while pos < n:
        m = min(chunk_elems, n - pos)
        flat[pos:pos + m] = torch.randn(m, generator=gen, dtype=torch.float32,
                                        device=device).to(torch.bfloat16)
        pos += m
    return out


def prefill_inputs(w: PrefillWorkload, device="cpu", L: Optional[int] = None,
                   B: Optional[int] = None):
    """Q [B, L, h_q, d], K and V [B, L, g, d], bf16 (projection layout)."""
    B = w.B if B is None else B
    L = w.L if L is None else L
    gen = _gen(w.seed, device)
    q = normal_bf16((B, L, w.h_q, w.d), gen, device)
    k = normal_bf16((B, L, w.g, w.d), gen, device)
    v = normal_bf16((B, L, w.g, w.d), gen, device)
    return q, k, v


def decode_inputs(w: DecodeWorkload, device="cpu", B: Optional[int] = None,
                  S_max: Optional[int] = None):
    """Q [B, h_q, d], K/V cache [B, g, S_max, d] bf16, lengths int32 [B].

    Lengths are uniform integers in [len_lo, len_hi] (clipped to S_max).
    Every cache row is filled, including rows past a sequence's length.
    """
    B = w.B if B is None else B
    S_max = w.S_max if S_max is None else S_max
    gen = _gen(w.seed, device)
    q = normal_bf16((B, w.h_q, w.d), gen, device)
    kc = normal_bf16((B, w.g, S_max, w.d), gen, device)
    vc = normal_bf16((B, w.g, S_max, w.d), gen, device)
    lo = min(w.len_lo, S_max)
    hi = min(w.len_hi, S_max)
    lens = torch.randint(lo, hi + 1, (B,), generator=gen, device=device,
                         dtype=torch.int64).to(torch.int32)
    return q, kc, vc, lens


def random_bf16(shape, seed: int, device="cpu"):
    """Convenience: one seeded N(0,1) bf16 tensor."""
    return normal_bf16(shape, _gen(seed, device), device)


def random_lengths(B: int, lo: int, hi: int, seed: int, device="cpu"):
    gen = _gen(seed, device)
    return torch.randint(lo, hi + 1, (B,), generator=gen, device=device,
                         dtype=torch.int64).to(torch.int32)
