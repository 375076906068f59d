"""Algorithmic work of each step of the GQA forward, used for roofline figures.

Counts are of the work the method has to do, not of what a kernel happens to
execute: masked-out score entries, padded cache rows, split-KV partials and
the duplicated K/V reads of an explicit head repeat are all excluded.
"""

from __future__ import annotations


def prefill_flops(B: int, L: int, h_q: int, d: int, causal: bool) -> int:
    """Multiply-add FLOPs of S = Q K^T and O = P V (2 flops per MAC each).

    Every query head does both products over the keys it can see; the count
    does not depend on the number of K/V heads g.  Causal attention sees
    L(L+1)/2 (query, key) pairs per head, non-causal L*L.
    """
    pairs = L * (L + 1) // 2 if causal else L * L
    return 4 * B * h_q * d * pairs


def prefill_bytes(B: int, L: int, h_q: int, g: int, d: int, out_bytes: int = 4) -> int:
    """Compulsory HBM bytes: read Q, K, V once (bf16), write O once."""
    return 2 * B * L * h_q * d + 2 * 2 * B * L * g * d + out_bytes * B * L * h_q * d


def kv_cache_bytes(B: int, g: int, S: int, d: int, elem_bytes: int = 2) -> int:
    """Size of a K plus V cache of S tokens per sequence: proportional to g."""
    return 2 * B * g * S * d * elem_bytes


def decode_kv_bytes(seq_lens, g: int, d: int, elem_bytes: int = 2) -> int:
    """K and V bytes a decode step must read: every valid row once per K/V head."""
    total_rows = sum(int(x) for x in seq_lens)
    return 2 * total_rows * g * d * elem_bytes


def decode_flops(seq_lens, h_q: int, d: int) -> int:
    """q.k and p.v multiply-adds of one decode token over its valid rows."""
    total_rows = sum(int(x) for x in seq_lens)
    return 4 * total_rows * h_q * d


def append_bytes(B: int, T: int, g: int, d: int, elem_bytes: int = 2) -> int:
    """Read T new K and V rows per sequence and write them into the cache."""
    return 2 * 2 * B * T * g * d * elem_bytes


def prefill_window_flops(B: int, L: int, h_q: int, d: int, window: int) -> int:
    """Causal prefill with a sliding window of W keys: query i sees
    min(i + 1, W) keys."""
    pairs = sum(min(i + 1, window) for i in range(L))
    return 4 * B * h_q * d * pairs


def prefill_cached_flops(seq_lens, T: int, h_q: int, d: int) -> int:
    """Chunked prefill of T new tokens per sequence over its cache: new token
    t of a sequence with n rows sits at position n - T + t and sees
    n - T + t + 1 keys."""
    pairs = sum(T * (int(n) - T) + T * (T + 1) // 2 for n in seq_lens)
    return 4 * h_q * d * pairs


def decode_window_kv_bytes(seq_lens, window: int, g: int, d: int, elem_bytes: int = 2) -> int:
    """K and V bytes of a windowed decode: the last min(len, W) rows."""
    total_rows = sum(min(int(x), window) for x in seq_lens)
    return 2 * total_rows * g * d * elem_bytes


def rope_append_bytes(B: int, T: int, h_q: int, g: int, d: int, elem_bytes: int = 2) -> int:
    """Fused RoPE append: read the new query, key and value rows and write the
    rotated queries and the cache rows (the cos/sin rows are L2-resident)."""
    return 2 * B * T * (h_q + 2 * g) * d * elem_bytes
