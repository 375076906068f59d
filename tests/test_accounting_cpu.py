"""The work counts behind every roofline figure, checked by brute force.

Each count is recomputed from the oracle's own visibility rule (which pair
(query, key) a head can see) or from the tensors a step has to move, so a
miscount in the closed forms (an off-by-one in the causal or window sums, a
missing factor of 2 for K and V) fails here.
"""

import numpy as np
import pytest

from grouped_query_attention_10_b300 import accounting
from oracle import gqa_oracle


def _visible_pairs(n_q, n_k, q_offset, window, causal=True):
    if not causal:
        return n_q * n_k
    return sum(1 for i in range(n_q) for j in range(n_k)
               if gqa_oracle._visible(i, j, q_offset, window))


@pytest.mark.parametrize("L", [1, 2, 7, 128, 300])
def test_prefill_flops_counts_visible_pairs(L):
    B, h_q, d = 2, 3, 8
    for causal in (True, False):
        want = 4 * B * h_q * d * _visible_pairs(L, L, 0, 0, causal)
        assert accounting.prefill_flops(B, L, h_q, d, causal) == want


@pytest.mark.parametrize("L,W", [(10, 1), (10, 3), (10, 10), (10, 50), (257, 64)])
def test_window_flops_counts_visible_pairs(L, W):
    B, h_q, d = 1, 2, 4
    want = 4 * B * h_q * d * _visible_pairs(L, L, 0, W)
    assert accounting.prefill_window_flops(B, L, h_q, d, W) == want


@pytest.mark.parametrize("lens,T", [([5, 9], 5), ([40, 17, 64], 8), ([1], 1)])
def test_cached_prefill_flops_counts_visible_pairs(lens, T):
    h_q, d = 3, 16
    pairs = sum(_visible_pairs(T, n, n - T, 0) for n in lens)
    assert accounting.prefill_cached_flops(lens, T, h_q, d) == 4 * h_q * d * pairs


def test_decode_bytes_read_each_valid_row_once_per_kv_head():
    lens, g, d = [3, 0, 11], 4, 64
    rows = sum(lens)
    assert accounting.decode_kv_bytes(lens, g, d) == 2 * rows * g * d * 2   # K and V, bf16
    assert accounting.decode_window_kv_bytes(lens, 5, g, d) == 2 * (3 + 0 + 5) * g * d * 2


def test_append_and_rope_append_bytes_count_the_tensors_moved():
    B, T, h_q, g, d = 2, 5, 8, 2, 64
    kv_new = 2 * np.zeros((B, T, g, d), np.uint16).nbytes        # K and V in
    assert accounting.append_bytes(B, T, g, d) == 2 * kv_new       # read + write
    q = np.zeros((B, T, h_q, d), np.uint16).nbytes
    assert accounting.rope_append_bytes(B, T, h_q, g, d) == 2 * (q + kv_new)
